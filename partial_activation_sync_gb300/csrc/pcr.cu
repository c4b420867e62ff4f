// Standalone partial channel-reduce (PCR) over t partial tensors.
//
// "Tensor-Parallelism with Partially Synchronized Activations", Introduction,
// definition of the partial channel-reduce: channels in S are summed over the t
// ranks, the others keep each rank's own value.
//
// HBM-bound: out of place every element of the t inputs is read once and every
// element of the t outputs written once (2 * t * N * h * elem bytes); in place
// only 16-byte chunks that hold a channel of S are touched.  One thread owns one
// 16-byte chunk of one row for all t ranks, so the t loads of a chunk are in
// flight together and the fp32 sum is a left fold in rank order (bit-exact).
// Channel membership is a bitmap in shared memory built from the sorted index
// list at block start.
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "caat_internal.h"

namespace caat {
namespace {

// The reduce kernels are launched as programmatic dependents of the previous
// launch in the stream (see launch_dependent): a block may start while that
// grid finishes, so it waits for it before its first access to global memory
// (the index list of S, then the inputs), and then lets the next grid start.
__device__ __forceinline__ void build_bitmap(uint32_t *bm, int64_t h, const int32_t *sel,
                                             int64_t n_sel)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t words = (h + 31) >> 5;
    if (sel == nullptr) {   // S = {0, ..., n_sel-1}
        for (int64_t w = threadIdx.x; w < words; w += blockDim.x) {
            const int64_t lo = w * 32;
            bm[w] = n_sel >= lo + 32 ? 0xffffffffu : (n_sel <= lo ? 0u : ((1u << (n_sel - lo)) - 1u));
        }
        __syncthreads();
        return;
    }
    for (int64_t w = threadIdx.x; w < words; w += blockDim.x) bm[w] = 0u;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < n_sel; i += blockDim.x) {
        const int32_t c = sel[i];
        if (c >= 0 && c < h) atomicOr(&bm[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t rn_bf16(float x)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint4 ld_vec(const void *p, bool streaming)
{
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
    return streaming ? __ldcs(q) : *q;
}

__device__ __forceinline__ void st_vec(void *p, uint4 v, bool streaming)
{
    uint4 *q = reinterpret_cast<uint4 *>(p);
    if (streaming) __stcs(q, v); else *q = v;
}

// sum of the t vectors (fp32 left fold), per 32-bit word of the chunk
template <bool BF16>
struct Acc;

template <>
struct Acc<false> {           // 4 x fp32
    float a[4];
    __device__ __forceinline__ void init(uint4 v)
    {
        a[0] = __uint_as_float(v.x); a[1] = __uint_as_float(v.y);
        a[2] = __uint_as_float(v.z); a[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ void add(uint4 v)
    {
        a[0] = a[0] + __uint_as_float(v.x); a[1] = a[1] + __uint_as_float(v.y);
        a[2] = a[2] + __uint_as_float(v.z); a[3] = a[3] + __uint_as_float(v.w);
    }
    // lanes whose bit is set take the sum, the others keep v
    __device__ __forceinline__ uint4 mix(uint4 v, uint32_t bits) const
    {
        uint4 o;
        o.x = (bits & 1u) ? __float_as_uint(a[0]) : v.x;
        o.y = (bits & 2u) ? __float_as_uint(a[1]) : v.y;
        o.z = (bits & 4u) ? __float_as_uint(a[2]) : v.z;
        o.w = (bits & 8u) ? __float_as_uint(a[3]) : v.w;
        return o;
    }
};

template <>
struct Acc<true> {            // 8 x bf16, two per 32-bit word
    float a[8];
    __device__ __forceinline__ void init(uint4 v)
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) { a[2 * i] = lo_bf16(w[i]); a[2 * i + 1] = hi_bf16(w[i]); }
    }
    __device__ __forceinline__ void add(uint4 v)
    {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] = a[2 * i] + lo_bf16(w[i]);
            a[2 * i + 1] = a[2 * i + 1] + hi_bf16(w[i]);
        }
    }
    __device__ __forceinline__ uint4 mix(uint4 v, uint32_t bits) const
    {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = (bits >> (2 * i)) & 1u ? rn_bf16(a[2 * i]) : (w[i] & 0xffffu);
            const uint32_t hi = (bits >> (2 * i + 1)) & 1u ? rn_bf16(a[2 * i + 1]) : (w[i] >> 16);
            w[i] = lo | (hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// TT > 0: compile-time rank count, all t chunks held in registers.
// TT == 0: any t; chunks that mix S and non-S channels re-read their input.
template <int TT, bool BF16, bool INPLACE>
__global__ void __launch_bounds__(256)
pcr_vec_kernel(int t, int64_t N, int64_t h, ConstPtrs in, int64_t ld_in, MutPtrs out,
               int64_t ld_out, const int32_t *__restrict__ sel, int64_t n_sel)
{
    extern __shared__ uint32_t bm[];
    build_bitmap(bm, h, sel, n_sel);

    constexpr int VEC = BF16 ? 8 : 4;        // elements per 16-byte chunk
    constexpr int ES = BF16 ? 2 : 4;         // element size
    constexpr uint32_t FULL = (1u << VEC) - 1u;
    constexpr bool STREAM = !INPLACE;
    const int T = TT > 0 ? TT : t;
    const int64_t cpr = h / VEC;

    for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
        const int64_t off_in = n * ld_in * ES;
        const int64_t off_out = n * ld_out * ES;
        for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < cpr;
             j += (int64_t)gridDim.x * blockDim.x) {
            const int64_t c0 = j * VEC;
            const uint32_t bits = (bm[c0 >> 5] >> (c0 & 31)) & FULL;
            const int64_t bi = off_in + c0 * ES, bo = off_out + c0 * ES;
            if (INPLACE && bits == 0u) continue;
            if (TT > 0) {
                uint4 v[TT > 0 ? TT : 1];
#pragma unroll
                for (int r = 0; r < (TT > 0 ? TT : 1); ++r)
                    v[r] = ld_vec((const char *)in.p[r] + bi, STREAM);
                if (bits == 0u) {
#pragma unroll
                    for (int r = 0; r < (TT > 0 ? TT : 1); ++r)
                        st_vec((char *)out.p[r] + bo, v[r], STREAM);
                } else {
                    Acc<BF16> acc;
                    acc.init(v[0]);
#pragma unroll
                    for (int r = 1; r < (TT > 0 ? TT : 1); ++r) acc.add(v[r]);
#pragma unroll
                    for (int r = 0; r < (TT > 0 ? TT : 1); ++r)
                        st_vec((char *)out.p[r] + bo, acc.mix(v[r], bits), STREAM);
                }
            } else {
                if (bits == 0u) {
                    for (int r = 0; r < T; ++r)
                        st_vec((char *)out.p[r] + bo, ld_vec((const char *)in.p[r] + bi, STREAM),
                               STREAM);
                } else {
                    Acc<BF16> acc;
                    acc.init(ld_vec((const char *)in.p[0] + bi, false));
                    for (int r = 1; r < T; ++r) acc.add(ld_vec((const char *)in.p[r] + bi, false));
                    for (int r = 0; r < T; ++r) {
                        const uint4 v = bits == FULL ? make_uint4(0, 0, 0, 0)
                                                     : ld_vec((const char *)in.p[r] + bi, false);
                        st_vec((char *)out.p[r] + bo, acc.mix(v, bits), STREAM);
                    }
                }
            }
        }
    }
}

// Any alignment, any h: one thread per (row, channel), all t ranks.
template <bool BF16, bool INPLACE>
__global__ void __launch_bounds__(256)
pcr_scalar_kernel(int t, int64_t N, int64_t h, ConstPtrs in, int64_t ld_in, MutPtrs out,
                  int64_t ld_out, const int32_t *__restrict__ sel, int64_t n_sel)
{
    extern __shared__ uint32_t bm[];
    build_bitmap(bm, h, sel, n_sel);
    for (int64_t n = blockIdx.y; n < N; n += gridDim.y) {
        for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < h;
             c += (int64_t)gridDim.x * blockDim.x) {
            const bool inS = (bm[c >> 5] >> (c & 31)) & 1u;
            const int64_t ii = n * ld_in + c, oo = n * ld_out + c;
            if (BF16) {
                if (inS) {
                    const uint16_t *p0 = (const uint16_t *)in.p[0];
                    float a = __uint_as_float((uint32_t)p0[ii] << 16);
                    for (int r = 1; r < t; ++r)
                        a = a + __uint_as_float((uint32_t)((const uint16_t *)in.p[r])[ii] << 16);
                    const uint16_t o = (uint16_t)rn_bf16(a);
                    for (int r = 0; r < t; ++r) ((uint16_t *)out.p[r])[oo] = o;
                } else if (!INPLACE) {
                    for (int r = 0; r < t; ++r)
                        ((uint16_t *)out.p[r])[oo] = ((const uint16_t *)in.p[r])[ii];
                }
            } else {
                if (inS) {
                    float a = ((const float *)in.p[0])[ii];
                    for (int r = 1; r < t; ++r) a = a + ((const float *)in.p[r])[ii];
                    for (int r = 0; r < t; ++r) ((float *)out.p[r])[oo] = a;
                } else if (!INPLACE) {
                    for (int r = 0; r < t; ++r) ((float *)out.p[r])[oo] = ((const float *)in.p[r])[ii];
                }
            }
        }
    }
}

// out[n, c] = in_0[n, c] + ... + in_{t-1}[n, c] for c < s (bf16, fp32 left fold
// in rank order, one rounding): the channels of a contiguous S, reduced once
// instead of into every rank's copy.
// Block (x, y): x walks the 8-channel chunks of a row, y the rows of the block's
// row group, so a row narrower than 256 chunks still fills whole warps.
template <int TT>
__global__ void __launch_bounds__(256)
pcr_colsum_kernel(int t, int64_t N, int64_t s, ConstPtrs in, int64_t ld_in, uint16_t *__restrict__ out,
                  int64_t ld_out)
{
    const int T = TT > 0 ? TT : t;
    const int64_t cpr = s / 8;
    // a programmatic dependent of the previous launch: wait for it before reading
    // its outputs, then let the next grid start its setup
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t n = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; n < N; n += (int64_t)gridDim.y * blockDim.y) {
        for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < cpr;
             j += (int64_t)gridDim.x * blockDim.x) {
            const int64_t bi = (n * ld_in + j * 8) * 2;
            Acc<true> acc;
            if (TT > 0) {
                uint4 v[TT > 0 ? TT : 1];
#pragma unroll
                for (int r = 0; r < (TT > 0 ? TT : 1); ++r) v[r] = ld_vec((const char *)in.p[r] + bi, true);
                acc.init(v[0]);
#pragma unroll
                for (int r = 1; r < (TT > 0 ? TT : 1); ++r) acc.add(v[r]);
            } else {
                acc.init(ld_vec((const char *)in.p[0] + bi, true));
                for (int r = 1; r < T; ++r) acc.add(ld_vec((const char *)in.p[r] + bi, true));
            }
            st_vec(out + n * ld_out + j * 8, acc.mix(make_uint4(0, 0, 0, 0), 0xffu), false);
        }
    }
}


template <int TT, bool BF16, bool INPLACE>
void launch_vec(dim3 grid, dim3 block, size_t smem, cudaStream_t s, int t, int64_t N, int64_t h,
                const ConstPtrs &in, int64_t ld_in, const MutPtrs &out, int64_t ld_out,
                const int32_t *sel, int64_t n_sel)
{
    launch_dependent(pcr_vec_kernel<TT, BF16, INPLACE>, grid, block, smem, s, t, N, h, in, ld_in, out, ld_out,
                     sel, n_sel);
}

template <bool BF16, bool INPLACE>
void dispatch_vec(dim3 grid, dim3 block, size_t smem, cudaStream_t s, int t, int64_t N,
                  int64_t h, const ConstPtrs &in, int64_t ld_in, const MutPtrs &out,
                  int64_t ld_out, const int32_t *sel, int64_t n_sel)
{
#define CAAT_PCR_CASE(TT_) \
    case TT_: launch_vec<TT_, BF16, INPLACE>(grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel); break;
    switch (t) {
        CAAT_PCR_CASE(1) CAAT_PCR_CASE(2) CAAT_PCR_CASE(3) CAAT_PCR_CASE(4)
        CAAT_PCR_CASE(5) CAAT_PCR_CASE(6) CAAT_PCR_CASE(7) CAAT_PCR_CASE(8)
        default: launch_vec<0, BF16, INPLACE>(grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
    }
#undef CAAT_PCR_CASE
}

}  // namespace

caat_status launch_pcr_colsum(int t, int64_t N, int64_t s, const ConstPtrs &in, int64_t ld_in, void *out,
                              int64_t ld_out, cudaStream_t st)
{
    if (N == 0 || s == 0) return CAAT_OK;
    if (s % 8 || ld_in % 8 || ld_out % 8 || (uintptr_t)out % 16) return CAAT_ERR_UNSUPPORTED;
    for (int r = 0; r < t; ++r)
        if ((uintptr_t)in.p[r] % 16) return CAAT_ERR_UNSUPPORTED;
    // blocks of about 256 threads: units (8-channel chunks) of a row across x,
    // as many rows as fit across y; at most eight blocks per SM, rows strided
    const int64_t units = s / 8;
    const int bx = units >= 256 ? 256 : (int)units;
    const int by = 256 / bx;
    const int64_t gx = (units + bx - 1) / bx;
    int64_t gy = (N + by - 1) / by;
    const int64_t cap = ((int64_t)num_sms() * 8 + gx - 1) / gx;
    if (gy > cap) gy = cap;
    if (gy > 65535) gy = 65535;
    const dim3 grid((unsigned)gx, (unsigned)gy), bx2((unsigned)bx, (unsigned)by);
    uint16_t *o = (uint16_t *)out;
    switch (t) {
    case 2: launch_dependent(pcr_colsum_kernel<2>, grid, bx2, 0, st, t, N, s, in, ld_in, o, ld_out); break;
    case 4: launch_dependent(pcr_colsum_kernel<4>, grid, bx2, 0, st, t, N, s, in, ld_in, o, ld_out); break;
    case 8: launch_dependent(pcr_colsum_kernel<8>, grid, bx2, 0, st, t, N, s, in, ld_in, o, ld_out); break;
    default: launch_dependent(pcr_colsum_kernel<0>, grid, bx2, 0, st, t, N, s, in, ld_in, o, ld_out); break;
    }
    note_launch("pcr_colsum");
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

caat_status launch_pcr(int t, int64_t N, int64_t h, caat_dtype dt, const ConstPtrs &in,
                       int64_t ld_in, const MutPtrs &out, int64_t ld_out, bool in_place,
                       const int32_t *sel, int64_t n_sel, cudaStream_t s)
{
    if (N == 0 || h == 0) return CAAT_OK;
    if (in_place && n_sel == 0) return CAAT_OK;
    if (h > CAAT_MAX_H_BITMAP) return CAAT_ERR_UNSUPPORTED;
    const bool bf16 = dt == CAAT_BF16;
    const int es = bf16 ? 2 : 4, vec = 16 / es;
    bool vec_ok = (h % vec == 0) && (ld_in % vec == 0) && (ld_out % vec == 0);
    for (int r = 0; r < t && vec_ok; ++r)
        vec_ok = ((uintptr_t)in.p[r] % 16 == 0) && ((uintptr_t)out.p[r] % 16 == 0);
    const size_t smem = (size_t)((h + 31) / 32) * 4;
    const int64_t units = vec_ok ? h / vec : h;         // work items per row
    const int bx = units >= 256 ? 256 : (int)((units + 31) / 32 * 32);
    int64_t gx = (units + bx - 1) / bx;
    const int64_t target = (int64_t)num_sms() * (2048 / bx) * 2;   // two full waves
    if (gx > target) gx = target;
    int64_t gy = (target + gx - 1) / gx;
    if (gy > N) gy = N;
    if (gy > 65535) gy = 65535;
    const dim3 grid((unsigned)gx, (unsigned)gy), block(bx);
    if (vec_ok) {
        if (bf16) {
            if (in_place) dispatch_vec<true, true>(grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
            else dispatch_vec<true, false>(grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
        } else {
            if (in_place) dispatch_vec<false, true>(grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
            else dispatch_vec<false, false>(grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
        }
        note_launch("pcr_vec");
    } else {
        if (bf16) {
            if (in_place) launch_dependent(pcr_scalar_kernel<true, true>, grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
            else launch_dependent(pcr_scalar_kernel<true, false>, grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
        } else {
            if (in_place) launch_dependent(pcr_scalar_kernel<false, true>, grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
            else launch_dependent(pcr_scalar_kernel<false, false>, grid, block, smem, s, t, N, h, in, ld_in, out, ld_out, sel, n_sel);
        }
        note_launch("pcr_scalar");
    }
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

}  // namespace caat
