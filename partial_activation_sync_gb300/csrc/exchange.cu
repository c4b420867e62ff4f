// Local steps of the partial channel-reduce across processes (one GPU each):
// pack the channels of S into a dense send buffer, fold the blocks the other
// ranks sent in rank order, and scatter the reduced channels back.
//
// "Tensor-Parallelism with Partially Synchronized Activations", Introduction:
// the partial channel-reduce replaces the all-reduce after a row-parallel layer
// and sums only the channels of S over the ranks; the other channels never leave
// their rank.  Across GPUs the sum over S is an all-reduce of an [N, |S|] buffer;
// these kernels are the parts of it that run on each GPU (the transfers between
// GPUs are the caller's collectives).  The fold is a left fold in rank order in
// fp32 with one rounding, so the result does not depend on how the collectives
// split the work.
//
// All three are HBM-bound copies: 16-byte vectors when the layout allows,
// element by element otherwise.
#include <cuda_bf16.h>

#include <type_traits>

#include "caat_internal.h"

namespace caat {
namespace {

constexpr int THREADS = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf16_rn(float x) { return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// P[n, i] = Y[n, c_i], c_i = sel[i] (or i when sel is null).  ES = element bytes.
template <int ES>
__global__ void __launch_bounds__(THREADS) pack_scalar_kernel(int64_t N, int64_t s, const uint8_t *Y, int64_t ldy,
                                                              const int32_t *sel, uint8_t *P, int64_t ldp)
{
    using E = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
    const int64_t total = N * s;
    for (int64_t e = (int64_t)blockIdx.x * THREADS + threadIdx.x; e < total; e += (int64_t)gridDim.x * THREADS) {
        const int64_t n = e / s, i = e - n * s;
        const int64_t c = sel != nullptr ? (int64_t)__ldg(sel + i) : i;
        reinterpret_cast<E *>(P)[n * ldp + i] = reinterpret_cast<const E *>(Y)[n * ldy + c];
    }
}

// Y_k[n, c_i] = P[n, i] for every output k
template <int ES>
__global__ void __launch_bounds__(THREADS) unpack_scalar_kernel(int64_t N, int64_t s, const uint8_t *P, int64_t ldp,
                                                                const int32_t *sel, MutPtrs Y, int n_out, int64_t ldy)
{
    using E = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
    const int64_t total = N * s;
    for (int64_t e = (int64_t)blockIdx.x * THREADS + threadIdx.x; e < total; e += (int64_t)gridDim.x * THREADS) {
        const int64_t n = e / s, i = e - n * s;
        const int64_t c = sel != nullptr ? (int64_t)__ldg(sel + i) : i;
        const E v = reinterpret_cast<const E *>(P)[n * ldp + i];
        for (int k = 0; k < n_out; ++k) reinterpret_cast<E *>(Y.p[k])[n * ldy + c] = v;
    }
}

// Contiguous S with 16-byte aligned rows: copy [N, s] between two strided
// matrices in 16-byte vectors (vpr vectors per row), to one or several outputs.
__global__ void __launch_bounds__(THREADS) copy_vec_kernel(int64_t N, int64_t vpr, const uint4 *src, int64_t lds_v,
                                                           MutPtrs dst, int n_out, int64_t ldd_v)
{
    const int64_t total = N * vpr;
    for (int64_t e = (int64_t)blockIdx.x * THREADS + threadIdx.x; e < total; e += (int64_t)gridDim.x * THREADS) {
        const int64_t n = e / vpr, v = e - n * vpr;
        const uint4 x = __ldcs(src + n * lds_v + v);
        for (int k = 0; k < n_out; ++k) __stcs(reinterpret_cast<uint4 *>(dst.p[k]) + n * ldd_v + v, x);
    }
}

// out[n, c] = in_0[n, c] + ... + in_{t-1}[n, c] (block q at in + q * rank_stride),
// fp32 left fold in rank order, one rounding; 16-byte vectors (vpr per row).
template <bool BF16>
__global__ void __launch_bounds__(THREADS) fold_vec_kernel(int t, int64_t rows, int64_t vpr, const uint4 *in,
                                                           int64_t ld_v, int64_t rank_stride_v, uint4 *out,
                                                           int64_t ldo_v)
{
    const int64_t total = rows * vpr;
    for (int64_t e = (int64_t)blockIdx.x * THREADS + threadIdx.x; e < total; e += (int64_t)gridDim.x * THREADS) {
        const int64_t n = e / vpr, v = e - n * vpr;
        const uint4 *src = in + n * ld_v + v;
        float a[8];
        const uint4 x0 = __ldcs(src);
        const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w};
        if (BF16) {
#pragma unroll
            for (int j = 0; j < 4; ++j) { a[2 * j] = bf16_lo(w0[j]); a[2 * j + 1] = bf16_hi(w0[j]); }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) a[j] = __uint_as_float(w0[j]);
        }
        for (int q = 1; q < t; ++q) {
            const uint4 x = __ldcs(src + (int64_t)q * rank_stride_v);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            if (BF16) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    a[2 * j] = a[2 * j] + bf16_lo(w[j]);
                    a[2 * j + 1] = a[2 * j + 1] + bf16_hi(w[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) a[j] = a[j] + __uint_as_float(w[j]);
            }
        }
        uint32_t o[4];
        if (BF16) {
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = bf16_rn(a[2 * j]) | (bf16_rn(a[2 * j + 1]) << 16);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) o[j] = __float_as_uint(a[j]);
        }
        __stcs(out + n * ldo_v + v, make_uint4(o[0], o[1], o[2], o[3]));
    }
}

template <bool BF16>
__global__ void __launch_bounds__(THREADS) fold_scalar_kernel(int t, int64_t rows, int64_t cols, const void *in,
                                                              int64_t ld, int64_t rank_stride, void *out, int64_t ldo)
{
    const int64_t total = rows * cols;
    for (int64_t e = (int64_t)blockIdx.x * THREADS + threadIdx.x; e < total; e += (int64_t)gridDim.x * THREADS) {
        const int64_t n = e / cols, c = e - n * cols;
        float a = 0.0f;
        for (int q = 0; q < t; ++q) {
            const int64_t off = (int64_t)q * rank_stride + n * ld + c;
            const float x = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(in)[off] << 16)
                                 : reinterpret_cast<const float *>(in)[off];
            a = q == 0 ? x : a + x;
        }
        if (BF16) reinterpret_cast<uint16_t *>(out)[n * ldo + c] = (uint16_t)bf16_rn(a);
        else reinterpret_cast<float *>(out)[n * ldo + c] = a;
    }
}

int grid_for(int64_t items)
{
    const int64_t per = (int64_t)THREADS * 4;
    int64_t g = (items + per - 1) / per;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

inline bool al16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

struct Span { uintptr_t lo, hi; };
inline Span span_rows(const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t es)
{
    const int64_t n = rows > 0 && cols > 0 ? ((rows - 1) * ld + cols) * es : 0;
    return {(uintptr_t)p, (uintptr_t)p + (uintptr_t)n};
}
inline bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

}  // namespace
}  // namespace caat

using namespace caat;

extern "C" caat_status caat_pcr_pack(int64_t N, int64_t h, caat_dtype dt, const void *Y, int64_t ldy,
                                     const int32_t *sel, int64_t n_sel, void *P, int64_t ldp,
                                     caat_stream_t stream)
{
    if (N < 0 || h < 0 || n_sel < 0 || n_sel > h || ldy < h || ldp < n_sel) return CAAT_ERR_INVALID_ARG;
    if (dt != CAAT_F32 && dt != CAAT_BF16) return CAAT_ERR_INVALID_ARG;
    if (N == 0 || n_sel == 0) return CAAT_OK;
    if (const caat_status cs = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) return cs;
    if (Y == nullptr || P == nullptr) return CAAT_ERR_INVALID_ARG;
    const int64_t es = dt == CAAT_BF16 ? 2 : 4;
    if (overlap(span_rows(P, N, n_sel, ldp, es), span_rows(Y, N, h, ldy, es)) ||
        (sel != nullptr && overlap(span_rows(P, N, n_sel, ldp, es), {(uintptr_t)sel, (uintptr_t)(sel + n_sel)})))
        return CAAT_ERR_INVALID_ARG;
    const cudaStream_t s = (cudaStream_t)stream;
    const int64_t epv = 16 / es;   // elements per 16-byte vector
    if (sel == nullptr && n_sel % epv == 0 && ldy % epv == 0 && ldp % epv == 0 && al16(Y) && al16(P)) {
        MutPtrs d{};
        d.p[0] = P;
        const int64_t vpr = n_sel / epv;
        copy_vec_kernel<<<grid_for(N * vpr), THREADS, 0, s>>>(N, vpr, (const uint4 *)Y, ldy / epv, d, 1, ldp / epv);
        note_launch("pcr_pack_vec");
    } else {
        if (es == 2)
            pack_scalar_kernel<2><<<grid_for(N * n_sel), THREADS, 0, s>>>(N, n_sel, (const uint8_t *)Y, ldy, sel,
                                                                          (uint8_t *)P, ldp);
        else
            pack_scalar_kernel<4><<<grid_for(N * n_sel), THREADS, 0, s>>>(N, n_sel, (const uint8_t *)Y, ldy, sel,
                                                                          (uint8_t *)P, ldp);
        note_launch("pcr_pack");
    }
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

extern "C" caat_status caat_pcr_unpack(int64_t N, int64_t h, caat_dtype dt, const void *P, int64_t ldp,
                                       const int32_t *sel, int64_t n_sel, void *const *Y, int n_out,
                                       int64_t ldy, caat_stream_t stream)
{
    if (N < 0 || h < 0 || n_sel < 0 || n_sel > h || ldy < h || ldp < n_sel) return CAAT_ERR_INVALID_ARG;
    if (dt != CAAT_F32 && dt != CAAT_BF16) return CAAT_ERR_INVALID_ARG;
    if (n_out < 1 || n_out > CAAT_MAX_T || Y == nullptr) return CAAT_ERR_INVALID_ARG;
    if (N == 0 || n_sel == 0) return CAAT_OK;
    if (const caat_status cs = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) return cs;
    if (P == nullptr) return CAAT_ERR_INVALID_ARG;
    const int64_t es = dt == CAAT_BF16 ? 2 : 4;
    MutPtrs y{};
    const Span sp = span_rows(P, N, n_sel, ldp, es);
    for (int k = 0; k < n_out; ++k) {
        if (Y[k] == nullptr) return CAAT_ERR_INVALID_ARG;
        const Span sy = span_rows(Y[k], N, h, ldy, es);
        if (overlap(sy, sp)) return CAAT_ERR_INVALID_ARG;
        if (sel != nullptr && overlap(sy, {(uintptr_t)sel, (uintptr_t)(sel + n_sel)})) return CAAT_ERR_INVALID_ARG;
        for (int q = 0; q < k; ++q)
            if (overlap(sy, span_rows(Y[q], N, h, ldy, es))) return CAAT_ERR_INVALID_ARG;
        y.p[k] = Y[k];
    }
    const cudaStream_t s = (cudaStream_t)stream;
    const int64_t epv = 16 / es;
    bool vec = sel == nullptr && n_sel % epv == 0 && ldy % epv == 0 && ldp % epv == 0 && al16(P);
    for (int k = 0; k < n_out; ++k) vec = vec && al16(Y[k]);
    if (vec) {
        const int64_t vpr = n_sel / epv;
        copy_vec_kernel<<<grid_for(N * vpr), THREADS, 0, s>>>(N, vpr, (const uint4 *)P, ldp / epv, y, n_out,
                                                              ldy / epv);
        note_launch("pcr_unpack_vec");
    } else {
        if (es == 2)
            unpack_scalar_kernel<2><<<grid_for(N * n_sel), THREADS, 0, s>>>(N, n_sel, (const uint8_t *)P, ldp, sel,
                                                                            y, n_out, ldy);
        else
            unpack_scalar_kernel<4><<<grid_for(N * n_sel), THREADS, 0, s>>>(N, n_sel, (const uint8_t *)P, ldp, sel,
                                                                            y, n_out, ldy);
        note_launch("pcr_unpack");
    }
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

extern "C" caat_status caat_rank_fold(int t, int64_t rows, int64_t cols, caat_dtype dt, const void *in,
                                      int64_t ld_in, int64_t rank_stride, void *out, int64_t ld_out,
                                      caat_stream_t stream)
{
    if (t < 1 || t > 4096 || rows < 0 || cols < 0 || ld_in < cols || ld_out < cols) return CAAT_ERR_INVALID_ARG;
    if (dt != CAAT_F32 && dt != CAAT_BF16) return CAAT_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CAAT_OK;
    if (in == nullptr || out == nullptr) return CAAT_ERR_INVALID_ARG;
    const int64_t es = dt == CAAT_BF16 ? 2 : 4;
    // the t blocks must not overlap one another, nor the output any of them
    if (t > 1 && rank_stride < (rows - 1) * ld_in + cols) return CAAT_ERR_INVALID_ARG;
    const Span so = span_rows(out, rows, cols, ld_out, es);
    const Span si = {(uintptr_t)in, (uintptr_t)in + (uintptr_t)(((int64_t)(t - 1) * rank_stride + (rows - 1) * ld_in + cols) * es)};
    if (overlap(so, si)) return CAAT_ERR_INVALID_ARG;
    const cudaStream_t s = (cudaStream_t)stream;
    const int64_t epv = 16 / es;
    if (cols % epv == 0 && ld_in % epv == 0 && ld_out % epv == 0 && rank_stride % epv == 0 && al16(in) && al16(out)) {
        const int64_t vpr = cols / epv;
        if (es == 2)
            fold_vec_kernel<true><<<grid_for(rows * vpr), THREADS, 0, s>>>(t, rows, vpr, (const uint4 *)in, ld_in / epv,
                                                                           rank_stride / epv, (uint4 *)out, ld_out / epv);
        else
            fold_vec_kernel<false><<<grid_for(rows * vpr), THREADS, 0, s>>>(t, rows, vpr, (const uint4 *)in, ld_in / epv,
                                                                            rank_stride / epv, (uint4 *)out, ld_out / epv);
        note_launch("rank_fold_vec");
    } else {
        if (es == 2)
            fold_scalar_kernel<true><<<grid_for(rows * cols), THREADS, 0, s>>>(t, rows, cols, in, ld_in, rank_stride,
                                                                               out, ld_out);
        else
            fold_scalar_kernel<false><<<grid_for(rows * cols), THREADS, 0, s>>>(t, rows, cols, in, ld_in, rank_stride,
                                                                                out, ld_out);
        note_launch("rank_fold");
    }
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}
