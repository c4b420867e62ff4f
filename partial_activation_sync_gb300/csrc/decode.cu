// Row-parallel forward + partial channel-reduce for few tokens (decode, N < 16):
// weight streaming on the CUDA cores.
//
// "Tensor-Parallelism with Partially Synchronized Activations" (Introduction,
// partial channel-reduce; inference with the partial reduce in place of the
// all-reduce).  With a handful of tokens the layer reads every weight once and
// does only 2*N flops per weight, so it is bound by HBM bandwidth, and the MMA
// tile (128 rows) would be almost empty.
//
// Layout of the work: a warp owns CPW consecutive output channels.  Its 32 lanes
// form t groups of 32/t lanes; group r walks shard r's K slice of those channels'
// weight rows (16-byte loads, several in flight per lane) and of the NT token rows
// of X (read-only path, L1-resident: X is tiny).  The group's partial sums are
// combined by shuffles; for channels outside S the group writes rank r's output,
// for channels in S the partials of all groups are combined once more and every
// group writes the total into its rank's output.
#include <cuda_bf16.h>

#include "caat_internal.h"

namespace caat {
namespace {

constexpr int CPW = 4;          // channels per warp
constexpr int WARPS = 8;        // warps per block
constexpr int U = 4;            // 16-byte loads in flight per lane per channel

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void widen8(uint4 v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// NT token rows per pass (rows >= N read as zero and are not written), TT ranks.
template <int NT, int TT>
__global__ void __launch_bounds__(WARPS * 32)
rowpar_fwd_decode_kernel(const uint16_t *__restrict__ X, int64_t ldx, const uint16_t *__restrict__ W,
                         int64_t ldw, MutPtrs Y, int64_t ldy, int64_t N, int64_t K, int64_t h,
                         const int32_t *__restrict__ sel, int64_t n_sel)
{
    constexpr int G = 32 / TT;                       // lanes per shard group
    constexpr int CPB = WARPS * CPW;                 // channels per block (32)
    __shared__ uint32_t smask;                       // bit i: channel cb + i is in S
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = lane / G, gl = lane % G;
    const int64_t kt = K / TT;
    const int64_t cb = (int64_t)blockIdx.x * CPB;
    const int64_t c0 = cb + (int64_t)warp * CPW;
    const int64_t row0 = (int64_t)blockIdx.y * NT;

    // membership of this block's channels: every thread scans a slice of S
    if (threadIdx.x == 0) smask = 0u;
    __syncthreads();
    if (sel == nullptr) {                            // S = {0, ..., n_sel-1}
        if (threadIdx.x == 0)
            smask = n_sel >= cb + CPB ? 0xffffffffu : (n_sel <= cb ? 0u : ((1u << (uint32_t)(n_sel - cb)) - 1u));
    } else {
        for (int64_t i = threadIdx.x; i < n_sel; i += WARPS * 32) {
            const int64_t c = sel[i];
            if (c >= cb && c < cb + CPB) atomicOr(&smask, 1u << (uint32_t)(c - cb));
        }
    }
    __syncthreads();
    if (c0 >= h) return;                             // whole warp

    float acc[CPW][NT];
#pragma unroll
    for (int c = 0; c < CPW; ++c)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[c][n] = 0.f;

    const int64_t kbeg = (int64_t)r * kt, kend = kbeg + kt;
    const uint16_t *wrow[CPW];
#pragma unroll
    for (int c = 0; c < CPW; ++c) wrow[c] = W + (c0 + c < h ? c0 + c : c0) * ldw;
    const uint16_t *xrow[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) xrow[n] = X + (row0 + n < N ? row0 + n : row0) * ldx;

    for (int64_t kb = kbeg + (int64_t)gl * 8; kb < kend; kb += (int64_t)G * 8 * U) {
        uint4 wv[U][CPW];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = kb + (int64_t)u * G * 8;
#pragma unroll
            for (int c = 0; c < CPW; ++c)
                wv[u][c] = (k < kend && c0 + c < h) ? ld_stream(wrow[c] + k) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = kb + (int64_t)u * G * 8;
            if (k < kend) {
                float xf[NT][8];
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    const uint4 xv = row0 + n < N ? __ldg(reinterpret_cast<const uint4 *>(xrow[n] + k))
                                                  : make_uint4(0, 0, 0, 0);
                    widen8(xv, xf[n]);
                }
#pragma unroll
                for (int c = 0; c < CPW; ++c) {
                    float wf[8];
                    widen8(wv[u][c], wf);
#pragma unroll
                    for (int n = 0; n < NT; ++n)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[c][n] = fmaf(wf[e], xf[n][e], acc[c][n]);
                }
            }
        }
    }

    // partial of shard r: sum over the group's lanes
#pragma unroll
    for (int off = G / 2; off >= 1; off >>= 1)
#pragma unroll
        for (int c = 0; c < CPW; ++c)
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[c][n] += __shfl_xor_sync(0xffffffffu, acc[c][n], off);
    // total over shards (for the channels of S)
    float tot[CPW][NT];
#pragma unroll
    for (int c = 0; c < CPW; ++c)
#pragma unroll
        for (int n = 0; n < NT; ++n) tot[c][n] = acc[c][n];
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
#pragma unroll
        for (int c = 0; c < CPW; ++c)
#pragma unroll
            for (int n = 0; n < NT; ++n) tot[c][n] += __shfl_xor_sync(0xffffffffu, tot[c][n], off);

    if (gl == 0) {
        uint16_t *yr = (uint16_t *)Y.p[r];
        const uint32_t m = smask >> (warp * CPW);
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            const int64_t ch = c0 + c;
            if (ch >= h) break;
            const bool s = (m >> c) & 1u;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                if (row0 + n >= N) break;
                yr[(row0 + n) * ldy + ch] = __bfloat16_as_ushort(__float2bfloat16_rn(s ? tot[c][n] : acc[c][n]));
            }
        }
    }
}

template <int NT>
void launch_nt(int t, dim3 grid, cudaStream_t s, const uint16_t *X, int64_t ldx, const uint16_t *W,
               int64_t ldw, const MutPtrs &Y, int64_t ldy, int64_t N, int64_t K, int64_t h,
               const int32_t *sel, int64_t n_sel)
{
#define CAAT_DEC_CASE(TT_) \
    case TT_: rowpar_fwd_decode_kernel<NT, TT_><<<grid, WARPS * 32, 0, s>>>(X, ldx, W, ldw, Y, ldy, N, K, h, sel, n_sel); break;
    switch (t) {
        CAAT_DEC_CASE(1) CAAT_DEC_CASE(2) CAAT_DEC_CASE(4) CAAT_DEC_CASE(8) CAAT_DEC_CASE(16) CAAT_DEC_CASE(32)
    }
#undef CAAT_DEC_CASE
}

}  // namespace

caat_status launch_rowpar_fwd_decode(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                     const void *W, int64_t ldw, const MutPtrs &Y, int64_t ldy,
                                     const int32_t *sel, int64_t n_sel, cudaStream_t s)
{
    if (t != 1 && t != 2 && t != 4 && t != 8 && t != 16 && t != 32) return CAAT_ERR_UNSUPPORTED;
    const int64_t kt = K / t;
    if (N < 1 || N > 64 || kt < 8 || kt % 8 != 0 || ldx % 8 != 0 || ldw % 8 != 0) return CAAT_ERR_UNSUPPORTED;
    if ((uintptr_t)X % 16 != 0 || (uintptr_t)W % 16 != 0) return CAAT_ERR_UNSUPPORTED;
    const int nt = N >= 8 ? 8 : (N >= 4 ? 4 : (N >= 2 ? 2 : 1));
    const int64_t chans_per_block = (int64_t)WARPS * CPW;
    const int64_t gx = (h + chans_per_block - 1) / chans_per_block;
    const int64_t gy = (N + nt - 1) / nt;
    if (gx > INT32_MAX || gy > 65535) return CAAT_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)gx, (unsigned)gy);
    const uint16_t *x = (const uint16_t *)X, *w = (const uint16_t *)W;
    switch (nt) {
    case 8: launch_nt<8>(t, grid, s, x, ldx, w, ldw, Y, ldy, N, K, h, sel, n_sel); break;
    case 4: launch_nt<4>(t, grid, s, x, ldx, w, ldw, Y, ldy, N, K, h, sel, n_sel); break;
    case 2: launch_nt<2>(t, grid, s, x, ldx, w, ldw, Y, ldy, N, K, h, sel, n_sel); break;
    default: launch_nt<1>(t, grid, s, x, ldx, w, ldw, Y, ldy, N, K, h, sel, n_sel); break;
    }
    note_launch("rowpar_fwd_decode");
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

}  // namespace caat
