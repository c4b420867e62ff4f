// CUDA-core (FFMA) GEMM paths: any strides, fp32 or bf16 storage, fp32 FMA.
//
// These are the exact-arithmetic paths of the library: the fp32 row-parallel
// layer (no TF32 anywhere), layouts the tensor-core kernels do not take, and the
// backward GEMMs.  64x64 output tile per 256-thread block, 4x4 outputs per thread,
// k-slices of 16 staged through shared memory.
//
// Row-parallel forward ("Tensor-Parallelism with Partially Synchronized
// Activations", Introduction, partial channel-reduce paragraph): for each output
// tile the block runs the t shards one after another; after shard r the channels
// outside S are final and go to Y[r], the channels of S add the shard's partial
// sum into a running total (rank order), written to every Y[r] at the end.
#include <cuda_bf16.h>

#include "caat_internal.h"

namespace caat {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <bool BF16>
__device__ __forceinline__ float ld_elem(const void *base, int64_t idx)
{
    if (BF16) return __uint_as_float((uint32_t)((const uint16_t *)base)[idx] << 16);
    return ((const float *)base)[idx];
}

template <bool BF16>
__device__ __forceinline__ void st_elem(void *base, int64_t idx, float v)
{
    if (BF16) ((uint16_t *)base)[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    else ((float *)base)[idx] = v;
}

// Stage A (BM x BK, element (m, k) at A[m*s0 + k*s1]) and B (BK x BN, element
// (k, n) at B[k*t0 + n*t1]) into shared memory as float, zero outside
// [0, M) x [k_lo, k_hi) x [0, Nn).
template <bool BF16>
__device__ __forceinline__ void stage_tiles(float (*As)[BM + 4], float (*Bs)[BN + 4],
                                            const void *A, int64_t s0, int64_t s1,
                                            const void *B, int64_t t0, int64_t t1,
                                            int64_t m0, int64_t n0, int64_t k0, int64_t k_hi,
                                            int64_t M, int64_t Nn)
{
    const int tid = threadIdx.x;
    // A: if k is the unit stride, consecutive threads walk k; else they walk m.
#pragma unroll
    for (int i = 0; i < (BM * BK) / NT; ++i) {
        const int e = tid + i * NT;
        int mm, kk;
        if (s1 == 1) { mm = e / BK; kk = e % BK; } else { mm = e % BM; kk = e / BM; }
        const int64_t m = m0 + mm, k = k0 + kk;
        As[kk][mm] = (m < M && k < k_hi) ? ld_elem<BF16>(A, m * s0 + k * s1) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < (BK * BN) / NT; ++i) {
        const int e = tid + i * NT;
        int kk, nn;
        if (t1 == 1) { kk = e / BN; nn = e % BN; } else { kk = e % BK; nn = e / BK; }
        const int64_t k = k0 + kk, n = n0 + nn;
        Bs[kk][nn] = (n < Nn && k < k_hi) ? ld_elem<BF16>(B, k * t0 + n * t1) : 0.f;
    }
}

__device__ __forceinline__ void mma_tile(const float (*As)[BM + 4], const float (*Bs)[BN + 4],
                                         float acc[4][4], int ty, int tx)
{
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
        float a[4], b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

// is channel c in the sorted list sel[0..n)?  (sel == null: S = {0..n-1})
__device__ __forceinline__ bool in_sorted(const int32_t *sel, int64_t n, int64_t c)
{
    if (sel == nullptr) return c < n;
    int64_t lo = 0, hi = n;
    while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (sel[mid] < c) lo = mid + 1; else hi = mid;
    }
    return lo < n && sel[lo] == c;
}

template <bool BF16>
__global__ void __launch_bounds__(NT)
rowpar_fwd_simt_kernel(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                       const void *W, int64_t w_rs, int64_t w_cs, MutPtrs Y, int64_t ldy,
                       const int32_t *__restrict__ sel, int64_t n_sel)
{
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ unsigned char inS[BN];
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int64_t kt = K / t;
    if (tid < BN) inS[tid] = (n0 + tid < h) ? (unsigned char)in_sorted(sel, n_sel, n0 + tid) : 0;
    __syncthreads();

    float sum[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sum[i][j] = 0.f;

    for (int r = 0; r < t; ++r) {
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        const int64_t k_lo = (int64_t)r * kt, k_hi = k_lo + kt;
        for (int64_t k0 = k_lo; k0 < k_hi; k0 += BK) {
            stage_tiles<BF16>(As, Bs, X, ldx, 1, W, w_rs, w_cs, m0, n0, k0, k_hi, N, h);
            __syncthreads();
            mma_tile(As, Bs, acc, ty, tx);
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = m0 + ty + 16 * i;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int nn = tx + 16 * j;
                const int64_t n = n0 + nn;
                if (inS[nn]) {
                    sum[i][j] = r == 0 ? acc[i][j] : sum[i][j] + acc[i][j];
                } else if (m < N && n < h) {
                    st_elem<BF16>(Y.p[r], m * ldy + n, acc[i][j]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty + 16 * i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int nn = tx + 16 * j;
            const int64_t n = n0 + nn;
            if (inS[nn] && m < N && n < h)
                for (int r = 0; r < t; ++r) st_elem<BF16>(Y.p[r], m * ldy + n, sum[i][j]);
        }
    }
}

template <bool BF16>
__global__ void __launch_bounds__(NT)
batched_gemm_simt_kernel(int64_t M, int64_t Nn, int64_t Kk, ConstPtrs A, int64_t sa0,
                         int64_t sa1, ConstPtrs B, int64_t sb0, int64_t sb1, MutPtrs C,
                         int64_t sc0, int64_t sc1)
{
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
    const int b = blockIdx.z;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int64_t k0 = 0; k0 < Kk; k0 += BK) {
        stage_tiles<BF16>(As, Bs, A.p[b], sa0, sa1, B.p[b], sb0, sb1, m0, n0, k0, Kk, M, Nn);
        __syncthreads();
        mma_tile(As, Bs, acc, ty, tx);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty + 16 * i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx + 16 * j;
            if (m < M && n < Nn) st_elem<BF16>(C.p[b], m * sc0 + n * sc1, acc[i][j]);
        }
    }
}

}  // namespace

caat_status launch_rowpar_fwd_simt(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                   const void *X, int64_t ldx, const void *W, int64_t w_rs,
                                   int64_t w_cs, const MutPtrs &Y, int64_t ldy,
                                   const int32_t *sel, int64_t n_sel, cudaStream_t s)
{
    if (N == 0 || h == 0) return CAAT_OK;
    const int64_t gx = (h + BN - 1) / BN, gy = (N + BM - 1) / BM;
    if (gy > 65535) return CAAT_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)gx, (unsigned)gy);
    if (dt == CAAT_BF16)
        rowpar_fwd_simt_kernel<true><<<grid, NT, 0, s>>>(t, N, K, h, X, ldx, W, w_rs, w_cs, Y, ldy, sel, n_sel);
    else
        rowpar_fwd_simt_kernel<false><<<grid, NT, 0, s>>>(t, N, K, h, X, ldx, W, w_rs, w_cs, Y, ldy, sel, n_sel);
    note_launch("rowpar_fwd_simt");
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

caat_status launch_batched_gemm_simt(const BatchedGemm &g, cudaStream_t s)
{
    if (g.M == 0 || g.Nn == 0 || g.batches == 0) return CAAT_OK;
    const int64_t gx = (g.Nn + BN - 1) / BN, gy = (g.M + BM - 1) / BM;
    if (gy > 65535 || g.batches > 65535) return CAAT_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)g.batches);
    if (g.dt == CAAT_BF16)
        batched_gemm_simt_kernel<true><<<grid, NT, 0, s>>>(g.M, g.Nn, g.Kk, g.A, g.sa0, g.sa1, g.B, g.sb0, g.sb1, g.C, g.sc0, g.sc1);
    else
        batched_gemm_simt_kernel<false><<<grid, NT, 0, s>>>(g.M, g.Nn, g.Kk, g.A, g.sa0, g.sa1, g.B, g.sb0, g.sb1, g.C, g.sc0, g.sc1);
    note_launch("batched_gemm_simt");
    return cudaGetLastError() == cudaSuccess ? CAAT_OK : CAAT_ERR_CUDA;
}

}  // namespace caat
