// Internal declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "caat.h"

#define CAAT_MAX_T 64
// Channel-membership bitmaps live in shared memory: h <= 2^18 channels = 32 KB.
#define CAAT_MAX_H_BITMAP (1 << 18)

namespace caat {

struct ConstPtrs { const void *p[CAAT_MAX_T]; };
struct MutPtrs { void *p[CAAT_MAX_T]; };

// bookkeeping visible through caat_last_kernel / caat_launch_count
void note_launch(const char *kernel_name, int launches = 1);

// Device error word (one per device, zeroed by caat_get_device_status).
int *device_error_word();          // device address for the current device, or null

int num_sms();                     // SM count of the current device (cached)

// Per-call host work done once per device and kernel: the kernel's dynamic
// shared-memory limit (set on first use) and, for cluster launches, how many
// clusters of the given shape can be co-resident (queried on first use; cfg's
// grid is ignored).  Both cache the answer per (device, kernel, size).
caat_status prepare_kernel_smem(const void *kern, int smem_bytes);
int max_active_clusters(const void *kern, const cudaLaunchConfig_t &cfg);   // < 1: none / error

// ---- standalone partial channel-reduce (pcr.cu)
caat_status launch_pcr(int t, int64_t N, int64_t h, caat_dtype dt,
                       const ConstPtrs &in, int64_t ld_in, const MutPtrs &out, int64_t ld_out,
                       bool in_place, const int32_t *sel, int64_t n_sel, cudaStream_t s);

// Sum over ranks of the first s channels only, into one bf16 [N, s] buffer
// (contiguous S; the same fold and rounding as launch_pcr's S channels).
caat_status launch_pcr_colsum(int t, int64_t N, int64_t s, const ConstPtrs &in, int64_t ld_in, void *out,
                              int64_t ld_out, cudaStream_t st);

// ---- SIMT (CUDA-core) GEMM paths (gemm_simt.cu)
// Row-parallel forward with the PCR epilogue, any strides, f32 or bf16.
caat_status launch_rowpar_fwd_simt(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                   const void *X, int64_t ldx, const void *W, int64_t w_rs,
                                   int64_t w_cs, const MutPtrs &Y, int64_t ldy,
                                   const int32_t *sel, int64_t n_sel, cudaStream_t s);

// Batched strided GEMM, C_b = A_b B_b, fp32 accumulate, one batch per rank.
// Element (i, j) of A_b is at A[b] + i*sa0 + j*sa1 (likewise B, C).
struct BatchedGemm {
    int batches;
    int64_t M, Nn, Kk;
    caat_dtype dt;
    ConstPtrs A; int64_t sa0, sa1;
    ConstPtrs B; int64_t sb0, sb1;
    MutPtrs C;   int64_t sc0, sc1;
};
caat_status launch_batched_gemm_simt(const BatchedGemm &g, cudaStream_t s);

// ---- tcgen05 tensor-core paths (gemm_tc.cu)
// Returns CAAT_ERR_UNSUPPORTED (without launching) when the shape/layout is not
// one the tensor-core kernel takes; the caller then picks another kernel.
// few tokens (1 <= N <= 8192, t <= 8): tensor cores with the operands swapped, one
// cluster of t shard-CTAs per (128-channel block, chunk of up to 128 tokens).
// Above 128 tokens it declines (CAAT_ERR_UNSUPPORTED) a grid of more than four
// CTAs per SM, where the tile kernel is the faster one.
caat_status launch_rowpar_fwd_skinny(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                     const void *W, int64_t ldw, const MutPtrs &Y, int64_t ldy,
                                     const int32_t *sel, int64_t n_sel, cudaStream_t s);

// YS == nullptr: the t outputs Y [N, h].  Otherwise the compact outputs (a
// contiguous S, sel == nullptr, n_sel a multiple of 64): YS [N, n_sel] (row
// stride ldys) once and Y = YN, t outputs [N, h - n_sel] (row stride ldy).
// A launch as a programmatic dependent of the previous launch in the stream
// (CAAT_PDL=0: a plain launch).  The kernel waits for that launch
// (griddepcontrol.wait) before it touches memory, so only its start-up overlaps
// the previous grid's end.  Launch errors are read by the caller.
template <typename... Params, typename... Args>
void launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    const char *env = std::getenv("CAAT_PDL");
    if (env == nullptr || std::strcmp(env, "0") != 0) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    (void)cudaLaunchKernelEx(&cfg, kern, args...);
}

caat_status launch_rowpar_fwd_tc(int t, int64_t N, int64_t K, int64_t h,
                                 const void *X, int64_t ldx, const void *W, int64_t ldw,
                                 const MutPtrs &Y, int64_t ldy,
                                 const int32_t *sel, int64_t n_sel, cudaStream_t s,
                                 void *YS = nullptr, int64_t ldys = 0);

// ---- few-token (decode) forward on the CUDA cores (decode.cu): 1 <= N <= 64,
// t in {1, 2, 4, 8, 16, 32}, bf16, W in the nn.Linear layout (row stride ldw).
caat_status launch_rowpar_fwd_decode(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                     const void *W, int64_t ldw, const MutPtrs &Y, int64_t ldy,
                                     const int32_t *sel, int64_t n_sel, cudaStream_t s);

// Debug check of an index list of S (api.cu): ascending, unique, in [0, h);
// active only with CAAT_CHECK_SEL=1.
caat_status check_sel_debug(const int32_t *sel, int64_t n_sel, int64_t h, cudaStream_t s);

// Tensor map for TMA (gemm_tc.cu): 128-byte swizzle, zero fill out of bounds;
// bf16 elements unless f32.
bool encode_tmap(CUtensorMap *tm, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, bool f32 = false);

// Tensor-core backward (gemm_tc_bwd.cu): dX and dW as two grouped tcgen05 GEMMs.
// W and dW in the nn.Linear layout ([h, K] storage, row strides ldw / ld_dw).
bool bwd_tc_supported(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                      const void *W, int64_t ldw, const ConstPtrs &dY, int64_t ld_dy, const void *dX,
                      int64_t lddx, const void *dW, int64_t ld_dw);
// wacc: fp32 scratch of h * K floats for a split reduction over tokens in dW
// (null: no split).  s_sum > 0: channels [0, s_sum) of every rank's gradient
// are read from the one reduced buffer dsum [N, s_sum] (row stride ld_dsum) and
// channels [s_sum, h) from dY_r; s_sum must be a multiple of 64.  own_compact:
// dY_r holds only channels [s_sum, h), at columns 0 .. h - s_sum - 1 (the compact
// form); otherwise dY_r is [N, h] and its first s_sum channels are not read.
// per host thread and device: a second stream and a fork / join event pair for
// running independent parts of one call side by side (null: stay on `main`)
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
SideStream *side_stream(cudaStream_t main);

caat_status launch_rowpar_bwd_tc(int t, int64_t N, int64_t K, int64_t h, const void *X, int64_t ldx,
                                 const void *W, int64_t ldw, const ConstPtrs &dY, int64_t ld_dy,
                                 void *dX, int64_t lddx, void *dW, int64_t ld_dw, float *wacc,
                                 int64_t s_sum, const void *dsum, int64_t ld_dsum, cudaStream_t s,
                                 bool own_compact = false, const int32_t *row_sel = nullptr,
                                 int64_t row_nsel = 0, void *dw_tmp = nullptr, void *w_perm = nullptr);

// bf16 rows [h, K] between channel order and the order "channels of S ascending,
// then the others" (sel: S, ascending, n_sel): to_s_first moves row c of src to
// row s_first_pos(c) of dst, else row s_first_pos(c) of src to row c of dst.
// row_sel in launch_rowpar_bwd_tc undoes that order on dW's rows: through the
// fp32 accumulator when dW is split over tokens, else through dw_tmp (bf16 [h, K],
// row stride K), which it then requires.  With w_perm (bf16 [h, K]) it first puts
// W's rows into that order there, for dX.
caat_status launch_permute_rows(const void *src, int64_t lds, void *dst, int64_t ldd, int64_t h, int64_t K,
                                const int32_t *sel, int64_t n_sel, bool to_s_first, cudaStream_t s);

}  // namespace caat
