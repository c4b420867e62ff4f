/*
 * caat.h -- C ABI of the GB300 (sm_103a) partial channel-reduce library.
 *
 * The operation comes from "Tensor-Parallelism with Partially Synchronized
 * Activations" (Lamprecht et al., NeurIPS 2025), Introduction, the paragraph that
 * defines the partial channel-reduce (PCR): after a tensor-parallel (row-parallel)
 * layer, only a subset S of the hidden channels is summed over the t ranks; on the
 * other channels each rank keeps the partial result it computed, so activations
 * differ across ranks.  S empty is the "ensemble" limit, S = all channels is the
 * vanilla all-reduce.  The same paragraph requires the backward pass to match the
 * forward.  The experimental setup fixes the size of S by the fraction p
 * (p = 0.5 with tensor-parallel dimension 8 for the 7B model).
 *
 * On one GPU the t ranks are emulated as t shards resident in the same memory.
 *
 * Conventions shared by every call
 *  - Every compute call is asynchronous on the stream `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and keeps no data between calls.  The
 *    backward calls may run part of their work on a library-owned side stream
 *    (one per host thread and device, created on first use outside stream
 *    capture): it forks from `stream` and joins back to it through events, so
 *    the call stays ordered on `stream` and can be captured in a CUDA graph.
 *    A caller that drives one host thread on several streams at once shares
 *    that side stream between them (still correct, possibly less concurrent).
 *  - Tuning switches read from the environment at each call (for comparisons
 *    and tests; the defaults choose by shape): CAAT_FWD_CLUSTER=1|2 (CTAs per
 *    cluster of the forward tile kernel), CAAT_FWD_BN=192|256 (its tile width),
 *    CAAT_FWD_ORDER=m|n (its work units row- or channel-block-major),
 *    CAAT_FWD_SCHED=rounds|first (every tile of it whole, in rounds, instead of
 *    cutting the tiles outside S into per-shard pieces that even out the SMs'
 *    load; or the whole tiles first and the pieces after them, instead of the
 *    pieces in runs around each worker's whole tiles),
 *    CAAT_FWD_STG=1 (one staging buffer per epilogue warp in the 256-wide tiles
 *    instead of two where shared memory allows), CAAT_FWD_DEEP=0|1 (the 192-wide
 *    single-CTA tiles with 4 ring stages and two staging buffers, or 5 stages and
 *    one; by default 5 for shards of 4 or more k-blocks), CAAT_FWD_WGT=1..t (the
 *    pieces a whole tile's time is worth in the balanced schedule; by default t,
 *    and for the compact outputs min(t, k-blocks per shard / 2 + 2)),
 *    CAAT_FWD_SKINNY=0 (no few-token tensor-core kernel), CAAT_FWD_SKINNY_MAX=n
 *    (the most tokens it takes: by default 256 for a contiguous S given by its
 *    size, 128 for an index list; above 128 it runs chunks of 128 tokens and
 *    declines a grid of more than four CTAs per SM), CAAT_BWD_SIDE_STREAM=0
 *    (backward on `stream` only), CAAT_BWD_RING=4 (the backward GEMMs' ring at 4
 *    stages whatever the tile width; single CTAs only), CAAT_BWD_PAIR=0 (the
 *    backward GEMMs on single CTAs instead of CTA pairs), CAAT_PDL=0 (the
 *    forward kernels, the backward GEMMs, the sum of the gradient's S channels
 *    and the standalone reduce launched plainly instead of as programmatic
 *    dependents of the previous launch in the stream, whose blocks may then start
 *    while that launch finishes; they wait for it before they touch memory).
 *  - CAAT_CHECK_SEL=1 (a debug switch) checks every index list of S: the list is
 *    copied to the host on the call's stream, which is synchronised, and must be
 *    ascending, unique and inside [0, h), else the call returns INVALID_ARG
 *    before anything is launched.  Without it the list is trusted (an invalid
 *    list gives undefined channel sets).  The check is skipped while the stream
 *    is being captured into a graph.
 *  - CAAT_PDL_WEIGHTS=1 is an opt-in for inference with static weights: the
 *    few-token kernel then reads the weight tiles of its first ring stages before
 *    waiting for the previous launch in the stream (X, S and the outputs still
 *    wait).  Set it only when no kernel launched right before a call writes that
 *    call's weights; otherwise the call may read stale weights.
 *  - bf16 layer work that no tensor-core kernel takes (for example a weight that
 *    is not K-contiguous, a shard width k_t that is not a multiple of 8, more
 *    than 16 ranks beyond a few tokens, pointers off 16 bytes) returns
 *    UNSUPPORTED, before anything is launched, unless CAAT_ALLOW_FALLBACK=1 is in
 *    the environment at the call: then it runs on the CUDA-core (FFMA) kernels,
 *    correct but one to two orders of magnitude slower.  fp32 always runs there
 *    (it has no tensor-core path).  Empty work (N, K or h zero) needs no opt-in.
 *  - "device pointer" = memory the caller allocated on the current CUDA device;
 *    the library never allocates or frees device memory and never keeps a pointer
 *    after the call returns.  Arrays "of t device pointers" are HOST arrays whose
 *    entries are device pointers; the library copies them before returning.
 *  - Matrices are dense in their last dimension unless a stride says otherwise;
 *    strides and leading dimensions are in ELEMENTS, not bytes.
 *  - Arguments are validated before anything is launched.  On any error nothing
 *    is written and nothing is launched.
 *  - bf16 data is stored as 16-bit words; all arithmetic accumulates in fp32.
 *  - No C++ exception crosses this interface.
 *  - Per device, the library sets each kernel's shared-memory limit and looks up
 *    its cluster occupancy once, on the kernel's first launch, and keeps the
 *    answers for the life of the process.  They do not survive cudaDeviceReset:
 *    a process that resets a device should not call the library on it again.
 */
#ifndef CAAT_H
#define CAAT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *caat_stream_t;

typedef enum {
    CAAT_OK = 0,
    CAAT_ERR_INVALID_ARG = 1,  /* a null pointer, a size or stride out of range       */
    CAAT_ERR_UNSUPPORTED = 2,  /* valid, but no kernel of this build takes it         */
    CAAT_ERR_CUDA = 3,         /* a CUDA runtime call or a launch failed              */
    CAAT_ERR_TIMEOUT = 4       /* a bounded device-side wait gave up (see below)      */
} caat_status;

typedef enum { CAAT_F32 = 0, CAAT_BF16 = 1 } caat_dtype;

/* Which channels make up S.  The paper fixes only its size. */
typedef enum {
    CAAT_S_CONTIGUOUS = 0,     /* S = {0, ..., s-1}                                   */
    CAAT_S_RANDOM = 1          /* first s entries of a seeded Fisher-Yates shuffle    */
} caat_layout;

/* Where the backward reduce sits (the paper requires only that it match the forward). */
typedef enum {
    CAAT_BWD_REDUCE_DOUT = 0,  /* dY = PCR(dOut): exact gradient of sum_r <dOut_r, Out_r> */
    CAAT_BWD_NO_REDUCE = 1     /* dY_r = dOut_r: the reduce is done by the matching       */
                               /* column-parallel layer's input gradient                   */
} caat_bwd_mode;

/*
 * caat_select_channels -- the synchronized channel set S (host only, no GPU).
 *
 * Paper: Introduction (PCR reduces "a subset of the channels"); experimental
 * setup (hyper-parameter p, the reduced fraction; p = 0.5).
 * s = floor(p*h + 1/2), clamped to [0, h].
 *   CAAT_S_CONTIGUOUS: S = {0..s-1}.
 *   CAAT_S_RANDOM:     permutation pi of {0..h-1} by Fisher-Yates, i = h-1 down to
 *                      1, j = splitmix64_next() mod (i+1), swap pi[i], pi[j]; the
 *                      splitmix64 state starts at `seed`.  S = sort(pi[0..s)).
 *                      Sets are nested: S(p1) is a subset of S(p2) when p1 <= p2.
 * idx:   host int32[h] written with S in ascending order (caller allocates h entries).
 * n_sel: host, receives s.
 * Errors: INVALID_ARG for h < 0 or h > 2^31-1, p outside [0,1] or NaN, an unknown
 * layout, or a null pointer (idx may be null when h == 0).
 */
caat_status caat_select_channels(int64_t h, double p, caat_layout layout, uint64_t seed,
                                 int32_t *idx, int64_t *n_sel);

/*
 * caat_partial_channel_reduce -- standalone PCR over t partial tensors.
 *
 * Paper: Introduction, definition of the partial channel-reduce.
 *   out_r[n, c] = in_0[n, c] + in_1[n, c] + ... + in_{t-1}[n, c]   if c in S
 *   out_r[n, c] = in_r[n, c]                                       otherwise
 * The sum is a left fold in rank order in fp32 (bit-reproducible); bf16 data is
 * widened exactly and rounded once (nearest-even) to bf16 at the end.
 * t:      1 .. 64 ranks.      N: rows (tokens), >= 0.    h: channels, 0 .. 2^24.
 * in:     host array of t device pointers, each [N, h] with row stride ld_in.
 * out:    host array of t device pointers, each [N, h] with row stride ld_out.
 *         out may equal in (in place: then only the channels of S are written).
 *         Otherwise the t outputs must not overlap any input.  No output may
 *         overlap sel.
 * sel:    device int32[n_sel], ascending, unique, each in [0, h)  (S);
 *         or null, which means the contiguous S = {0, ..., n_sel-1}.
 * Errors: INVALID_ARG for t out of range, negative sizes, ld < h, null pointers,
 *         or in/out arrays that are in place for some ranks and not for others.
 *         Unsorted or out-of-range entries of sel are not checked on the device;
 *         out-of-range entries are ignored by the kernel, duplicates are harmless.
 */
caat_status caat_partial_channel_reduce(int t, int64_t N, int64_t h, caat_dtype dt,
                                        const void *const *in, int64_t ld_in,
                                        void *const *out, int64_t ld_out,
                                        const int32_t *sel, int64_t n_sel,
                                        caat_stream_t stream);

/*
 * caat_rowpar_linear_fwd -- row-parallel linear layer fused with the PCR.
 *
 * Paper: Introduction (the PCR replaces the all-reduce that follows the
 * tensor-parallel block: attention out-projection, MLP down-projection).
 * K splits into t equal shards k_t = K/t; rank r owns X[:, r*k_t .. (r+1)*k_t)
 * and rows r*k_t .. (r+1)*k_t of W.  With Y_r = X_r W_r:
 *   Y[r][n, c] = Y_0[n, c] + ... + Y_{t-1}[n, c]  (= (X W)[n, c], full K)  if c in S
 *   Y[r][n, c] = Y_r[n, c]                                              otherwise
 * X:   device [N, K], row stride ldx.
 * W:   device, logical [K, h]: element (k, c) at W[k*w_rs + c*w_cs].
 *      (w_rs, w_cs) = (1, K) is torch's nn.Linear weight [h, K] (K contiguous),
 *      the layout the tensor-core path takes; (h, 1) is a row-major [K, h].
 * Y:   host array of t device pointers, each [N, h] with row stride ldy; they
 *      must not overlap each other, X, W or sel (else INVALID_ARG).
 * sel: device int32[n_sel], ascending and unique (S); or null for the contiguous
 *      S = {0, ..., n_sel-1}.  With the contiguous form and n_sel a multiple of 64,
 *      the backward reduces only the S channels, once, instead of materialising
 *      every rank's reduced gradient.  An index list of all h channels can only be
 *      {0, ..., h-1} and takes the contiguous paths.
 * Precision: bf16 in, fp32 accumulate, one rounding to bf16; or fp32 throughout
 * (fp32 FMA, no TF32).  One exception: with an index list of S (0 < n_sel < h)
 * the tile kernel (the calls the few-token kernel does not take) writes every
 * rank's whole partial first and the S channels then sum those bf16 partials in
 * rank order (fp32 fold, one more rounding), so they may differ from the
 * one-rounding sum by up to half an ulp of each partial.
 * Errors: INVALID_ARG for t outside 1..64, K % t != 0, negative sizes, a stride
 *         or leading dimension smaller than the row it spans, null pointers.
 *         UNSUPPORTED when no kernel takes the layout and alignment given (for
 *         bf16: no tensor-core kernel, and CAAT_ALLOW_FALLBACK is not 1).
 */
caat_status caat_rowpar_linear_fwd(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                   const void *X, int64_t ldx,
                                   const void *W, int64_t w_rs, int64_t w_cs,
                                   void *const *Y, int64_t ldy,
                                   const int32_t *sel, int64_t n_sel,
                                   caat_stream_t stream);

/*
 * caat_rowpar_linear_bwd -- gradients of the fused row-parallel layer.
 *
 * Paper: Introduction (forward and backward must agree; a mismatch diverges).
 * dOut: host array of t device pointers, each [N, h] with row stride ld_dout:
 *       the gradient arriving at each rank's output Y[r].
 * mode CAAT_BWD_REDUCE_DOUT: dY = PCR(dOut) with the same S (PCR is symmetric,
 *       so this is the exact gradient of sum_r <dOut_r, Y[r]>);
 * mode CAAT_BWD_NO_REDUCE:   dY_r = dOut_r.
 * Writes dX [N, K] (row stride lddx; shard r = columns r*k_t..) with
 *   dX[:, shard r] = dY_r W_r^T,
 * and dW, logical [K, h] with element (k, c) at dW[k*dw_rs + c*dw_cs], with
 *   dW[shard r, :] = X_r^T dY_r.
 * workspace: device scratch, 256-byte aligned, owned by the caller and no longer
 *       used once the stream passes the end of this call.  Its layout:
 *         [ reduced gradient: t buffers of [N, h], each rounded up to 256 bytes ]
 *           -- required in CAAT_BWD_REDUCE_DOUT mode when S is not empty and t > 1;
 *         [ fp32 accumulator of dW, [h, K], rounded up to 256 bytes ]
 *           -- optional (bf16 only): with it dW is reduced over tokens in several
 *              parts on more SMs, then rounded once to bf16.
 *       caat_rowpar_linear_bwd_workspace() returns the size of both parts; a
 *       workspace holding only the required part also works.  May be null when
 *       nothing is required.
 * Errors: as caat_rowpar_linear_fwd; INVALID_ARG also when ws_bytes is too small,
 *   or when dX, dW and the part of the workspace the call uses overlap each other
 *   or any input (X, W, a dOut_r, sel).
 */
size_t caat_rowpar_linear_bwd_workspace(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                        caat_bwd_mode mode);

caat_status caat_rowpar_linear_bwd(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                   const void *X, int64_t ldx,
                                   const void *W, int64_t w_rs, int64_t w_cs,
                                   const void *const *dOut, int64_t ld_dout,
                                   void *dX, int64_t lddx,
                                   void *dW, int64_t dw_rs, int64_t dw_cs,
                                   const int32_t *sel, int64_t n_sel, caat_bwd_mode mode,
                                   void *workspace, size_t ws_bytes,
                                   caat_stream_t stream);

/*
 * caat_rowpar_linear_fwd_compact -- caat_rowpar_linear_fwd with the t outputs in
 * compact form: the channels of S, which hold the same sum on every rank, are
 * stored once.
 *
 * Paper: Introduction (PCR: every rank gets the sum on S and keeps its own
 * partial elsewhere).  With the t ranks' outputs in one GPU's memory the t copies
 * of the S channels carry nothing beyond one of them.  With S = {s_0 < s_1 < ...}
 * and its complement {u_0 < u_1 < ...} this call writes
 *   YS[n, j]    = Y[r][n, s_j]      (the same for every r)
 *   YN[r][n, j] = Y[r][n, u_j]
 * with Y[r] as defined for caat_rowpar_linear_fwd: N*|S| + t*N*(h-|S|) elements
 * written instead of t*N*h.
 * YS:    device [N, n_sel], row stride ldys (unused when n_sel == 0).
 * YN:    host array of t device pointers, each [N, h - n_sel], row stride ldyn
 *        (unused when n_sel == h).  No output may overlap another, X, W, sel or
 *        the workspace.
 * sel, n_sel: S as for caat_rowpar_linear_fwd (null: the first n_sel channels).
 *        n_sel must be a multiple of 64 (else UNSUPPORTED), so that every
 *        64-channel chunk of a tile lies in S or outside it.
 * workspace: required only for an index list with 0 < n_sel < h: a copy of W
 *        with its channels in the order "S first" (which makes S contiguous for
 *        the kernel), h*K*2 bytes, 256-byte aligned;
 *        caat_rowpar_linear_compact_workspace(..., index_list = 1, backward = 0)
 *        gives the size.  Else it may be null.  The copy costs one read and one
 *        write of W per call.
 * Kernel: the tensor-core tile kernel only: bf16, W in the nn.Linear layout
 *        (w_rs == 1), N >= 16, k_t >= 64 and a multiple of 8, 16-byte aligned
 *        bases, row strides that are multiples of 8 elements.  Other shapes return
 *        UNSUPPORTED (the few-token kernels have no compact form); with an index
 *        list the workspace may have been written by then.
 * Errors: INVALID_ARG as caat_rowpar_linear_fwd (null or short outputs, overlaps,
 *        a workspace that is missing, short or misaligned); UNSUPPORTED as above.
 */
caat_status caat_rowpar_linear_fwd_compact(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                           const void *X, int64_t ldx,
                                           const void *W, int64_t w_rs, int64_t w_cs,
                                           void *YS, int64_t ldys, void *const *YN, int64_t ldyn,
                                           const int32_t *sel, int64_t n_sel,
                                           void *workspace, size_t ws_bytes, caat_stream_t stream);

/*
 * caat_rowpar_linear_bwd_compact -- gradients of caat_rowpar_linear_fwd_compact.
 *
 * dYS: device [N, n_sel], row stride lddys: the gradient arriving at YS.  YS is
 *      shared by every rank's downstream computation, so dYS already is the sum
 *      over the ranks of their gradients on S.
 * dYN: host array of t device pointers, each [N, h - n_sel], row stride lddyn:
 *      the gradient arriving at YN[r].
 * With dY_r the [N, h] gradient that holds dYS on the channels of S and dYN[r] on
 * the others (each in ascending channel order) this writes
 *   dX[:, shard r] = dY_r W_r^T   and   dW[shard r, :] = X_r^T dY_r,
 * which is caat_rowpar_linear_bwd in CAAT_BWD_REDUCE_DOUT mode for any dOut whose
 * S channels sum over the ranks to dYS and whose other channels are dYN[r]: the
 * reduce of the gradient has already happened.
 * workspace: 256-byte aligned, caat_rowpar_linear_compact_workspace(..., backward
 *      = 1) bytes.  For an index list with 0 < n_sel < h it starts with two
 *      required parts of h*K*2 bytes each (rounded to 256): W in the S-first
 *      order, and room to stage dW in that order before its rows return to
 *      channel order.  Then, for any S, the optional fp32 accumulator of dW,
 *      h*K*4 bytes rounded to 256.  With the accumulator, dW is reduced over
 *      tokens in several parts when its tiles do not fill the SMs; then rounded
 *      once.  With a contiguous S the workspace may be null.
 * Kernel: the tensor-core backward only: bf16, W and dW in the nn.Linear layout
 *      (w_rs == dw_rs == 1), N >= 128, h >= 256, n_sel a multiple of 64, the TMA
 *      alignment rules; else UNSUPPORTED.
 * Errors: INVALID_ARG as caat_rowpar_linear_bwd (dX, dW and the workspace must not
 *      overlap each other or an input; a required workspace missing or short).
 */
caat_status caat_rowpar_linear_bwd_compact(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                           const void *X, int64_t ldx,
                                           const void *W, int64_t w_rs, int64_t w_cs,
                                           const void *dYS, int64_t lddys,
                                           const void *const *dYN, int64_t lddyn,
                                           void *dX, int64_t lddx,
                                           void *dW, int64_t dw_rs, int64_t dw_cs,
                                           const int32_t *sel, int64_t n_sel,
                                           void *workspace, size_t ws_bytes,
                                           caat_stream_t stream);

/* Workspace bytes of the compact calls: index_list != 0 for an index list of S
 * with 0 < |S| < h, backward != 0 for caat_rowpar_linear_bwd_compact (whose part
 * for the dW accumulator is included).  0 for invalid arguments. */
size_t caat_rowpar_linear_compact_workspace(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                            int index_list, int backward);

/*
 * caat_rowpar_linear_bwd_noalloc -- caat_rowpar_linear_bwd without a caller
 * workspace.  The paper has no counterpart: this entry point exists for callers
 * that cannot call cudaMalloc (for example a host framework that owns all device
 * memory through its own pool allocator and forbids side allocations, or a
 * process whose memory budget is fixed at start-up).
 *
 * Instead of a caller-provided workspace it uses one library-owned device array
 * of CAAT_NOALLOC_SCRATCH_BYTES (16 MiB), declared at file scope in the library;
 * every GPU that loads the library holds that array until the process exits.
 * The call itself allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.
 *  - Arguments and results are exactly those of caat_rowpar_linear_bwd (same
 *    pointers, strides and modes), minus workspace / ws_bytes.
 *  - Size limit: in CAAT_BWD_REDUCE_DOUT mode with S not empty and t > 1 the
 *    reduced gradient needs t * N * h * (2 for bf16, 4 for fp32) bytes of scratch
 *    (each rank's part rounded up to 256 bytes); above 16 MiB the call returns
 *    CAAT_ERR_INVALID_ARG and launches nothing (use caat_rowpar_linear_bwd with a
 *    workspace instead).  CAAT_BWD_NO_REDUCE, an empty S or t == 1 need no
 *    scratch.  When the rest of the array also holds the optional fp32 dW
 *    accumulator (h * K * 4 bytes), it is used for it as well.
 *  - Every call that needs the scratch looks up the array's device address
 *    (cudaGetSymbolAddress, no allocation) on the current device, so the call
 *    stays valid after a cudaDeviceReset has moved the array.  The first call on
 *    a device loads the array with the module: make it before any stream capture.
 *  - All calls in the process share the one array, which keeps the last call's
 *    contents.  Calls whose work overlaps on the GPU (different streams, or other
 *    host threads, without ordering between them) race on it and corrupt each
 *    other's results: order them on one stream or with events.  Nothing in the
 *    array has to start at zero: each call writes every byte it later reads.
 */
#define CAAT_NOALLOC_SCRATCH_BYTES (16u << 20)

caat_status caat_rowpar_linear_bwd_noalloc(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                           const void *X, int64_t ldx,
                                           const void *W, int64_t w_rs, int64_t w_cs,
                                           const void *const *dOut, int64_t ld_dout,
                                           void *dX, int64_t lddx,
                                           void *dW, int64_t dw_rs, int64_t dw_cs,
                                           const int32_t *sel, int64_t n_sel, caat_bwd_mode mode,
                                           caat_stream_t stream);

/*
 * The column-parallel partner of the layer above (attention QKV, MLP up), for
 * Megatron's placement of the backward reduce: the row-parallel backward runs in
 * CAAT_BWD_NO_REDUCE mode and the partial channel-reduce moves to this layer's
 * input gradient ("Tensor-Parallelism with Partially Synchronized Activations",
 * Introduction: the reduce of forward and backward must agree).  Reading: the
 * input channels in S are one activation shared by the ranks, so their gradient
 * is the sum of the ranks' contributions; outside S each rank's input is its own.
 *
 * Layouts (elements, row-major unless strides say otherwise):
 *   A:  array of t device pointers; A[r] is rank r's input [N, h], row stride lda
 *       (under partial synchronization the ranks' inputs differ).
 *   W1: logical [h, K]; element (c, k) at W1[c*w1_rs + k*w1_cs].  Rank r owns the
 *       column block W1_r = W1[:, r*k_t .. (r+1)*k_t), k_t = K/t.
 *       This is the row-parallel W's [h, K] storage with the roles of the two
 *       dimensions swapped: K-contiguous (w1_cs == 1) takes the tensor cores.
 *   Z / dZ: [N, K], row stride ldz; column block r is rank r's output.
 *
 * caat_colpar_linear_fwd:  Z[:, block r] = A_r W1_r.  No reduce.
 * caat_colpar_linear_bwd:
 *   dA_r            = PCR_S(dZ_r W1_r^T)   (t buffers [N, h], row stride ldda):
 *                     c in S: sum over q of dZ_q W1_q^T[:, c]; otherwise rank r's own;
 *   dW1[:, block r] = A_r^T dZ_r            (element (c, k) at dW1[c*dw1_rs + k*dw1_cs]).
 *   dA is computed by the fused row-parallel forward kernel (dZ W1^T is
 *   row-parallel shaped), dW1 by the grouped backward GEMM.
 *   workspace: optional device scratch, 256-byte aligned, of at least
 *   caat_colpar_linear_bwd_workspace() bytes (bf16: an fp32 accumulator of dW1 that
 *   lets dW1 be reduced over tokens in parts); null is allowed.
 * Ownership: all buffers belong to the caller; nothing is kept after the call.
 * Errors: INVALID_ARG for a bad size, null pointer, stride below the row width,
 *   K % t != 0, n_sel outside [0, h], or outputs overlapping inputs (Z with any A_r
 *   or W1; dA_r with each other, any A_q, dZ, W1 or sel; dW1 and the fp32
 *   accumulator the call uses with each other and with every other buffer of the
 *   call); UNSUPPORTED / CUDA as
 *   caat_rowpar_linear_fwd.  sel as there (null = the first n_sel channels).
 *   The backward computes dW1 before dA: when only dA's product is declined
 *   (UNSUPPORTED), dW1 and the accumulator may already have been written.
 */
caat_status caat_colpar_linear_fwd(int t, int64_t N, int64_t h, int64_t K, caat_dtype dt,
                                   const void *const *A, int64_t lda,
                                   const void *W1, int64_t w1_rs, int64_t w1_cs,
                                   void *Z, int64_t ldz, caat_stream_t stream);

size_t caat_colpar_linear_bwd_workspace(int t, int64_t N, int64_t h, int64_t K, caat_dtype dt);

caat_status caat_colpar_linear_bwd(int t, int64_t N, int64_t h, int64_t K, caat_dtype dt,
                                   const void *const *A, int64_t lda,
                                   const void *W1, int64_t w1_rs, int64_t w1_cs,
                                   const void *dZ, int64_t ldz,
                                   void *const *dA, int64_t ldda,
                                   void *dW1, int64_t dw1_rs, int64_t dw1_cs,
                                   const int32_t *sel, int64_t n_sel,
                                   void *workspace, size_t ws_bytes, caat_stream_t stream);

/*
 * The partial channel-reduce across processes, one GPU each.  "Tensor-Parallelism
 * with Partially Synchronized Activations", Introduction: the partial
 * channel-reduce replaces the all-reduce after a row-parallel layer; only the
 * channels of S are summed over the ranks, the others stay on their rank.  Across
 * GPUs that sum is an all-reduce of an [N, |S|] buffer, which the caller's
 * collectives move; these three calls are the steps that run on each GPU:
 *   1. caat_pcr_pack:   P[n, i] = Y[n, S_i]        (the send buffer, dense)
 *   2. the collectives give each rank a block of rows of every rank's P;
 *      caat_rank_fold sums them in rank order      (fp32 left fold, one rounding)
 *   3. the collectives gather the folded rows; caat_pcr_unpack writes them back:
 *      Y_k[n, S_i] = P[n, i] for each of the n_out outputs of this process.
 * The fold order makes the result independent of how the rows were split.
 *
 * Common to the three: asynchronous on `stream`, device pointers owned by the
 * caller, strides in elements, bf16 or fp32 elements moved bit for bit (the fold
 * widens bf16 exactly and rounds once).  sel: device int32[n_sel], the channels of
 * S in [0, h) (ascending, unique), or null for S = {0, ..., n_sel-1}.  Errors:
 * INVALID_ARG for negative sizes, n_sel > h, a leading dimension below its row
 * width, null pointers where data is moved, or written buffers that overlap the
 * buffers they are computed from (or sel, or each other).  Out-of-range entries
 * of sel are not checked on the device.
 */
/* Y: [N, h], row stride ldy.  P: [N, n_sel], row stride ldp (>= n_sel). */
caat_status caat_pcr_pack(int64_t N, int64_t h, caat_dtype dt, const void *Y, int64_t ldy,
                          const int32_t *sel, int64_t n_sel, void *P, int64_t ldp,
                          caat_stream_t stream);

/* P: [N, n_sel], row stride ldp.  Y: host array of n_out (1 .. 64) device
 * pointers, each [N, h] with row stride ldy; only the channels of S are written. */
caat_status caat_pcr_unpack(int64_t N, int64_t h, caat_dtype dt, const void *P, int64_t ldp,
                            const int32_t *sel, int64_t n_sel, void *const *Y, int n_out,
                            int64_t ldy, caat_stream_t stream);

/* in: t (1 .. 4096) blocks of [rows, cols], row stride ld_in, block q starting
 * rank_stride elements after block q-1 (>= the span of one block).
 * out[n, c] = in_0[n, c] + in_1[n, c] + ... + in_{t-1}[n, c] (row stride ld_out). */
caat_status caat_rank_fold(int t, int64_t rows, int64_t cols, caat_dtype dt, const void *in,
                           int64_t ld_in, int64_t rank_stride, void *out, int64_t ld_out,
                           caat_stream_t stream);

/* Human-readable name of a status code (static string, never null). */
const char *caat_status_string(caat_status st);

/*
 * caat_get_device_status -- synchronizes `stream`, then reports and clears the
 * library's device-side error word of the current device.  Every wait inside the
 * tensor-core kernels is bounded; a wait that gives up records CAAT_ERR_TIMEOUT
 * there and the kernel exits (its outputs are then undefined) instead of hanging.
 * Returns CAAT_ERR_CUDA when the synchronization itself fails.
 */
caat_status caat_get_device_status(caat_stream_t stream);

/*
 * caat_debug_set_wait -- test hook for the device-side failure path.  Not part of
 * the computation; production code leaves it alone.
 *
 * Sets, for every later launch of the forward tile kernel (the tcgen05 kernel
 * that caat_rowpar_linear_fwd uses from 65 tokens up, and caat_colpar_linear_bwd
 * through it), the limit of each of its mbarrier waits (limit_ns; 0 restores the
 * default of 2 s; else 1 us .. 10 s) and an injected failure:
 *   CAAT_INJECT_NONE        normal operation;
 *   CAAT_INJECT_SKIP_LOADS  the kernel's TMA producer issues no load, so the MMA
 *                           issuer's first wait for operands can never complete.
 *                           That wait gives up after limit_ns, the kernel records
 *                           CAAT_ERR_TIMEOUT, every role leaves its loop, and the
 *                           CTA exits after releasing its TMEM.  The outputs are
 *                           then undefined; caat_get_device_status reports (and
 *                           clears) the timeout.  Nothing is in flight when the
 *                           kernel ends: no copy and no MMA was ever issued.
 * The setting is process-wide and read at each launch.  Errors: INVALID_ARG for a
 * limit outside the range or an unknown injection.
 */
typedef enum { CAAT_INJECT_NONE = 0, CAAT_INJECT_SKIP_LOADS = 1 } caat_inject;

caat_status caat_debug_set_wait(uint64_t limit_ns, caat_inject inject);

/*
 * caat_last_kernel -- which kernel the last successful call on this host thread
 * used (static string, e.g. "pcr_vec", "rowpar_fwd_tc", "rowpar_fwd_simt"); for a
 * call that launches several kernels, its main one.  For tests and benchmarks.
 */
const char *caat_last_kernel(void);

/* Number of kernels this host thread has launched through the library so far. */
uint64_t caat_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* CAAT_H */
