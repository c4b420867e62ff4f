// C-ABI entry points: argument validation, kernel choice, launch bookkeeping.
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "caat_internal.h"

namespace caat {

namespace {
thread_local const char *t_last_kernel = "none";
thread_local uint64_t t_launches = 0;
int g_sms[128];
std::mutex g_mu;
}  // namespace

// Debug check of an index list of S (CAAT_CHECK_SEL=1): the list is copied to
// the host on the call's stream, which is then synchronised, and must be
// ascending, unique and inside [0, h).  Skipped while the stream is being
// captured (a synchronising copy cannot be captured) and for the contiguous form.
caat_status check_sel_debug(const int32_t *sel, int64_t n_sel, int64_t h, cudaStream_t s)
{
    const char *env = std::getenv("CAAT_CHECK_SEL");
    if (env == nullptr || std::strcmp(env, "1") != 0 || sel == nullptr || n_sel <= 0) return CAAT_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return CAAT_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return CAAT_OK;
    std::vector<int32_t> host((size_t)n_sel);
    if (cudaMemcpyAsync(host.data(), sel, (size_t)n_sel * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CAAT_ERR_CUDA;
    for (int64_t i = 0; i < n_sel; ++i) {
        if (host[(size_t)i] < 0 || host[(size_t)i] >= h) return CAAT_ERR_INVALID_ARG;
        if (i > 0 && host[(size_t)i] <= host[(size_t)i - 1]) return CAAT_ERR_INVALID_ARG;
    }
    return CAAT_OK;
}

void note_launch(const char *kernel_name, int launches)
{
    t_last_kernel = kernel_name;
    t_launches += (uint64_t)launches;
}

int num_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

namespace {
struct KernelKey {
    int dev;
    const void *kern;
    int a, b;
};
std::mutex g_kmu;
KernelKey g_smem_done[256];
int g_n_smem = 0;
struct ClusterEntry {
    KernelKey k;
    int active;
};
ClusterEntry g_clusters[256];
int g_n_clusters = 0;
}  // namespace

caat_status prepare_kernel_smem(const void *kern, int smem_bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CAAT_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_kmu);
    for (int i = 0; i < g_n_smem; ++i)
        if (g_smem_done[i].dev == dev && g_smem_done[i].kern == kern && g_smem_done[i].a >= smem_bytes)
            return CAAT_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return CAAT_ERR_CUDA;
    if (g_n_smem < 256) g_smem_done[g_n_smem++] = {dev, kern, smem_bytes, 0};
    return CAAT_OK;
}

int max_active_clusters(const void *kern, const cudaLaunchConfig_t &cfg)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int cl = 1;
    for (unsigned i = 0; i < cfg.numAttrs; ++i)
        if (cfg.attrs[i].id == cudaLaunchAttributeClusterDimension) cl = (int)cfg.attrs[i].val.clusterDim.x;
    const int smem = (int)cfg.dynamicSmemBytes;
    std::lock_guard<std::mutex> lk(g_kmu);
    for (int i = 0; i < g_n_clusters; ++i) {
        const KernelKey &k = g_clusters[i].k;
        if (k.dev == dev && k.kern == kern && k.a == cl && k.b == smem) return g_clusters[i].active;
    }
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess) return -1;
    if (g_n_clusters < 256) g_clusters[g_n_clusters++] = {{dev, kern, cl, smem}, active};
    return active;
}

// defined next to the kernels that own the device error word
caat_status read_and_clear_device_error();

namespace {

inline int64_t elem_size(caat_dtype dt) { return dt == CAAT_BF16 ? 2 : 4; }

inline bool valid_dtype(caat_dtype dt) { return dt == CAAT_F32 || dt == CAAT_BF16; }

// [lo, hi) byte range of a row-strided [rows, cols] matrix
struct Span { uintptr_t lo, hi; };
inline Span span_of(const void *p, int64_t rows, int64_t cols, int64_t ld, int64_t es)
{
    const uintptr_t lo = (uintptr_t)p;
    const int64_t n = rows > 0 && cols > 0 ? ((rows - 1) * ld + cols) * es : 0;
    return {lo, lo + (uintptr_t)n};
}
// [lo, hi) byte range of a [rows, cols] matrix with element strides (rs, cs)
inline Span span_strided(const void *p, int64_t rows, int64_t cols, int64_t rs, int64_t cs, int64_t es)
{
    const uintptr_t lo = (uintptr_t)p;
    const int64_t n = rows > 0 && cols > 0 ? ((rows - 1) * rs + (cols - 1) * cs + 1) * es : 0;
    return {lo, lo + (uintptr_t)n};
}
inline Span span_bytes(const void *p, size_t n) { return {(uintptr_t)p, (uintptr_t)p + n}; }
inline bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }
// the device index list of S (int32[n_sel]) when one is given
inline Span span_sel(const int32_t *sel, int64_t n_sel) { return span_bytes(sel, sel != nullptr && n_sel > 0 ? (size_t)n_sel * 4 : 0); }

}  // namespace
}  // namespace caat

using namespace caat;

extern "C" const char *caat_status_string(caat_status st)
{
    switch (st) {
    case CAAT_OK: return "CAAT_OK";
    case CAAT_ERR_INVALID_ARG: return "CAAT_ERR_INVALID_ARG: invalid argument";
    case CAAT_ERR_UNSUPPORTED: return "CAAT_ERR_UNSUPPORTED: no kernel takes this layout or size";
    case CAAT_ERR_CUDA: return "CAAT_ERR_CUDA: a CUDA call or kernel launch failed";
    case CAAT_ERR_TIMEOUT: return "CAAT_ERR_TIMEOUT: a bounded device-side wait gave up";
    }
    return "CAAT: unknown status";
}

extern "C" const char *caat_last_kernel(void) { return t_last_kernel; }

extern "C" uint64_t caat_launch_count(void) { return t_launches; }

extern "C" caat_status caat_get_device_status(caat_stream_t stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CAAT_ERR_CUDA;
    return read_and_clear_device_error();
}

extern "C" caat_status caat_partial_channel_reduce(int t, int64_t N, int64_t h, caat_dtype dt,
                                                   const void *const *in, int64_t ld_in,
                                                   void *const *out, int64_t ld_out,
                                                   const int32_t *sel, int64_t n_sel,
                                                   caat_stream_t stream)
{
    if (t < 1 || t > CAAT_MAX_T || N < 0 || h < 0 || !valid_dtype(dt)) return CAAT_ERR_INVALID_ARG;
    if (in == nullptr || out == nullptr) return CAAT_ERR_INVALID_ARG;
    if (ld_in < h || ld_out < h || n_sel < 0 || n_sel > h) return CAAT_ERR_INVALID_ARG;
    if (const caat_status cs = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) return cs;
    const int64_t es = elem_size(dt);
    ConstPtrs pin{};
    MutPtrs pout{};
    int same = 0;
    for (int r = 0; r < t; ++r) {
        if ((N > 0 && h > 0) && (in[r] == nullptr || out[r] == nullptr)) return CAAT_ERR_INVALID_ARG;
        pin.p[r] = in[r];
        pout.p[r] = out[r];
        same += (in[r] == out[r]);
    }
    if (same != 0 && same != t) return CAAT_ERR_INVALID_ARG;
    const bool in_place = same == t;
    if (in_place && ld_in != ld_out) return CAAT_ERR_INVALID_ARG;
    for (int r = 0; r < t; ++r) {
        const Span so = span_of(out[r], N, h, ld_out, es);
        if (overlap(so, span_sel(sel, n_sel))) return CAAT_ERR_INVALID_ARG;
        for (int q = 0; q < t; ++q) {
            if (q != r && overlap(so, span_of(out[q], N, h, ld_out, es))) return CAAT_ERR_INVALID_ARG;
            if (!in_place && overlap(so, span_of(in[q], N, h, ld_in, es))) return CAAT_ERR_INVALID_ARG;
        }
    }
    if (sel != nullptr && n_sel == h) sel = nullptr;   // S = every channel: {0, ..., h-1}
    return launch_pcr(t, N, h, dt, pin, ld_in, pout, ld_out, in_place, sel, n_sel,
                      (cudaStream_t)stream);
}

namespace {

// An index list of S is ascending and unique in [0, h): with h entries it can
// only be {0, ..., h-1}, the contiguous S of full size (the plain all-reduce).
// The calls then take the contiguous paths, which need no bitmap and, in the
// backward, reduce the gradient once instead of materialising it per rank.
inline const int32_t *all_channels(const int32_t *sel, int64_t n_sel, int64_t h)
{
    return (sel != nullptr && n_sel == h) ? nullptr : sel;
}

caat_status check_layer_args(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                             const void *X, int64_t ldx, const void *W, int64_t w_rs,
                             int64_t w_cs, const int32_t *sel, int64_t n_sel)
{
    if (t < 1 || t > CAAT_MAX_T || N < 0 || K < 0 || h < 0 || !valid_dtype(dt))
        return CAAT_ERR_INVALID_ARG;
    if (K % t != 0) return CAAT_ERR_INVALID_ARG;
    if (ldx < K || n_sel < 0 || n_sel > h) return CAAT_ERR_INVALID_ARG;
    if (N > 0 && K > 0 && X == nullptr) return CAAT_ERR_INVALID_ARG;
    if (K > 0 && h > 0) {
        if (W == nullptr || w_rs < 1 || w_cs < 1) return CAAT_ERR_INVALID_ARG;
        // the two strides must not make distinct elements coincide
        const bool row_major = w_cs == 1 && w_rs >= h;
        const bool col_major = w_rs == 1 && w_cs >= K;
        const bool general = (w_rs >= h * w_cs) || (w_cs >= K * w_rs);
        if (!(row_major || col_major || general)) return CAAT_ERR_INVALID_ARG;
    }
    return CAAT_OK;
}

// bf16 work that no tensor-core kernel takes runs on the CUDA cores only when the
// caller opts in with CAAT_ALLOW_FALLBACK=1: that path is one to two orders of
// magnitude slower, and a caller should learn of the cliff rather than meet it.
// fp32 has no tensor-core path (no TF32), so the CUDA-core kernels are its path.
bool cuda_core_path_allowed(caat_dtype dt)
{
    if (dt != CAAT_BF16) return true;
    const char *e = std::getenv("CAAT_ALLOW_FALLBACK");
    return e != nullptr && std::strcmp(e, "1") == 0;
}

}  // namespace

extern "C" caat_status caat_rowpar_linear_fwd(int t, int64_t N, int64_t K, int64_t h,
                                              caat_dtype dt, const void *X, int64_t ldx,
                                              const void *W, int64_t w_rs, int64_t w_cs,
                                              void *const *Y, int64_t ldy,
                                              const int32_t *sel, int64_t n_sel,
                                              caat_stream_t stream)
{
    caat_status st = check_layer_args(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, sel, n_sel);
    if (st != CAAT_OK) return st;
    if ((st = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) != CAAT_OK) return st;
    if (Y == nullptr || ldy < h) return CAAT_ERR_INVALID_ARG;
    const int64_t es = elem_size(dt);
    MutPtrs py{};
    for (int r = 0; r < t; ++r) {
        if (N > 0 && h > 0 && Y[r] == nullptr) return CAAT_ERR_INVALID_ARG;
        py.p[r] = Y[r];
    }
    for (int r = 0; r < t; ++r) {
        const Span so = span_of(Y[r], N, h, ldy, es);
        for (int q = r + 1; q < t; ++q)
            if (overlap(so, span_of(Y[q], N, h, ldy, es))) return CAAT_ERR_INVALID_ARG;
        if (overlap(so, span_of(X, N, K, ldx, es)) || overlap(so, span_strided(W, K, h, w_rs, w_cs, es)) ||
            overlap(so, span_sel(sel, n_sel)))
            return CAAT_ERR_INVALID_ARG;
    }
    if (N == 0 || h == 0) return CAAT_OK;
    sel = all_channels(sel, n_sel, h);
    const cudaStream_t s = (cudaStream_t)stream;
    if (dt == CAAT_BF16 && w_rs == 1 && K > 0) {
        // a few tokens: the swapped-operand tensor-core kernel (one cluster of
        // shard-CTAs per channel block), else weight streaming on the CUDA cores;
        // otherwise the tile kernel (decode kernel again if that one declines).
        // CAAT_FWD_SKINNY=0 turns the first one off (for comparisons);
        // CAAT_FWD_SKINNY_MAX=n moves its token bound (chunks of 128 tokens above 128).
        const char *skinny_env = std::getenv("CAAT_FWD_SKINNY");
        const bool skinny_on = skinny_env == nullptr || std::strcmp(skinny_env, "0") != 0;
        // A contiguous S given by its size, up to 256 tokens: at the 7B shapes two
        // chunks (512 CTAs, two per SM) beat the tile kernel, whose whole tiles of S
        // run all t shards on one CTA (out-proj 33.9 -> 28.2 us at 160 tokens, 34.1
        // -> 32.1 at 256; down-proj 66.1 -> 44.8 and 66.9 -> 48.8); from three chunks
        // on the extra waves lose.  With an index list the tile kernel cuts every
        // tile into per-shard pieces (the S sums then fold rounded partials) and is
        // the faster one above 128 tokens (256 tokens: 23.9 / 35.4 us).
        int64_t skinny_max = sel == nullptr ? 256 : 128;
        if (const char *e = std::getenv("CAAT_FWD_SKINNY_MAX")) skinny_max = std::atoll(e);
        if (N <= skinny_max && skinny_on) {
            st = launch_rowpar_fwd_skinny(t, N, K, h, X, ldx, W, w_cs, py, ldy, sel, n_sel, s);
            if (st != CAAT_ERR_UNSUPPORTED) return st;
        }
        if (N < 16) {
            st = launch_rowpar_fwd_decode(t, N, K, h, X, ldx, W, w_cs, py, ldy, sel, n_sel, s);
            if (st != CAAT_ERR_UNSUPPORTED) return st;
        }
        st = launch_rowpar_fwd_tc(t, N, K, h, X, ldx, W, w_cs, py, ldy, sel, n_sel, s);
        if (st != CAAT_ERR_UNSUPPORTED) return st;
        st = launch_rowpar_fwd_decode(t, N, K, h, X, ldx, W, w_cs, py, ldy, sel, n_sel, s);
        if (st != CAAT_ERR_UNSUPPORTED) return st;
    }
    // K == 0 only writes zeros (an empty sum)
    if (K > 0 && !cuda_core_path_allowed(dt)) return CAAT_ERR_UNSUPPORTED;
    return launch_rowpar_fwd_simt(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, py, ldy, sel, n_sel, s);
}

namespace {

// bytes of the reduced-gradient region: one [N, h] buffer per rank, each rounded
// up to 256 bytes (REDUCE_DOUT only)
size_t dy_region_bytes(int t, int64_t N, int64_t h, caat_dtype dt, caat_bwd_mode mode)
{
    if (mode != CAAT_BWD_REDUCE_DOUT) return 0;
    const size_t per = ((size_t)N * (size_t)h * (size_t)elem_size(dt) + 255) / 256 * 256;
    return per * (size_t)t;
}

// bytes of the fp32 accumulator of dW [h, K] used by the split reduction (bf16)
size_t wacc_region_bytes(int64_t K, int64_t h, caat_dtype dt)
{
    if (dt != CAAT_BF16) return 0;
    return ((size_t)K * (size_t)h * 4 + 255) / 256 * 256;
}


// Whether the tensor-core GEMMs take the gradient products of rowpar_grads.
bool grads_on_tensor_cores(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt, const void *X,
                           int64_t ldx, const void *W, int64_t w_rs, int64_t w_cs, const ConstPtrs &dy,
                           int64_t ld_dy, void *dX, int64_t lddx, void *dW, int64_t dw_rs, int64_t dw_cs)
{
    return dt == CAAT_BF16 && (dX == nullptr || w_rs == 1) && (dW == nullptr || dw_rs == 1) && N > 0 &&
           h > 0 && K > 0 &&
           bwd_tc_supported(t, N, K, h, X, dW != nullptr ? ldx : 0, W, dX != nullptr ? w_cs : 0, dy, ld_dy,
                            dX, dX != nullptr ? lddx : 0, dW, dW != nullptr ? dw_cs : 0);
}

// dX[:, shard r] = dY_r W_r^T and dW[shard r, :] = X_r^T dY_r for every rank
// (dY: t pointers [N, h], row stride ld_dy).  A null dX or dW skips that
// product; X is read only for dW, W only for dX.
caat_status rowpar_grads(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt, const void *X,
                         int64_t ldx, const void *W, int64_t w_rs, int64_t w_cs, const ConstPtrs &dy,
                         int64_t ld_dy, void *dX, int64_t lddx, void *dW, int64_t dw_rs,
                         int64_t dw_cs, float *wacc, cudaStream_t s)
{
    if (K == 0) return CAAT_OK;   // dX has no columns, dW no rows
    const int64_t es = elem_size(dt);
    const int64_t kt = K / t;
    caat_status st;
    if (grads_on_tensor_cores(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, dy, ld_dy, dX, lddx, dW, dw_rs, dw_cs)) {
        st = launch_rowpar_bwd_tc(t, N, K, h, X, ldx, W, w_cs, dy, ld_dy, dX, lddx, dW, dw_cs, wacc, 0,
                                  nullptr, 0, s);
        if (st != CAAT_ERR_UNSUPPORTED) return st;
    }
    if (h == 0) {
        // no channels: the gradient of X is zero and dW has no columns
        if (dX != nullptr && N > 0 &&
            cudaMemset2DAsync(dX, (size_t)(lddx * es), 0, (size_t)(K * es), (size_t)N, s) != cudaSuccess)
            return CAAT_ERR_CUDA;
        return CAAT_OK;
    }
    // N == 0 only writes zeros into dW (an empty sum)
    if (N > 0 && !cuda_core_path_allowed(dt)) return CAAT_ERR_UNSUPPORTED;
    if (dX != nullptr) {
        // dX[:, shard r] = dY_r W_r^T : M = N, Nn = kt, Kk = h
        BatchedGemm gx{};
        gx.batches = t; gx.M = N; gx.Nn = kt; gx.Kk = h; gx.dt = dt;
        gx.sa0 = ld_dy; gx.sa1 = 1;
        gx.sb0 = w_cs; gx.sb1 = w_rs;
        gx.sc0 = lddx; gx.sc1 = 1;
        for (int r = 0; r < t; ++r) {
            gx.A.p[r] = dy.p[r];
            gx.B.p[r] = (const char *)W + (size_t)(r * kt * w_rs * es);
            gx.C.p[r] = (char *)dX + (size_t)(r * kt * es);
        }
        st = launch_batched_gemm_simt(gx, s);   // no-op when N == 0
        if (st != CAAT_OK) return st;
    }
    if (dW == nullptr) return CAAT_OK;
    // dW[shard r, :] = X_r^T dY_r : M = kt, Nn = h, Kk = N
    BatchedGemm gw{};
    gw.batches = t; gw.M = kt; gw.Nn = h; gw.Kk = N; gw.dt = dt;
    gw.sa0 = 1; gw.sa1 = ldx;
    gw.sb0 = ld_dy; gw.sb1 = 1;
    gw.sc0 = dw_rs; gw.sc1 = dw_cs;
    for (int r = 0; r < t; ++r) {
        gw.A.p[r] = (const char *)X + (size_t)(r * kt * es);
        gw.B.p[r] = dy.p[r];
        gw.C.p[r] = (char *)dW + (size_t)(r * kt * dw_rs * es);
    }
    return launch_batched_gemm_simt(gw, s);   // N == 0 (empty sum) writes zeros
}
}  // namespace

extern "C" size_t caat_rowpar_linear_bwd_workspace(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                                   caat_bwd_mode mode)
{
    if (t < 1 || t > CAAT_MAX_T || N < 0 || K < 0 || h < 0 || !valid_dtype(dt)) return 0;
    if (mode != CAAT_BWD_REDUCE_DOUT && mode != CAAT_BWD_NO_REDUCE) return 0;
    return dy_region_bytes(t, N, h, dt, mode) + wacc_region_bytes(K, h, dt);
}

extern "C" caat_status caat_rowpar_linear_bwd(int t, int64_t N, int64_t K, int64_t h,
                                              caat_dtype dt, const void *X, int64_t ldx,
                                              const void *W, int64_t w_rs, int64_t w_cs,
                                              const void *const *dOut, int64_t ld_dout,
                                              void *dX, int64_t lddx,
                                              void *dW, int64_t dw_rs, int64_t dw_cs,
                                              const int32_t *sel, int64_t n_sel,
                                              caat_bwd_mode mode, void *workspace,
                                              size_t ws_bytes, caat_stream_t stream)
{
    caat_status st = check_layer_args(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, sel, n_sel);
    if (st != CAAT_OK) return st;
    if ((st = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) != CAAT_OK) return st;
    if (mode != CAAT_BWD_REDUCE_DOUT && mode != CAAT_BWD_NO_REDUCE) return CAAT_ERR_INVALID_ARG;
    if (dOut == nullptr || ld_dout < h || lddx < K) return CAAT_ERR_INVALID_ARG;
    if (N > 0 && K > 0 && dX == nullptr) return CAAT_ERR_INVALID_ARG;
    if (K > 0 && h > 0) {
        if (dW == nullptr || dw_rs < 1 || dw_cs < 1) return CAAT_ERR_INVALID_ARG;
        const bool ok = (dw_cs == 1 && dw_rs >= h) || (dw_rs == 1 && dw_cs >= K) ||
                        (dw_rs >= h * dw_cs) || (dw_cs >= K * dw_rs);
        if (!ok) return CAAT_ERR_INVALID_ARG;
    }
    for (int r = 0; r < t; ++r)
        if (N > 0 && h > 0 && dOut[r] == nullptr) return CAAT_ERR_INVALID_ARG;
    const bool reduce = mode == CAAT_BWD_REDUCE_DOUT && n_sel > 0 && t > 1;
    // the reduced-gradient region is required; the dW accumulator after it is
    // optional (without it dW is not split over tokens)
    const size_t need = reduce ? dy_region_bytes(t, N, h, dt, mode) : 0;
    if (need > 0 && (workspace == nullptr || ws_bytes < need || ((uintptr_t)workspace & 255)))
        return CAAT_ERR_INVALID_ARG;
    float *wacc = nullptr;
    if (workspace != nullptr && ((uintptr_t)workspace & 255) == 0 &&
        ws_bytes >= need + wacc_region_bytes(K, h, dt) && wacc_region_bytes(K, h, dt) > 0)
        wacc = (float *)((char *)workspace + need);

    // written regions (dX, dW, the part of the workspace this call uses) must not
    // overlap each other or any input
    {
        const int64_t es = elem_size(dt);
        const Span w_dx = span_of(dX, N, K, lddx, es);
        const Span w_dw = span_strided(dW, K, h, dw_rs, dw_cs, es);
        const Span w_ws = span_bytes(workspace, need + (wacc != nullptr ? wacc_region_bytes(K, h, dt) : 0));
        const Span outs[3] = {w_dx, w_dw, w_ws};
        if (overlap(w_dx, w_dw) || overlap(w_dx, w_ws) || overlap(w_dw, w_ws)) return CAAT_ERR_INVALID_ARG;
        for (const Span &o : outs) {
            if (overlap(o, span_of(X, N, K, ldx, es)) || overlap(o, span_strided(W, K, h, w_rs, w_cs, es)) ||
                overlap(o, span_sel(sel, n_sel)))
                return CAAT_ERR_INVALID_ARG;
            for (int r = 0; r < t; ++r)
                if (overlap(o, span_of(dOut[r], N, h, ld_dout, es))) return CAAT_ERR_INVALID_ARG;
        }
    }

    sel = all_channels(sel, n_sel, h);
    const cudaStream_t s = (cudaStream_t)stream;
    ConstPtrs dy{};
    int64_t ld_dy = ld_dout;

    // Contiguous S (sel == null) on the tensor-core path: reduce only the S
    // channels, once, into [N, s]; the GEMMs read them from there and the other
    // channels straight from each rank's dOut (no t-fold copy of the gradient).
    if (reduce && sel == nullptr && n_sel % 64 == 0 && dt == CAAT_BF16 && w_rs == 1 && dw_rs == 1 &&
        N > 0 && h > 0 && K > 0) {
        ConstPtrs src{};
        for (int r = 0; r < t; ++r) src.p[r] = dOut[r];
        if (bwd_tc_supported(t, N, K, h, X, ldx, W, w_cs, src, ld_dout, dX, lddx, dW, dw_cs) &&
            ((uintptr_t)workspace & 255) == 0) {
            st = launch_pcr_colsum(t, N, n_sel, src, ld_dout, workspace, n_sel, s);
            if (st == CAAT_OK)
                st = launch_rowpar_bwd_tc(t, N, K, h, X, ldx, W, w_cs, src, ld_dout, dX, lddx, dW, dw_cs,
                                          wacc, n_sel, workspace, n_sel, s);
            if (st != CAAT_ERR_UNSUPPORTED) return st;
        }
    }

    // without the opt-in, refuse bf16 work the tensor cores will not take before
    // anything is launched (the GEMMs would read the reduced gradient from the
    // workspace, row stride h)
    if (dt == CAAT_BF16 && N > 0 && K > 0 && h > 0 && !cuda_core_path_allowed(dt)) {
        ConstPtrs probe{};
        for (int r = 0; r < t; ++r)
            probe.p[r] = reduce ? (const void *)((char *)workspace + need / (size_t)t * (size_t)r) : dOut[r];
        if (!grads_on_tensor_cores(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, probe, reduce ? h : ld_dout, dX, lddx,
                                   dW, dw_rs, dw_cs))
            return CAAT_ERR_UNSUPPORTED;
    }

    if (reduce) {
        const size_t per = need / (size_t)t;
        ConstPtrs src{};
        MutPtrs dst{};
        for (int r = 0; r < t; ++r) {
            src.p[r] = dOut[r];
            dst.p[r] = (char *)workspace + per * (size_t)r;
            dy.p[r] = dst.p[r];
        }
        st = launch_pcr(t, N, h, dt, src, ld_dout, dst, h, false, sel, n_sel, s);
        if (st != CAAT_OK) return st;
        ld_dy = h;
    } else {
        for (int r = 0; r < t; ++r) dy.p[r] = dOut[r];
    }
    return rowpar_grads(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, dy, ld_dy, dX, lddx, dW, dw_rs, dw_cs,
                        wacc, s);
}


// ------------------------------------------------- compact outputs
// The t outputs with the S channels (the same on every rank) stored once:
// YS [N, |S|] and YN[r] [N, h - |S|], each in ascending channel order.  A
// contiguous S runs the tile kernels directly; an index list of S runs them on a
// copy of W whose channels are in the order "S first" (the workspace), which
// makes S contiguous, and puts dW's rows back in channel order at the end.

namespace {

size_t wperm_region_bytes(int64_t K, int64_t h) { return ((size_t)K * (size_t)h * 2 + 255) / 256 * 256; }

}  // namespace

extern "C" size_t caat_rowpar_linear_compact_workspace(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                                       int index_list, int backward)
{
    if (t < 1 || t > CAAT_MAX_T || N < 0 || K < 0 || h < 0 || !valid_dtype(dt)) return 0;
    // forward: W in the S-first order; backward: that, then dW staged in the same
    // order, then the optional fp32 accumulator of dW
    if (!backward) return index_list ? wperm_region_bytes(K, h) : 0;
    return (index_list ? 2 * wperm_region_bytes(K, h) : 0) + wacc_region_bytes(K, h, dt);
}

extern "C" caat_status caat_rowpar_linear_fwd_compact(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                                      const void *X, int64_t ldx,
                                                      const void *W, int64_t w_rs, int64_t w_cs,
                                                      void *YS, int64_t ldys, void *const *YN, int64_t ldyn,
                                                      const int32_t *sel, int64_t n_sel,
                                                      void *workspace, size_t ws_bytes, caat_stream_t stream)
{
    caat_status st = check_layer_args(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, sel, n_sel);
    if (st != CAAT_OK) return st;
    if ((st = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) != CAAT_OK) return st;
    sel = all_channels(sel, n_sel, h);
    const int64_t h_own = h - n_sel;
    if (N > 0 && n_sel > 0 && (YS == nullptr || ldys < n_sel)) return CAAT_ERR_INVALID_ARG;
    if (N > 0 && h_own > 0 && (YN == nullptr || ldyn < h_own)) return CAAT_ERR_INVALID_ARG;
    const int64_t es = elem_size(dt);
    // an index list of S with 0 < |S| < h needs W in the S-first order
    const bool perm = sel != nullptr && n_sel > 0 && n_sel < h && K > 0;
    const size_t need = perm ? wperm_region_bytes(K, h) : 0;
    if (need > 0 && (workspace == nullptr || ws_bytes < need || ((uintptr_t)workspace & 255)))
        return CAAT_ERR_INVALID_ARG;
    MutPtrs py{};
    if (h_own > 0)
        for (int r = 0; r < t; ++r) {
            if (N > 0 && YN[r] == nullptr) return CAAT_ERR_INVALID_ARG;
            py.p[r] = YN[r];
        }
    {
        const Span sx = span_of(X, N, K, ldx, es), sw = span_strided(W, K, h, w_rs, w_cs, es);
        const Span ss = span_of(YS, N, n_sel, ldys, es), sl = span_sel(sel, n_sel);
        const Span sws = span_bytes(workspace, need);
        if (overlap(ss, sx) || overlap(ss, sw) || overlap(ss, sl) || overlap(ss, sws)) return CAAT_ERR_INVALID_ARG;
        if (overlap(sws, sx) || overlap(sws, sw) || overlap(sws, sl)) return CAAT_ERR_INVALID_ARG;
        for (int r = 0; h_own > 0 && r < t; ++r) {
            const Span so = span_of(YN[r], N, h_own, ldyn, es);
            if (overlap(so, ss) || overlap(so, sx) || overlap(so, sw) || overlap(so, sl) || overlap(so, sws))
                return CAAT_ERR_INVALID_ARG;
            for (int q = r + 1; q < t; ++q)
                if (overlap(so, span_of(YN[q], N, h_own, ldyn, es))) return CAAT_ERR_INVALID_ARG;
        }
    }
    if (N == 0 || h == 0) return CAAT_OK;
    if (n_sel % 64 != 0 || dt != CAAT_BF16 || w_rs != 1) return CAAT_ERR_UNSUPPORTED;
    const cudaStream_t s = (cudaStream_t)stream;
    if (K == 0) {
        // empty sums: zeros
        if (n_sel > 0 && cudaMemset2DAsync(YS, (size_t)(ldys * es), 0, (size_t)(n_sel * es), (size_t)N, s) != cudaSuccess)
            return CAAT_ERR_CUDA;
        for (int r = 0; h_own > 0 && r < t; ++r)
            if (cudaMemset2DAsync(YN[r], (size_t)(ldyn * es), 0, (size_t)(h_own * es), (size_t)N, s) != cudaSuccess)
                return CAAT_ERR_CUDA;
        return CAAT_OK;
    }
    const void *Wk = W;
    int64_t ldw = w_cs;
    if (perm) {
        // the tile kernel's shape rules first, so that nothing runs for a call it declines
        if (N < 16 || (K / t) < 64 || (K / t) % 8 != 0) return CAAT_ERR_UNSUPPORTED;
        if ((st = launch_permute_rows(W, w_cs, workspace, K, h, K, sel, n_sel, true, s)) != CAAT_OK) return st;
        Wk = workspace;
        ldw = K;
    }
    // with no S channel the compact form is the plain one (YN[r] = Y[r])
    return launch_rowpar_fwd_tc(t, N, K, h, X, ldx, Wk, ldw, py, ldyn, nullptr, n_sel, s,
                                n_sel > 0 ? YS : nullptr, ldys);
}

extern "C" caat_status caat_rowpar_linear_bwd_compact(int t, int64_t N, int64_t K, int64_t h, caat_dtype dt,
                                                      const void *X, int64_t ldx,
                                                      const void *W, int64_t w_rs, int64_t w_cs,
                                                      const void *dYS, int64_t lddys,
                                                      const void *const *dYN, int64_t lddyn,
                                                      void *dX, int64_t lddx,
                                                      void *dW, int64_t dw_rs, int64_t dw_cs,
                                                      const int32_t *sel, int64_t n_sel,
                                                      void *workspace, size_t ws_bytes, caat_stream_t stream)
{
    caat_status st = check_layer_args(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, sel, n_sel);
    if (st != CAAT_OK) return st;
    if ((st = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) != CAAT_OK) return st;
    sel = all_channels(sel, n_sel, h);
    const int64_t h_own = h - n_sel;
    if (N > 0 && n_sel > 0 && (dYS == nullptr || lddys < n_sel)) return CAAT_ERR_INVALID_ARG;
    if (N > 0 && h_own > 0 && (dYN == nullptr || lddyn < h_own)) return CAAT_ERR_INVALID_ARG;
    if (lddx < K || (N > 0 && K > 0 && dX == nullptr)) return CAAT_ERR_INVALID_ARG;
    if (K > 0 && h > 0) {
        if (dW == nullptr || dw_rs < 1 || dw_cs < 1) return CAAT_ERR_INVALID_ARG;
        const bool ok = (dw_cs == 1 && dw_rs >= h) || (dw_rs == 1 && dw_cs >= K) ||
                        (dw_rs >= h * dw_cs) || (dw_cs >= K * dw_rs);
        if (!ok) return CAAT_ERR_INVALID_ARG;
    }
    ConstPtrs dy{};
    if (h_own > 0)
        for (int r = 0; r < t; ++r) {
            if (N > 0 && dYN[r] == nullptr) return CAAT_ERR_INVALID_ARG;
            dy.p[r] = dYN[r];
        }
    const int64_t es = elem_size(dt);
    // an index list of S: W in the S-first order and room to stage dW in that
    // order are required (dW's rows then return to channel order); the fp32
    // accumulator after them stays optional
    const bool perm = sel != nullptr && n_sel > 0 && n_sel < h && K > 0 && N > 0;
    const size_t wperm = perm ? 2 * wperm_region_bytes(K, h) : 0;
    const size_t need = wperm;
    if (need > 0 && (workspace == nullptr || ws_bytes < need || ((uintptr_t)workspace & 255)))
        return CAAT_ERR_INVALID_ARG;
    float *wacc = nullptr;
    if (workspace != nullptr && ((uintptr_t)workspace & 255) == 0 && wacc_region_bytes(K, h, dt) > 0 &&
        ws_bytes >= wperm + wacc_region_bytes(K, h, dt))
        wacc = (float *)((char *)workspace + wperm);
    {
        const Span w_dx = span_of(dX, N, K, lddx, es);
        const Span w_dw = span_strided(dW, K, h, dw_rs, dw_cs, es);
        const Span w_ws = span_bytes(workspace, wperm + (wacc != nullptr ? wacc_region_bytes(K, h, dt) : 0));
        const Span outs[3] = {w_dx, w_dw, w_ws};
        if (overlap(w_dx, w_dw) || overlap(w_dx, w_ws) || overlap(w_dw, w_ws)) return CAAT_ERR_INVALID_ARG;
        for (const Span &o : outs) {
            if (overlap(o, span_of(X, N, K, ldx, es)) || overlap(o, span_strided(W, K, h, w_rs, w_cs, es)) ||
                overlap(o, span_of(dYS, N, n_sel, lddys, es)) || overlap(o, span_sel(sel, n_sel)))
                return CAAT_ERR_INVALID_ARG;
            for (int r = 0; h_own > 0 && r < t; ++r)
                if (overlap(o, span_of(dYN[r], N, h_own, lddyn, es))) return CAAT_ERR_INVALID_ARG;
        }
    }
    if (K == 0) return CAAT_OK;                      // dX has no columns, dW no rows
    const cudaStream_t s = (cudaStream_t)stream;
    if (h == 0) {                                    // no channels: dX = 0
        if (N > 0 && cudaMemset2DAsync(dX, (size_t)(lddx * es), 0, (size_t)(K * es), (size_t)N, s) != cudaSuccess)
            return CAAT_ERR_CUDA;
        return CAAT_OK;
    }
    if (n_sel % 64 != 0 || dt != CAAT_BF16 || w_rs != 1 || dw_rs != 1) return CAAT_ERR_UNSUPPORTED;
    if (N == 0) {                                    // empty sums over tokens: dW = 0 ([h, K] storage)
        if (cudaMemset2DAsync(dW, (size_t)(dw_cs * es), 0, (size_t)(K * es), (size_t)h, s) != cudaSuccess)
            return CAAT_ERR_CUDA;
        return CAAT_OK;
    }
    if (!bwd_tc_supported(t, N, K, h, X, ldx, W, w_cs, dy, lddyn, dX, lddx, dW, dw_cs) ||
        (n_sel > 0 && ((uintptr_t)dYS % 16 != 0 || lddys % 8 != 0)))
        return CAAT_ERR_UNSUPPORTED;
    // with an index list W is permuted inside, after the dW chain has forked off
    void *dw_tmp = perm ? (char *)workspace + wperm_region_bytes(K, h) : nullptr;
    return launch_rowpar_bwd_tc(t, N, K, h, X, ldx, W, w_cs, dy, lddyn, dX, lddx, dW, dw_cs, wacc, n_sel,
                                n_sel > 0 ? dYS : nullptr, lddys, s, true, perm ? sel : nullptr, n_sel, dw_tmp,
                                perm ? workspace : nullptr);
}


// ------------------------------------------------- column-parallel layer
// The column-parallel layer is the row-parallel one seen through W = W1^T
// (logical [K, h], strides (w1_cs, w1_rs)): its forward is the dX product of the
// row-parallel backward with dY_r = A_r, its input gradient is the fused
// row-parallel forward on dZ (GEMM + partial reduce), its weight gradient the dW
// product with X = dZ and dY_r = A_r.

namespace {

caat_status check_colpar_inputs(int t, int64_t N, int64_t h, const void *const *A, int64_t lda)
{
    if (A == nullptr || lda < h) return CAAT_ERR_INVALID_ARG;
    for (int r = 0; r < t; ++r)
        if (N > 0 && h > 0 && A[r] == nullptr) return CAAT_ERR_INVALID_ARG;
    return CAAT_OK;
}

}  // namespace

extern "C" caat_status caat_colpar_linear_fwd(int t, int64_t N, int64_t h, int64_t K, caat_dtype dt,
                                              const void *const *A, int64_t lda,
                                              const void *W1, int64_t w1_rs, int64_t w1_cs,
                                              void *Z, int64_t ldz, caat_stream_t stream)
{
    caat_status st = check_layer_args(t, N, K, h, dt, Z, ldz, W1, w1_cs, w1_rs, nullptr, 0);
    if (st != CAAT_OK) return st;
    st = check_colpar_inputs(t, N, h, A, lda);
    if (st != CAAT_OK) return st;
    const int64_t es = elem_size(dt);
    const Span sz = span_of(Z, N, K, ldz, es);
    if (overlap(sz, span_strided(W1, h, K, w1_rs, w1_cs, es))) return CAAT_ERR_INVALID_ARG;
    ConstPtrs a{};
    for (int r = 0; r < t; ++r) {
        if (overlap(sz, span_of(A[r], N, h, lda, es))) return CAAT_ERR_INVALID_ARG;
        a.p[r] = A[r];
    }
    if (N == 0) return CAAT_OK;
    return rowpar_grads(t, N, K, h, dt, nullptr, 0, W1, w1_cs, w1_rs, a, lda, Z, ldz, nullptr, 0, 0,
                        nullptr, (cudaStream_t)stream);
}

extern "C" size_t caat_colpar_linear_bwd_workspace(int t, int64_t N, int64_t h, int64_t K, caat_dtype dt)
{
    if (t < 1 || t > CAAT_MAX_T || N < 0 || K < 0 || h < 0 || !valid_dtype(dt)) return 0;
    return wacc_region_bytes(K, h, dt);
}

extern "C" caat_status caat_colpar_linear_bwd(int t, int64_t N, int64_t h, int64_t K, caat_dtype dt,
                                              const void *const *A, int64_t lda,
                                              const void *W1, int64_t w1_rs, int64_t w1_cs,
                                              const void *dZ, int64_t ldz,
                                              void *const *dA, int64_t ldda,
                                              void *dW1, int64_t dw1_rs, int64_t dw1_cs,
                                              const int32_t *sel, int64_t n_sel,
                                              void *workspace, size_t ws_bytes, caat_stream_t stream)
{
    caat_status st = check_layer_args(t, N, K, h, dt, dZ, ldz, W1, w1_cs, w1_rs, sel, n_sel);
    if (st != CAAT_OK) return st;
    if ((st = check_sel_debug(sel, n_sel, h, (cudaStream_t)stream)) != CAAT_OK) return st;
    st = check_colpar_inputs(t, N, h, A, lda);
    if (st != CAAT_OK) return st;
    if (dA == nullptr || ldda < h) return CAAT_ERR_INVALID_ARG;
    if (K > 0 && h > 0) {
        if (dW1 == nullptr || dw1_rs < 1 || dw1_cs < 1) return CAAT_ERR_INVALID_ARG;
        // logical dW = dW1^T: (k, c) strides (dw1_cs, dw1_rs)
        const int64_t a0 = dw1_cs, a1 = dw1_rs;
        const bool ok = (a1 == 1 && a0 >= h) || (a0 == 1 && a1 >= K) || (a0 >= h * a1) || (a1 >= K * a0);
        if (!ok) return CAAT_ERR_INVALID_ARG;
    }
    const int64_t es = elem_size(dt);
    ConstPtrs a{};
    for (int r = 0; r < t; ++r) {
        if (N > 0 && h > 0 && dA[r] == nullptr) return CAAT_ERR_INVALID_ARG;
        const Span sr = span_of(dA[r], N, h, ldda, es);
        for (int q = 0; q < t; ++q) {
            if (overlap(sr, span_of(A[q], N, h, lda, es))) return CAAT_ERR_INVALID_ARG;
            if (q > r && overlap(sr, span_of(dA[q], N, h, ldda, es))) return CAAT_ERR_INVALID_ARG;
        }
        if (overlap(sr, span_of(dZ, N, K, ldz, es)) || overlap(sr, span_strided(W1, h, K, w1_rs, w1_cs, es)) ||
            overlap(sr, span_sel(sel, n_sel)))
            return CAAT_ERR_INVALID_ARG;
        a.p[r] = A[r];
    }
    float *wacc = nullptr;
    if (workspace != nullptr && ((uintptr_t)workspace & 255) == 0 && wacc_region_bytes(K, h, dt) > 0 &&
        ws_bytes >= wacc_region_bytes(K, h, dt))
        wacc = (float *)workspace;
    {
        const Span w_dw = span_strided(dW1, h, K, dw1_rs, dw1_cs, es);
        const Span w_ws = span_bytes(wacc, wacc != nullptr ? wacc_region_bytes(K, h, dt) : 0);
        if (overlap(w_dw, w_ws)) return CAAT_ERR_INVALID_ARG;
        for (const Span &o : {w_dw, w_ws}) {
            if (overlap(o, span_of(dZ, N, K, ldz, es)) || overlap(o, span_strided(W1, h, K, w1_rs, w1_cs, es)) ||
                overlap(o, span_sel(sel, n_sel)))
                return CAAT_ERR_INVALID_ARG;
            for (int r = 0; r < t; ++r)
                if (overlap(o, span_of(A[r], N, h, lda, es)) || overlap(o, span_of(dA[r], N, h, ldda, es)))
                    return CAAT_ERR_INVALID_ARG;
        }
    }
    const cudaStream_t s = (cudaStream_t)stream;
    // dW1 and dA only read shared inputs: dW1 runs on the side stream next to dA
    SideStream *side = (N > 0 && K > 0 && h > 0) ? side_stream(s) : nullptr;
    cudaStream_t sw = s;
    if (side != nullptr) {
        if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
            return CAAT_ERR_CUDA;
        sw = side->s;
    }
    // dW1 = A_r^T dZ_r per block (the dW product with X = dZ, dY_r = A_r)
    st = rowpar_grads(t, N, K, h, dt, dZ, ldz, W1, w1_cs, w1_rs, a, lda, nullptr, 0, dW1, dw1_cs, dw1_rs,
                      wacc, sw);
    // dA = PCR_S(dZ_r W1_r^T): the fused row-parallel forward on (dZ, W1^T)
    if (st == CAAT_OK)
        st = caat_rowpar_linear_fwd(t, N, K, h, dt, dZ, ldz, W1, w1_cs, w1_rs, dA, ldda, sel, n_sel, stream);
    // the side stream joins back even after an error (a captured fork must join)
    if (side != nullptr &&
        (cudaEventRecord(side->join, sw) != cudaSuccess || cudaStreamWaitEvent(s, side->join, 0) != cudaSuccess))
        return CAAT_ERR_CUDA;
    return st;
}
