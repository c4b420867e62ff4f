// Backward of the fused row-parallel layer for callers that cannot allocate
// device memory themselves: the library's own statically sized scratch array
// stands in for the caller's workspace.
//
// Some callers cannot call cudaMalloc: a host framework that hands every byte
// of device memory to its own pool allocator and forbids side allocations, or a
// process that fixes its memory budget when it starts.  For them this file holds
// a file-scope device array of CAAT_NOALLOC_SCRATCH_BYTES; every GPU that loads
// the library keeps it until the process exits.
#include "caat_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CAAT_NOALLOC_SCRATCH_BYTES];

// In host code the array's name is a host-side shadow, not a device address;
// the device address comes from the runtime for the current device.  It is
// looked up on every call (no allocation, a few microseconds at most), so a
// device reset that reloads the module and moves the array leaves nothing stale.
caat_status scratch_address(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CAAT_ERR_CUDA;
    *out = p;
    return CAAT_OK;
}

}  // namespace

extern "C" caat_status caat_rowpar_linear_bwd_noalloc(
    int t, int64_t N, int64_t K, int64_t h, caat_dtype dt, const void *X, int64_t ldx,
    const void *W, int64_t w_rs, int64_t w_cs, const void *const *dOut, int64_t ld_dout,
    void *dX, int64_t lddx, void *dW, int64_t dw_rs, int64_t dw_cs, const int32_t *sel,
    int64_t n_sel, caat_bwd_mode mode, caat_stream_t stream)
{
    // The reduced gradient is needed only when the backward sums something: the
    // reduce placement, a non-empty S and more than one rank (the same condition
    // as caat_rowpar_linear_bwd's).  Size check before any product that could
    // overflow.
    const bool reduce = mode == CAAT_BWD_REDUCE_DOUT && n_sel > 0 && t > 1;
    if (reduce && N > 0 && h > 0) {
        const double bytes = (double)t * (double)N * (double)h * (dt == CAAT_BF16 ? 2.0 : 4.0);
        if (bytes > (double)CAAT_NOALLOC_SCRATCH_BYTES) return CAAT_ERR_INVALID_ARG;
    }
    // the part of the workspace the backward cannot do without: the reduced
    // gradient, t buffers of [N, h] rounded up to 256 bytes each
    size_t need = 0;
    if (reduce && N > 0 && h > 0)
        need = (size_t)t * (((size_t)N * (size_t)h * (dt == CAAT_BF16 ? 2u : 4u) + 255) / 256 * 256);
    if (need > (size_t)CAAT_NOALLOC_SCRATCH_BYTES) return CAAT_ERR_INVALID_ARG;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    // the scratch also serves, when it is large enough, as the optional fp32
    // accumulator of the token-split dW reduction, so offer it for any size
    const bool uses_scratch = t >= 1 && N > 0 && h > 0 && K > 0;
    if (uses_scratch) {
        const caat_status st = scratch_address(&ws);
        if (st != CAAT_OK) return st;
        ws_bytes = (size_t)CAAT_NOALLOC_SCRATCH_BYTES;
    }
    // the reduced gradient fills the whole [t, N, h] region it uses before it is
    // read, and the dW accumulator is cleared on the stream before use, so
    // nothing left over from an earlier call can leak into this one
    return caat_rowpar_linear_bwd(t, N, K, h, dt, X, ldx, W, w_rs, w_cs, dOut, ld_dout, dX, lddx,
                                  dW, dw_rs, dw_cs, sel, n_sel, mode, ws, ws_bytes, stream);
}
