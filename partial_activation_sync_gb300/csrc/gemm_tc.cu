// tcgen05 / TMEM / TMA tensor-core kernels (sm_103a).
#include "caat_internal.h"

namespace caat {

__device__ int g_caat_dev_error;

caat_status read_and_clear_device_error()
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_caat_dev_error, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_caat_dev_error, &zero, sizeof(int)) != cudaSuccess) return CAAT_ERR_CUDA;
        return (caat_status)v;
    }
    return CAAT_OK;
}

caat_status launch_rowpar_fwd_tc(int, int64_t, int64_t, int64_t, const void *, int64_t,
                                 const void *, int64_t, const MutPtrs &, int64_t,
                                 const int32_t *, int64_t, cudaStream_t)
{
    return CAAT_ERR_UNSUPPORTED;
}

}  // namespace caat
