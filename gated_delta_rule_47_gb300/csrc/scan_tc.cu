// scan_tc.cu -- tcgen05 path of the chunkwise scan (placeholder: not yet
// taken; every call goes to the SIMT path).
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {

namespace {
__device__ unsigned int g_tc_error = 0;
}

bool scan_tc_supported(const ScanArgs &) { return false; }
size_t scan_tc_workspace_bytes(const ScanArgs &) { return 0; }
int launch_scan_tc(const ScanArgs &, cudaStream_t) { return GDN_ERR_UNSUPPORTED; }

int scan_tc_read_clear_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero)) != cudaSuccess) return GDN_ERR_CUDA;
    return v ? GDN_ERR_TIMEOUT : GDN_OK;
}

int scan_tc_set_wait_limit(unsigned long long) { return GDN_OK; }

}  // namespace gdn
