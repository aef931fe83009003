// vh_scan_tc.cu -- tensor-core (tcgen05) scan kernel: not built yet; every
// shape falls through to the CUDA-core kernel.
#include "vh_common.cuh"

namespace vh {

cudaError_t launch_scan_tc(const ScanArgs &, int, bool, cudaStream_t, bool *handled)
{
    *handled = false;
    return cudaSuccess;
}

}  // namespace vh
