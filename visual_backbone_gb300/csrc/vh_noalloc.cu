// vh_noalloc.cu -- vh_scan_forward_static: the VisionHOPE-exact forward (outer query
// projection) for callers that may not allocate device memory.
//
// Some callers can't call cudaMalloc, or size and keep a workspace buffer: a plug-in
// running inside a host application that owns every device allocation (an inference
// server, a runtime with a pre-sized memory pool) must work with the memory it is given.
// The exact readout needs scratch for its normalised query planes, which
// vh_scan_forward takes from the caller's workspace.  This entry point takes it from a
// fixed array compiled into the library instead, and otherwise runs the same kernels
// through vh_scan_forward.
#include "vh_common.cuh"

namespace vh {
vh_status record_error(vh_status s, const char *fmt, ...);
}

namespace {

// The query planes: 6 bytes per element of x (three bf16 pieces).  Every GPU that loads
// the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_qscratch[kStaticScratchBytes];

// The array's device address in the current context, looked up on every call (a device
// reset that recreates the primary context can move the array, so nothing is cached).
cudaError_t scratch_address(void **ptr)
{
    *ptr = nullptr;
    return cudaGetSymbolAddress(ptr, g_qscratch);
}

}  // namespace

extern "C" vh_status vh_scan_forward_static(const void *x, const float *memories0,
                                            const vh_params *p, int H, int W, unsigned dirs,
                                            int chunk, float *out)
{
    if (!p || !p->w_query)
        return vh::record_error(VH_ERR_INVALID_ARG,
                                "vh_scan_forward_static runs the outer-query readout (w_query); "
                                "without it vh_scan_forward needs no scratch");
    if (p->batch < 1 || H < 1 || W < 1 || p->channels < 1)
        return vh::record_error(VH_ERR_INVALID_ARG, "sizes must be >= 1");
    const size_t need = (size_t)6 * p->batch * H * W * p->channels;
    if (need > kStaticScratchBytes)
        return vh::record_error(VH_ERR_WORKSPACE,
                                "vh_scan_forward_static: the query planes need %zu bytes, the "
                                "static scratch holds %zu (B*H*W*channels <= %zu)",
                                need, kStaticScratchBytes, kStaticScratchBytes / 6);
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return vh::record_error(VH_ERR_CUDA, "looking up the static scratch: %s",
                                cudaGetErrorString(e));
    // every query plane is rewritten before it is read, so nothing needs clearing
    vh_params q = *p;
    q.workspace = scratch;
    q.workspace_bytes = kStaticScratchBytes;
    return vh_scan_forward(x, memories0, &q, H, W, dirs, chunk, out);
}
