// vh_api.cu -- host side of the libvh C ABI: argument validation, kernel
// dispatch, error reporting.  See include/vh.h for the contract.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "vh_common.cuh"

namespace vh {
cudaError_t launch_scan_simt(const ScanArgs &a, int d, bool bf16, cudaStream_t st);
cudaError_t launch_scan_tc(const ScanArgs &a, int d, bool bf16, cudaStream_t st, bool *handled);
cudaError_t launch_qproj(const void *x, bool bf16, int d, const float *wq, const float *skip,
                         const float *dir_scale, unsigned dirs, __nv_bfloat16 *qhat, float *out,
                         int accumulate, long npix, int Cc, float knorm_eps, cudaStream_t st);
}  // namespace vh

namespace {

thread_local char g_err[512] = "";

vh_status fail(vh_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

vh_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(VH_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

vh_status check_common(const vh_params *p, int H, int W)
{
    if (!p) return fail(VH_ERR_INVALID_ARG, "params is NULL");
    if (p->batch < 1 || H < 1 || W < 1 || p->channels < 1 || p->head_dim < 1)
        return fail(VH_ERR_INVALID_ARG, "sizes must be >= 1 (B=%d H=%d W=%d Cc=%d d=%d)",
                    p->batch, H, W, p->channels, p->head_dim);
    if (p->head_dim != 16 && p->head_dim != 32 && p->head_dim != 64)
        return fail(VH_ERR_UNSUPPORTED, "head_dim %d not built (16, 32, 64)", p->head_dim);
    if (p->channels % p->head_dim)
        return fail(VH_ERR_INVALID_ARG, "channels %d is not a multiple of head_dim %d",
                    p->channels, p->head_dim);
    if (p->x_dtype != VH_DTYPE_F32 && p->x_dtype != VH_DTYPE_BF16)
        return fail(VH_ERR_UNSUPPORTED, "x_dtype %d", (int)p->x_dtype);
    const double n = (double)H * (double)W;
    if (n * (double)p->channels >= 2147483647.0)
        return fail(VH_ERR_INVALID_ARG, "H*W*channels %.0f exceeds 2^31-1 per image", n * p->channels);
    return VH_OK;
}

}  // namespace

extern "C" {

void vh_params_init(vh_params *p)
{
    if (!p) return;
    std::memset(p, 0, sizeof *p);
    p->x_dtype = VH_DTYPE_BF16;
    p->gamma_eta = 0.025f;
    p->alpha_init = 0.9f;
    p->eta_bias = 0.0f;
    p->eps = 1e-6f;
    p->knorm_eps = 1e-6f;
    p->inj_inward = 1e-3f;
    p->spec_inward = 1e-6f;
    p->kk_floor = 1e-20f;
    p->gate_mode = VH_GATE_GENERATED;
    p->impl = VH_IMPL_AUTO;
}

const char *vh_status_string(vh_status s)
{
    switch (s) {
    case VH_OK: return "ok";
    case VH_ERR_INVALID_ARG: return "invalid argument";
    case VH_ERR_UNSUPPORTED: return "unsupported configuration";
    case VH_ERR_CUDA: return "CUDA error";
    case VH_ERR_WORKSPACE: return "workspace error";
    case VH_ERR_NONFINITE: return "non-finite value";
    case VH_ERR_TIMEOUT: return "timeout";
    }
    return "unknown status";
}

const char *vh_last_error(void) { return g_err; }

int vh_version(void) { return 100; }

size_t vh_workspace_size(const vh_params *p, int H, int W, unsigned, int)
{
    if (!p || !p->w_query || p->batch < 1 || H < 1 || W < 1 || p->channels < 1) return 0;
    return (size_t)6 * p->batch * H * W * p->channels;
}

vh_status vh_check(const unsigned long long *stats, void *stream)
{
    g_err[0] = '\0';
    if (!stats) return fail(VH_ERR_INVALID_ARG, "stats is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long h[VH_STAT_COUNT];
    cudaError_t e = cudaMemcpyAsync(h, stats, sizeof h, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return cuda_fail(e, "reading stats");
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "synchronising the stream");
    if (h[VH_STAT_TIMEOUT])
        return fail(VH_ERR_TIMEOUT, "%llu CTA(s) gave up a bounded wait; results are invalid",
                    h[VH_STAT_TIMEOUT]);
    if (h[VH_STAT_NONFINITE])
        return fail(VH_ERR_NONFINITE, "%llu non-finite readout value(s)", h[VH_STAT_NONFINITE]);
    return VH_OK;
}

vh_status vh_scan_forward(const void *x, const float *memories0, const vh_params *p, int H,
                          int W, unsigned dirs, int chunk, float *out)
{
    g_err[0] = '\0';
    vh_status s = check_common(p, H, W);
    if (s != VH_OK) return s;
    if (!x || !memories0 || !out) return fail(VH_ERR_INVALID_ARG, "x, memories0 and out must be non-NULL");
    if (!aligned16(x) || !aligned16(out))
        return fail(VH_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(memories0) & 3u) || (p->memories_out && (reinterpret_cast<uintptr_t>(p->memories_out) & 3u)))
        return fail(VH_ERR_INVALID_ARG, "memories must be 4-byte aligned");
    if (dirs == 0 || (dirs & ~15u)) return fail(VH_ERR_INVALID_ARG, "dirs mask 0x%x invalid", dirs);
    if (chunk < 0) return fail(VH_ERR_INVALID_ARG, "chunk %d < 0", chunk);
    if (p->gate_mode < 0 || p->gate_mode > 2) return fail(VH_ERR_INVALID_ARG, "gate_mode %d", p->gate_mode);
    if (!(p->alpha_init > 0.0f && p->alpha_init < 1.0f))
        return fail(VH_ERR_INVALID_ARG, "alpha_init %g must lie in (0,1)", (double)p->alpha_init);
    if (p->impl < VH_IMPL_AUTO || p->impl > VH_IMPL_TC) return fail(VH_ERR_INVALID_ARG, "impl %d", p->impl);
    if (p->control_flags & ~(unsigned)VH_CTRL_ALL)
        return fail(VH_ERR_INVALID_ARG, "control_flags 0x%x has unknown bits", p->control_flags);

    const int d = p->head_dim, nh = p->channels / d, B = p->batch;
    const size_t N = (size_t)H * W;
    const size_t xbytes = (size_t)B * N * p->channels * (p->x_dtype == VH_DTYPE_BF16 ? 2 : 4);
    const size_t obytes = (size_t)B * N * p->channels * 4;
    const char *xb = static_cast<const char *>(x), *oc = reinterpret_cast<const char *>(out);
    if (xb < oc + obytes && oc < xb + xbytes) return fail(VH_ERR_INVALID_ARG, "out aliases x");
    const bool exact = p->w_query != nullptr;
    if (exact) {
        const size_t qbytes = (size_t)6 * B * N * p->channels;
        const char *wb = static_cast<const char *>(p->workspace);
        if (!wb || p->workspace_bytes < qbytes || !aligned16(wb))
            return fail(VH_ERR_WORKSPACE, "w_query needs a 16-byte aligned workspace of %zu bytes "
                        "(have %zu)", qbytes, p->workspace ? p->workspace_bytes : (size_t)0);
        if ((wb < oc + obytes && oc < wb + qbytes) || (wb < xb + xbytes && xb < wb + qbytes))
            return fail(VH_ERR_INVALID_ARG, "workspace aliases x or out");
        if (reinterpret_cast<uintptr_t>(p->w_query) & 3u)
            return fail(VH_ERR_INVALID_ARG, "w_query must be 4-byte aligned");
    }
    if (p->skip && (reinterpret_cast<uintptr_t>(p->skip) & 3u))
        return fail(VH_ERR_INVALID_ARG, "skip must be 4-byte aligned");

    vh::ScanArgs a{};
    a.x = x;
    a.mem0 = memories0;
    a.out = out;
    a.mem_out = p->memories_out;
    a.dir_scale = p->dir_scale;
    a.stats = p->stats;
    a.B = B; a.H = H; a.W = W; a.nh = nh; a.Cc = p->channels;
    a.ndirs = 0;
    for (int r = 0; r < 4; ++r)
        if (dirs & (1u << r)) a.dir_list[a.ndirs++] = r;
    a.chunk = chunk;
    a.gamma_eta = p->gamma_eta;
    a.alpha_logit = (float)std::log((double)p->alpha_init / (1.0 - (double)p->alpha_init));
    a.eta_bias = p->eta_bias;
    a.eps = p->eps;
    a.knorm_eps = p->knorm_eps;
    a.inj_factor = 1.0f - p->inj_inward;
    a.spec_factor = 1.0f - p->spec_inward;
    a.kk_floor = p->kk_floor;
    a.gate_mode = p->gate_mode;
    a.forced_eta = p->forced_eta;
    a.forced_alpha = p->forced_alpha;
    a.control_flags = p->control_flags;
    a.qhat = exact ? static_cast<const __nv_bfloat16 *>(p->workspace) : nullptr;

    cudaStream_t st = static_cast<cudaStream_t>(p->stream);
    cudaError_t e = cudaSuccess;
    const bool bf16 = p->x_dtype == VH_DTYPE_BF16;
    if (!p->accumulate && !p->skip) {
        e = cudaMemsetAsync(out, 0, obytes, st);
        if (e != cudaSuccess) return cuda_fail(e, "zeroing out");
    }
    if (exact || p->skip) {  // outer queries and / or the skip term seeding out
        e = vh::launch_qproj(x, bf16, d, p->w_query, p->skip, p->dir_scale, dirs,
                             static_cast<__nv_bfloat16 *>(p->workspace), out, p->accumulate,
                             (long)(B * N), p->channels, p->knorm_eps, st);
        if (e != cudaSuccess) return cuda_fail(e, "query projection launch");
    }
    bool handled = false;
    if (p->impl != VH_IMPL_SIMT) {
        e = vh::launch_scan_tc(a, d, bf16, st, &handled);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core scan launch");
        if (!handled && p->impl == VH_IMPL_TC)
            return fail(VH_ERR_UNSUPPORTED, "no tensor-core kernel for d=%d dtype=%d chunk=%d",
                        d, (int)p->x_dtype, chunk);
    }
    if (!handled) {
        e = vh::launch_scan_simt(a, d, bf16, st);
        if (e != cudaSuccess) return cuda_fail(e, "scan launch");
    }
    return VH_OK;
}

}  // extern "C"

namespace {

template <typename XT>
__global__ void permute_kernel(const XT *__restrict__ x, XT *__restrict__ seq, int H, int W,
                               int Cc, int route, size_t total)
{
    const size_t N = (size_t)H * W;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total;
         e += (size_t)gridDim.x * blockDim.x) {
        const size_t c = e % Cc, bt = e / Cc;
        const size_t t = bt % N, b = bt / N;
        const int pix = vh::route_pixel(route, (int)t, H, W);
        seq[e] = x[(b * N + pix) * Cc + c];
    }
}

}  // namespace

extern "C" vh_status vh_debug_permute(const void *x, const vh_params *p, int H, int W, int route,
                                      void *seq)
{
    g_err[0] = '\0';
    vh_status s = check_common(p, H, W);
    if (s != VH_OK) return s;
    if (!x || !seq) return fail(VH_ERR_INVALID_ARG, "x and seq must be non-NULL");
    if (route < 0 || route > 3) return fail(VH_ERR_INVALID_ARG, "route %d", route);
    const size_t total = (size_t)p->batch * H * W * p->channels;
    cudaStream_t st = static_cast<cudaStream_t>(p->stream);
    const unsigned grid = (unsigned)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
    if (p->x_dtype == VH_DTYPE_BF16)
        permute_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(x),
                                             static_cast<__nv_bfloat16 *>(seq), H, W, p->channels,
                                             route, total);
    else
        permute_kernel<<<grid, 256, 0, st>>>(static_cast<const float *>(x), static_cast<float *>(seq),
                                             H, W, p->channels, route, total);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "permute launch");
    return VH_OK;
}
