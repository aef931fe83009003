// vh_api.cu -- host side of the libvh C ABI: argument validation, kernel
// dispatch, error reporting.  See include/vh.h for the contract.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "vh_common.cuh"

namespace vh {
cudaError_t launch_scan_simt(const ScanArgs &a, int d, bool bf16, cudaStream_t st);
cudaError_t launch_scan_tc(const ScanArgs &a, int d, bool bf16, cudaStream_t st, bool *handled,
                           int gain);
cudaError_t launch_gelu_debug(const float *a, __nv_bfloat16 *out, long long n, cudaStream_t st);
cudaError_t launch_scan_tc64(const ScanArgs &a, int d, bool bf16, cudaStream_t st, bool *handled,
                             int gain);
cudaError_t launch_qproj(const void *x, bool bf16, int d, const float *wq, const float *skip,
                         const float *dir_scale, unsigned dirs, __nv_bfloat16 *qhat, float *out,
                         int accumulate, long npix, int Cc, float knorm_eps, cudaStream_t st);
cudaError_t launch_scan_bwd(const BwdArgs &ba, int d, bool bf16, cudaStream_t st);
cudaError_t launch_cpe_ln(const float *x, const float *cw, const float *cb, const float *g,
                          const float *beta, float eps, float *x0, __nv_bfloat16 *a, int B, int H,
                          int W, int D, bool split, cudaStream_t st);
cudaError_t launch_ln(const float *x, const float *g, const float *beta, float eps,
                      __nv_bfloat16 *a, long npix, int D, bool split, cudaStream_t st);
cudaError_t launch_dwgate(const float *u, const float *w, const float *b, void *z, long npix, int C,
                          int H, int W, bool f32, cudaStream_t st);
cudaError_t launch_posdw(const float *y, const void *z, const float *w, const float *b, void *yb,
                         long npix, int C, int H, int W, bool f32, cudaStream_t st);
cudaError_t launch_gemm_tc(int M, int N, int K, const __nv_bfloat16 *w, const __nv_bfloat16 *act,
                           const float *bias, const float *res, void *out, int epi,
                           cudaStream_t st);
size_t bwd_floats_per_scan(int d, int nck, int lmax);
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

vh_status check_scan(const vh_params *p, unsigned dirs, int chunk)
{
    if (dirs == 0 || (dirs & ~15u)) return fail(VH_ERR_INVALID_ARG, "dirs mask 0x%x invalid", dirs);
    if (chunk < 0) return fail(VH_ERR_INVALID_ARG, "chunk %d < 0", chunk);
    if (p->gate_mode < 0 || p->gate_mode > 2) return fail(VH_ERR_INVALID_ARG, "gate_mode %d", p->gate_mode);
    if (!(p->alpha_init > 0.0f && p->alpha_init < 1.0f))
        return fail(VH_ERR_INVALID_ARG, "alpha_init %g must lie in (0,1)", (double)p->alpha_init);
    if (p->impl < VH_IMPL_AUTO || p->impl > VH_IMPL_TC_PIPE) return fail(VH_ERR_INVALID_ARG, "impl %d", p->impl);
    if (p->control_flags & ~(unsigned)VH_CTRL_ALL)
        return fail(VH_ERR_INVALID_ARG, "control_flags 0x%x has unknown bits", p->control_flags);
    return VH_OK;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    const char *x = static_cast<const char *>(a), *y = static_cast<const char *>(b);
    return a && b && x < y + nb && y < x + na;
}

vh::ScanArgs make_args(const void *x, const float *memories0, const vh_params *p, int H, int W,
                       unsigned dirs, int chunk, float *out)
{
    vh::ScanArgs a{};
    const int nh = p->channels / p->head_dim;
    a.x = x;
    a.mem0 = memories0;
    a.out = out;
    a.mem_out = p->memories_out;
    a.dir_scale = p->dir_scale;
    a.stats = p->stats;
    a.B = p->batch; a.H = H; a.W = W; a.nh = nh; a.Cc = p->channels;
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
    a.wait_limit = p->wait_limit;
    a.withhold_first_copy = p->withhold_first_copy;

    return a;
}

// Routes enabled in `dirs`: chunks of the longest-chunked route's count and the longest
// chunk, both as provisioned per scan by the backward workspace.
void bwd_extent(int H, int W, unsigned dirs, int chunk, int *nck, int *lmax)
{
    const int N = H * W;
    *nck = 0;
    *lmax = 0;
    for (int r = 0; r < 4; ++r) {
        if (!(dirs & (1u << r))) continue;
        const int Cr = vh::route_chunk(r, chunk, H, W);
        const int L = Cr < N ? Cr : N;
        const int n = (N + Cr - 1) / Cr;
        if (n > *nck) *nck = n;
        if (L > *lmax) *lmax = L;
    }
}

// The backward's pre-pass on the tensor-core forward also writes every token's record
// (k, q, delta and raw scalars) where that kernel applies: head_dim 32, bf16 x, chunks
// aligned with rows and columns.
bool bwd_token_records(const vh_params *p, int H, int W, int chunk)
{
    return p->impl != VH_IMPL_SIMT && p->head_dim == 32 && p->x_dtype == VH_DTYPE_BF16 &&
           (chunk == 0 || (chunk == W && chunk == H)) && p->channels % 8 == 0;
}

// Byte offsets of the block's intermediates in its workspace (256-byte aligned regions).
struct BlockLayout {
    size_t x0, a, u, z, yb, h, qhat, w3, total;  // w3: the GEMM weights tripled along K (f32 mode)
};

BlockLayout block_layout(const vh_params *p, const vh_block_weights *w, int H, int W)
{
    BlockLayout L{};
    const size_t N = (size_t)p->batch * H * W, D = w->dim, Dm = p->channels, Hd = w->hidden;
    // fp32-intermediate test mode: GEMM activations as three bf16 pieces, fp32 Z
    const size_t pc = w->f32_intermediates ? 3 : 1;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o += (bytes + 255) & ~(size_t)255; return at; };
    L.x0 = take(N * D * 4);
    L.a = take(N * D * 2 * pc);
    L.u = take(N * Dm * 4);
    L.z = take(N * Dm * (w->f32_intermediates ? 4 : 2));
    L.yb = take(N * Dm * 2 * pc);
    L.h = take(N * Hd * 2 * pc);
    L.qhat = take(p->w_query ? 6 * N * Dm : 0);
    L.w3 = take(w->f32_intermediates ? 3 * 2 * (Dm * D + D * Dm + Hd * D + D * Hd) : 0);
    L.total = o;
    return L;
}

}  // namespace

namespace vh {
// Record a failure from another translation unit of the library (same thread-local text
// as the entry points here).
vh_status record_error(vh_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}
}  // namespace vh

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
    case VH_ERR_BOUNDS: return "index out of bounds";
    }
    return "unknown status";
}

const char *vh_last_error(void) { return g_err; }

int vh_version(void) { return 100; }

int vh_debug_bounds_build(void)
{
#ifdef VH_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

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
    if (h[VH_STAT_BOUNDS])
        return fail(VH_ERR_BOUNDS, "%llu index check(s) failed; results are invalid", h[VH_STAT_BOUNDS]);
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
    s = check_scan(p, dirs, chunk);
    if (s != VH_OK) return s;

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
    if (p->wait_limit < 0) return fail(VH_ERR_INVALID_ARG, "wait_limit %lld < 0", p->wait_limit);
    if (p->withhold_first_copy &&
        (p->head_dim != 32 || p->x_dtype != VH_DTYPE_BF16 || p->impl == VH_IMPL_SIMT ||
         !(chunk == 0 || (chunk == W && chunk == H)) || p->channels % 8))
        return fail(VH_ERR_INVALID_ARG, "withhold_first_copy is a hook of the head_dim 32 "
                    "tensor-core kernel (bf16 x, row/column chunks)");

    vh::ScanArgs a = make_args(x, memories0, p, H, W, dirs, chunk, out);
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
        if (d == 64)
            e = vh::launch_scan_tc64(a, d, bf16, st, &handled, p->impl);
        else
            e = vh::launch_scan_tc(a, d, bf16, st, &handled, p->impl);
        if (e == cudaErrorNotSupported)
            return fail(VH_ERR_UNSUPPORTED, "the WY gain needs the method as defined (no control_flags, "
                        "no w_query) and H, W <= 64 (head_dim 32) or <= 32 (head_dim 64); the "
                        "pipelined form needs head_dim 32 and the method as defined");
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core scan launch");
        if (!handled && p->impl != VH_IMPL_AUTO)
            return fail(VH_ERR_UNSUPPORTED, "no tensor-core kernel for d=%d dtype=%d chunk=%d",
                        d, (int)p->x_dtype, chunk);
    }
    if (!handled) {
        e = vh::launch_scan_simt(a, d, bf16, st);
        if (e != cudaSuccess) return cuda_fail(e, "scan launch");
    }
    return VH_OK;
}

size_t vh_block_workspace_size(const vh_params *p, const vh_block_weights *w, int H, int W)
{
    if (!p || !w || p->batch < 1 || H < 1 || W < 1 || p->channels < 1 || w->dim < 1 ||
        w->hidden < 1)
        return 0;
    return block_layout(p, w, H, W).total;
}

vh_status vh_block_forward(const float *x, const float *memories0, const vh_params *p,
                           const vh_block_weights *w, int H, int W, float *out)
{
    g_err[0] = '\0';
    vh_status s = check_common(p, H, W);
    if (s != VH_OK) return s;
    if (!w) return fail(VH_ERR_INVALID_ARG, "weights is NULL");
    if (!x || !memories0 || !out) return fail(VH_ERR_INVALID_ARG, "x, memories0 and out must be non-NULL");
    if (p->x_dtype != VH_DTYPE_BF16) return fail(VH_ERR_UNSUPPORTED, "the block runs the operator on bf16 Z");
    if (p->accumulate || p->memories_out)
        return fail(VH_ERR_INVALID_ARG, "accumulate and memories_out are not used by the block");
    if (w->dim < 8 || w->dim > 1024 || w->dim % 8 || w->hidden < 8 || w->hidden % 8)
        return fail(VH_ERR_INVALID_ARG, "dim %d (8..1024, multiple of 8) / hidden %d (multiple of 8)",
                    w->dim, w->hidden);
    const void *need[] = {w->cpe_w, w->cpe_b, w->ln1_g, w->ln1_b, w->w_in, w->b_in, w->dw_w, w->dw_b,
                          w->pos_w, w->pos_b, w->w_out, w->b_out, w->ln2_g, w->ln2_b, w->w_ff1,
                          w->b_ff1, w->w_ff2, w->b_ff2};
    for (const void *q : need)
        if (!q) return fail(VH_ERR_INVALID_ARG, "every weight pointer must be non-NULL");
    const void *gw[] = {w->w_in, w->w_out, w->w_ff1, w->w_ff2};
    for (const void *q : gw)
        if (!aligned16(q)) return fail(VH_ERR_INVALID_ARG, "GEMM weights must be 16-byte aligned");
    if (!aligned16(x) || !aligned16(out)) return fail(VH_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    const BlockLayout L = block_layout(p, w, H, W);
    if (!p->workspace || p->workspace_bytes < L.total || !aligned16(p->workspace))
        return fail(VH_ERR_WORKSPACE, "the block needs a 16-byte aligned workspace of %zu bytes (have %zu)",
                    L.total, p->workspace ? p->workspace_bytes : (size_t)0);
    const int B = p->batch, D = w->dim, Dm = p->channels, Hd = w->hidden;
    const long N = (long)B * H * W;
    const size_t xb = (size_t)N * D * 4;
    if (overlaps(x, xb, out, xb) || overlaps(x, xb, p->workspace, L.total) ||
        overlaps(out, xb, p->workspace, L.total))
        return fail(VH_ERR_INVALID_ARG, "x, out and the workspace must not overlap");
    const float eps = w->ln_eps > 0.0f ? w->ln_eps : 1e-5f;
    const bool f32 = w->f32_intermediates != 0;
    const int pc = f32 ? 3 : 1;  // bf16 pieces per GEMM activation
    char *ws = static_cast<char *>(p->workspace);
    float *x0 = reinterpret_cast<float *>(ws + L.x0);
    __nv_bfloat16 *a = reinterpret_cast<__nv_bfloat16 *>(ws + L.a);
    float *u = reinterpret_cast<float *>(ws + L.u);  // U, then Y
    void *z = ws + L.z;
    __nv_bfloat16 *yb = reinterpret_cast<__nv_bfloat16 *>(ws + L.yb);
    __nv_bfloat16 *h = reinterpret_cast<__nv_bfloat16 *>(ws + L.h);
    auto bw = [](const void *q) { return static_cast<const __nv_bfloat16 *>(q); };
    cudaStream_t st = static_cast<cudaStream_t>(p->stream);
    cudaError_t e = cudaSuccess;
    // the GEMM weights, tripled along K in f32 mode: [rows][3K] = [W | W | W], so that the
    // product with the three pieces of an activation row is its fp32 product
    const __nv_bfloat16 *w_in = bw(w->w_in), *w_out = bw(w->w_out), *w_ff1 = bw(w->w_ff1),
                        *w_ff2 = bw(w->w_ff2);
    if (f32) {
        __nv_bfloat16 *w3 = reinterpret_cast<__nv_bfloat16 *>(ws + L.w3);
        const struct { const __nv_bfloat16 *src; int rows, K; const __nv_bfloat16 **use; } mats[4] = {
            {w_in, Dm, D, &w_in}, {w_out, D, Dm, &w_out}, {w_ff1, Hd, D, &w_ff1}, {w_ff2, D, Hd, &w_ff2}};
        for (const auto &m : mats) {
            for (int k = 0; k < 3 && e == cudaSuccess; ++k)
                e = cudaMemcpy2DAsync(w3 + (size_t)k * m.K, (size_t)3 * m.K * 2, m.src, (size_t)m.K * 2,
                                      (size_t)m.K * 2, m.rows, cudaMemcpyDeviceToDevice, st);
            *m.use = w3;
            w3 += (size_t)3 * m.K * m.rows;
        }
        if (e != cudaSuccess) return cuda_fail(e, "tripling the GEMM weights");
    }
    // X0 = X + CPE(X), A = LN1(X0)
    if ((e = vh::launch_cpe_ln(x, w->cpe_w, w->cpe_b, w->ln1_g, w->ln1_b, eps, x0, a, B, H, W, D, f32, st)))
        return cuda_fail(e, "CPE + LN1 launch");
    // U = A W_in^T + b_in
    if ((e = vh::launch_gemm_tc((int)N, Dm, pc * D, w_in, a, w->b_in, nullptr, u, 0, st)))
        return cuda_fail(e, "Proj_in GEMM launch");
    // Z = U + SiLU(DW(U))
    if ((e = vh::launch_dwgate(u, w->dw_w, w->dw_b, z, N, Dm, H, W, f32, st)))
        return cuda_fail(e, "gated depthwise launch");
    // Y = F_VH(Z), into U's buffer
    vh_params q = *p;
    q.workspace = p->w_query ? ws + L.qhat : nullptr;
    q.workspace_bytes = p->w_query ? 6 * (size_t)N * Dm : 0;
    if (f32) q.x_dtype = VH_DTYPE_F32;
    if ((s = vh_scan_forward(z, memories0, &q, H, W, VH_DIR_ALL, 0, u)) != VH_OK) return s;
    // Y += DW_pos(Z), cast (f32 mode: split) for Proj_out
    if ((e = vh::launch_posdw(u, z, w->pos_w, w->pos_b, yb, N, Dm, H, W, f32, st)))
        return cuda_fail(e, "positional depthwise launch");
    // X1 = X0 + Y W_out^T + b_out, into out
    if ((e = vh::launch_gemm_tc((int)N, D, pc * Dm, w_out, yb, w->b_out, x0, out, 0, st)))
        return cuda_fail(e, "Proj_out GEMM launch");
    // out = X1 + W_ff2 GELU(W_ff1 LN2(X1) + b_ff1) + b_ff2
    if ((e = vh::launch_ln(out, w->ln2_g, w->ln2_b, eps, a, N, D, f32, st)))
        return cuda_fail(e, "LN2 launch");
    // H = bf16(GELU(bf16(LN2(X1) W_ff1^T) + b_ff1)) (GELU in the GEMM's epilogue; f32 mode:
    // GELU of the unrounded product, as three pieces), then out = X1 + H W_ff2^T + b_ff2
    if ((e = vh::launch_gemm_tc((int)N, Hd, pc * D, w_ff1, a, w->b_ff1, nullptr, h, f32 ? 2 : 1, st)))
        return cuda_fail(e, "FFN1 GEMM launch");
    if ((e = vh::launch_gemm_tc((int)N, D, pc * Hd, w_ff2, h, w->b_ff2, out, out, 0, st)))
        return cuda_fail(e, "FFN2 GEMM launch");
    return VH_OK;
}

size_t vh_backward_workspace_size(const vh_params *p, int H, int W, unsigned dirs, int chunk)
{
    if (!p || p->batch < 1 || H < 1 || W < 1 || p->head_dim < 1 || p->channels < p->head_dim ||
        dirs == 0 || (dirs & ~15u) || chunk < 0)
        return 0;
    int nck, lmax, nd = 0;
    bwd_extent(H, W, dirs, chunk, &nck, &lmax);
    for (int r = 0; r < 4; ++r) nd += (dirs >> r) & 1;
    const size_t scans = (size_t)p->batch * nd * (p->channels / p->head_dim);
    size_t floats = scans * vh::bwd_floats_per_scan(p->head_dim, nck, lmax);
    if (bwd_token_records(p, H, W, chunk))
        floats += scans * (size_t)H * W * vh::token_rec_floats(p->head_dim);
    return floats * sizeof(float);
}

vh_status vh_scan_backward(const void *x, const float *memories0, const vh_params *p, int H,
                           int W, unsigned dirs, int chunk, const float *dout,
                           const float *dmem_final, float *dx, float *dmem0)
{
    g_err[0] = '\0';
    vh_status s = check_common(p, H, W);
    if (s != VH_OK) return s;
    s = check_scan(p, dirs, chunk);
    if (s != VH_OK) return s;
    if (!x || !memories0 || !dout || !dx || !dmem0)
        return fail(VH_ERR_INVALID_ARG, "x, memories0, dout, dx and dmem0 must be non-NULL");
    if (!aligned16(x) || !aligned16(dx))
        return fail(VH_ERR_INVALID_ARG, "x and dx must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(memories0) & 3u) || (reinterpret_cast<uintptr_t>(dout) & 3u) ||
        (reinterpret_cast<uintptr_t>(dmem0) & 3u) || (reinterpret_cast<uintptr_t>(dmem_final) & 3u))
        return fail(VH_ERR_INVALID_ARG, "memories0, dout, dmem_final and dmem0 must be 4-byte aligned");
    if (p->control_flags || p->w_query || p->skip)
        return fail(VH_ERR_UNSUPPORTED, "the backward covers the method as defined "
                    "(no control_flags, w_query or skip)");
    const int d = p->head_dim, nh = p->channels / d, B = p->batch;
    const size_t N = (size_t)H * W;
    const size_t xbytes = (size_t)B * N * p->channels * (p->x_dtype == VH_DTYPE_BF16 ? 2 : 4);
    const size_t gbytes = (size_t)B * N * p->channels * 4;
    const size_t mbytes = (size_t)4 * nh * (4 * d * d + 2 * d) * 4;
    const size_t wbytes = vh_backward_workspace_size(p, H, W, dirs, chunk);
    if (!p->workspace || p->workspace_bytes < wbytes || !aligned16(p->workspace))
        return fail(VH_ERR_WORKSPACE, "the backward needs a 16-byte aligned workspace of %zu bytes "
                    "(have %zu)", wbytes, p->workspace ? p->workspace_bytes : (size_t)0);
    const void *ins[4] = {x, dout, memories0, dmem_final};
    const size_t insz[4] = {xbytes, gbytes, mbytes, (size_t)B * mbytes};  // dmem_final: B blocks
    void *outs[3] = {dx, dmem0, p->workspace};
    const size_t outsz[3] = {gbytes, mbytes, wbytes};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 4; ++j)
            if (overlaps(outs[i], outsz[i], ins[j], insz[j]))
                return fail(VH_ERR_INVALID_ARG, "an output or the workspace aliases an input");
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], outsz[i], outs[j], outsz[j]))
                return fail(VH_ERR_INVALID_ARG, "outputs / workspace overlap");
    }

    vh::BwdArgs ba{};
    ba.s = make_args(x, memories0, p, H, W, dirs, chunk, nullptr);
    ba.s.mem_out = nullptr;  // (p->stats stays: the pre-pass counts as a forward call, and
                             // both kernels count expired waits and failed index checks)
    ba.dout = dout;
    ba.dmem_final = dmem_final;
    ba.dx = dx;
    ba.dmem0 = dmem0;
    ba.ws = static_cast<float *>(p->workspace);
    bwd_extent(H, W, dirs, chunk, &ba.nck, &ba.lmax);
    cudaStream_t st = static_cast<cudaStream_t>(p->stream);
    cudaError_t e = cudaMemsetAsync(dx, 0, gbytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dmem0, 0, mbytes, st);
    if (e != cudaSuccess) return cuda_fail(e, "zeroing dx / dmem0");
    const bool bf16 = p->x_dtype == VH_DTYPE_BF16;
    if (p->impl != VH_IMPL_SIMT) {
        // the boundary states and token records from the tensor-core forward (no readout
        // adds), where it applies; the records follow the per-scan blocks
        vh::ScanArgs f = ba.s;
        f.out = nullptr;
        f.ckpt = ba.ws;
        f.ckpt_stride = vh::bwd_floats_per_scan(d, ba.nck, ba.lmax);
        if (bwd_token_records(p, H, W, chunk)) {
            f.rec = ba.ws + (size_t)ba.s.B * ba.s.ndirs * ba.s.nh * f.ckpt_stride;
            f.rec_stride = N * vh::token_rec_floats(d);
        }
        bool handled = false;
        e = vh::launch_scan_tc(f, d, bf16, st, &handled, VH_IMPL_TC_RECUR);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core forward launch");
        ba.have_ckpt = handled ? 1 : 0;
        if (handled) {
            ba.s.rec = f.rec;
            ba.s.rec_stride = f.rec_stride;
        }
    }
    e = vh::launch_scan_bwd(ba, d, bf16, st);
    if (e != cudaSuccess) return cuda_fail(e, "backward scan launch");
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

extern "C" vh_status vh_debug_gelu(const float *a, void *out, long long n, void *stream)
{
    g_err[0] = '\0';
    if (n < 0) return fail(VH_ERR_INVALID_ARG, "n %lld", n);
    if (n > 0 && (!a || !out)) return fail(VH_ERR_INVALID_ARG, "a and out must be non-NULL");
    cudaError_t e = vh::launch_gelu_debug(a, static_cast<__nv_bfloat16 *>(out), n,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gelu launch");
    return VH_OK;
}

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
