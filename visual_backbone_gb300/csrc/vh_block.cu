// vh_block.cu -- the VisionHOPE block around the operator ("VisionHOPE: Visual Backbones
// as Self-Modifying Learning Systems", Sec. 2.3 Eq. (27), App. B.5), inference on NHWC
// activations:
//
//   X0  = X + CPE(X)                     CPE = 3 x 3 depthwise conv (+bias)
//   U   = Proj_in(LN1(X0))               D -> D_m
//   Z   = U + SiLU(DW3x3(U))             gated depthwise residual branch
//   Y   = F_VH(Z) + DW3x3(Z)             exact operator + depthwise positional skip
//   X1  = X0 + Proj_out(Y)               D_m -> D
//   out = X1 + W2 GELU(W1 LN2(X1) + b1) + b2
//
// The four pointwise layers are plain GEMMs on bf16 operands with fp32 accumulation
// (cuBLASLt, bias and residual in its epilogue).  The kernels here do the rest, each one
// pass over the activations: CPE + LN1 (one warp per pixel), the gated branch, the
// positional branch with the cast for Proj_out, LN2, GELU.  bf16 rounding points: LN1's
// and LN2's outputs, Z, Y before Proj_out, GELU's output.
#include <cublasLt.h>

#include <mutex>

#include "vh_common.cuh"

namespace vh {

// ------------------------------------------------------------------ kernels

// Per pixel (one warp): x0 = x + b + sum_{3x3} w x (depthwise, zero padding) and
// a = bf16(LN(x0) * g + beta).  Channels c = lane + 32 m, m < MAXC.
template <int MAXC>
__global__ void __launch_bounds__(256) cpe_ln_kernel(const float *__restrict__ x,
                                                     const float *__restrict__ cw,
                                                     const float *__restrict__ cb,
                                                     const float *__restrict__ g,
                                                     const float *__restrict__ beta, float eps,
                                                     float *__restrict__ x0,
                                                     __nv_bfloat16 *__restrict__ a, int B, int H,
                                                     int W, int D)
{
    const int lane = threadIdx.x & 31;
    const long npix = (long)B * H * W;
    for (long pix = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5; pix < npix;
         pix += ((long)gridDim.x * blockDim.x) >> 5) {
        const int j = (int)(pix % W), i = (int)((pix / W) % H);
        const long b = pix / ((long)H * W);
        float v[MAXC];
        float s = 0.0f;
#pragma unroll
        for (int m = 0; m < MAXC; ++m) {
            const int c = lane + 32 * m;
            v[m] = 0.0f;
            if (c < D) {
                float acc = cb[c] + x[pix * D + c];
#pragma unroll
                for (int di = -1; di <= 1; ++di) {
                    const int ii = i + di;
                    if (ii < 0 || ii >= H) continue;
#pragma unroll
                    for (int dj = -1; dj <= 1; ++dj) {
                        const int jj = j + dj;
                        if (jj < 0 || jj >= W) continue;
                        acc = fmaf(cw[c * 9 + (di + 1) * 3 + (dj + 1)],
                                   x[((b * H + ii) * W + jj) * D + c], acc);
                    }
                }
                v[m] = acc;
                x0[pix * D + c] = acc;
                s += acc;
            }
        }
        const float mu = warp_sum(s) / D;
        float q = 0.0f;
#pragma unroll
        for (int m = 0; m < MAXC; ++m)
            if (lane + 32 * m < D) q = fmaf(v[m] - mu, v[m] - mu, q);
        const float rs = rsqrtf(warp_sum(q) / D + eps);
#pragma unroll
        for (int m = 0; m < MAXC; ++m) {
            const int c = lane + 32 * m;
            if (c < D) a[pix * D + c] = __float2bfloat16_rn((v[m] - mu) * rs * g[c] + beta[c]);
        }
    }
}

// Per pixel (one warp): a = bf16(LN(x) * g + beta).
template <int MAXC>
__global__ void __launch_bounds__(256) ln_kernel(const float *__restrict__ x,
                                                 const float *__restrict__ g,
                                                 const float *__restrict__ beta, float eps,
                                                 __nv_bfloat16 *__restrict__ a, long npix, int D)
{
    const int lane = threadIdx.x & 31;
    for (long pix = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5; pix < npix;
         pix += ((long)gridDim.x * blockDim.x) >> 5) {
        float v[MAXC];
        float s = 0.0f;
#pragma unroll
        for (int m = 0; m < MAXC; ++m) {
            const int c = lane + 32 * m;
            v[m] = c < D ? x[pix * D + c] : 0.0f;
            s += v[m];
        }
        const float mu = warp_sum(s) / D;
        float q = 0.0f;
#pragma unroll
        for (int m = 0; m < MAXC; ++m)
            if (lane + 32 * m < D) q = fmaf(v[m] - mu, v[m] - mu, q);
        const float rs = rsqrtf(warp_sum(q) / D + eps);
#pragma unroll
        for (int m = 0; m < MAXC; ++m) {
            const int c = lane + 32 * m;
            if (c < D) a[pix * D + c] = __float2bfloat16_rn((v[m] - mu) * rs * g[c] + beta[c]);
        }
    }
}

// 3 x 3 depthwise cross-correlation with zero padding at element e (pixel, channel c)
// of an NHWC tensor of type T with C channels.
template <typename T>
__device__ __forceinline__ float dw3(const T *__restrict__ src, const float *__restrict__ w,
                                     long e, int c, int C, int H, int W)
{
    const long pix = e / C;
    const int j = (int)(pix % W), i = (int)((pix / W) % H);
    const long b = pix / ((long)H * W);
    float acc = 0.0f;
#pragma unroll
    for (int di = -1; di <= 1; ++di) {
        const int ii = i + di;
        if (ii < 0 || ii >= H) continue;
#pragma unroll
        for (int dj = -1; dj <= 1; ++dj) {
            const int jj = j + dj;
            if (jj < 0 || jj >= W) continue;
            acc = fmaf(w[c * 9 + (di + 1) * 3 + (dj + 1)],
                       XElem<T>::to_f(src[((b * H + ii) * W + jj) * C + c]), acc);
        }
    }
    return acc;
}

// z = bf16(u + SiLU(dw(u) + b)): the gated depthwise residual branch.
__global__ void __launch_bounds__(256) dwgate_kernel(const float *__restrict__ u,
                                                     const float *__restrict__ w,
                                                     const float *__restrict__ bias,
                                                     __nv_bfloat16 *__restrict__ z, long total,
                                                     int C, int H, int W)
{
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < total;
         e += (long)gridDim.x * blockDim.x) {
        const int c = (int)(e % C);
        const float a = dw3(u, w, e, c, C, H, W) + bias[c];
        const float s = a / (1.0f + __expf(-a));
        z[e] = __float2bfloat16_rn(u[e] + s);
    }
}

// yb = bf16(y + dw(z) + b): the positional branch around the operator, cast for Proj_out.
__global__ void __launch_bounds__(256) posdw_kernel(const float *__restrict__ y,
                                                    const __nv_bfloat16 *__restrict__ z,
                                                    const float *__restrict__ w,
                                                    const float *__restrict__ bias,
                                                    __nv_bfloat16 *__restrict__ yb, long total,
                                                    int C, int H, int W)
{
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < total;
         e += (long)gridDim.x * blockDim.x) {
        const int c = (int)(e % C);
        yb[e] = __float2bfloat16_rn(y[e] + dw3(z, w, e, c, C, H, W) + bias[c]);
    }
}

// h = bf16(GELU(a)), GELU(a) = a (1 + erf(a / sqrt 2)) / 2, four elements per thread.
__global__ void __launch_bounds__(256) gelu_kernel(const float4 *__restrict__ a,
                                                   __nv_bfloat162 *__restrict__ h, long n4)
{
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n4;
         e += (long)gridDim.x * blockDim.x) {
        const float4 v = a[e];
        const float k = 0.70710678118654752f;
        const float g0 = 0.5f * v.x * (1.0f + erff(v.x * k));
        const float g1 = 0.5f * v.y * (1.0f + erff(v.y * k));
        const float g2 = 0.5f * v.z * (1.0f + erff(v.z * k));
        const float g3 = 0.5f * v.w * (1.0f + erff(v.w * k));
        h[2 * e] = __floats2bfloat162_rn(g0, g1);
        h[2 * e + 1] = __floats2bfloat162_rn(g2, g3);
    }
}

// ------------------------------------------------------------------ GEMMs (cuBLASLt)

namespace {

std::mutex g_lt_mu;
cublasLtHandle_t g_lt[64] = {};

cublasStatus_t lt_handle(cublasLtHandle_t *h)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CUBLAS_STATUS_NOT_INITIALIZED;
    std::lock_guard<std::mutex> lk(g_lt_mu);
    if (!g_lt[dev]) {
        const cublasStatus_t s = cublasLtCreate(&g_lt[dev]);
        if (s != CUBLAS_STATUS_SUCCESS) return s;
    }
    *h = g_lt[dev];
    return CUBLAS_STATUS_SUCCESS;
}

}  // namespace

// out[n][m] = act[n][k] . wt[m][k]^T + bias[m] (+ res[n][m]): row-major bf16 operands,
// fp32 result, fp32 accumulation.  res may equal out.  Returns the cublasStatus_t.
int block_gemm(int m, int n, int k, const __nv_bfloat16 *wt, const __nv_bfloat16 *act,
               const float *bias, const float *res, float *out, void *ws, size_t ws_bytes,
               cudaStream_t st)
{
    cublasLtHandle_t lt;
    cublasStatus_t s = lt_handle(&lt);
    if (s != CUBLAS_STATUS_SUCCESS) return (int)s;
    // column-major view: out^T (m x n) = wt (k x m)^T . act^T (k x n) [+ res^T]
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    const cublasOperation_t tA = CUBLAS_OP_T, tB = CUBLAS_OP_N;
    const cublasLtEpilogue_t epi = CUBLASLT_EPILOGUE_BIAS;
    const float alpha = 1.0f, beta = res ? 1.0f : 0.0f;
    cublasLtMatmulHeuristicResult_t hr{};
    int found = 0;
    do {
        if ((s = cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F))) break;
        if ((s = cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &tA, sizeof tA))) break;
        if ((s = cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tB, sizeof tB))) break;
        if ((s = cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_EPILOGUE, &epi, sizeof epi))) break;
        if ((s = cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof bias))) break;
        if ((s = cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, k, m, k))) break;
        if ((s = cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, k, n, k))) break;
        if ((s = cublasLtMatrixLayoutCreate(&lc, CUDA_R_32F, m, n, m))) break;
        if ((s = cublasLtMatmulPreferenceCreate(&pref))) break;
        if ((s = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                                      &ws_bytes, sizeof ws_bytes))) break;
        if ((s = cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, lc, lc, pref, 1, &hr, &found))) break;
        if (!found) { s = CUBLAS_STATUS_NOT_SUPPORTED; break; }
        s = cublasLtMatmul(lt, op, &alpha, wt, la, act, lb, &beta, res ? res : out, lc, out, lc,
                           &hr.algo, ws, ws_bytes, st);
    } while (0);
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return (int)s;
}

// ------------------------------------------------------------------ launches

namespace {

unsigned grid_for(long threads)
{
    long g = (threads + 255) / 256;
    const long cap = 152L * 16;  // a few waves of resident blocks; grid-stride beyond
    return (unsigned)(g < cap ? (g > 0 ? g : 1) : cap);
}

}  // namespace

cudaError_t launch_cpe_ln(const float *x, const float *cw, const float *cb, const float *g,
                          const float *beta, float eps, float *x0, __nv_bfloat16 *a, int B, int H,
                          int W, int D, cudaStream_t st)
{
    const long npix = (long)B * H * W;
    const unsigned grid = grid_for(npix * 32);
    if (D <= 256)
        cpe_ln_kernel<8><<<grid, 256, 0, st>>>(x, cw, cb, g, beta, eps, x0, a, B, H, W, D);
    else
        cpe_ln_kernel<32><<<grid, 256, 0, st>>>(x, cw, cb, g, beta, eps, x0, a, B, H, W, D);
    return cudaGetLastError();
}

cudaError_t launch_ln(const float *x, const float *g, const float *beta, float eps,
                      __nv_bfloat16 *a, long npix, int D, cudaStream_t st)
{
    const unsigned grid = grid_for(npix * 32);
    if (D <= 256)
        ln_kernel<8><<<grid, 256, 0, st>>>(x, g, beta, eps, a, npix, D);
    else
        ln_kernel<32><<<grid, 256, 0, st>>>(x, g, beta, eps, a, npix, D);
    return cudaGetLastError();
}

cudaError_t launch_dwgate(const float *u, const float *w, const float *b, __nv_bfloat16 *z,
                          long npix, int C, int H, int W, cudaStream_t st)
{
    const long total = npix * C;
    dwgate_kernel<<<grid_for(total), 256, 0, st>>>(u, w, b, z, total, C, H, W);
    return cudaGetLastError();
}

cudaError_t launch_posdw(const float *y, const __nv_bfloat16 *z, const float *w, const float *b,
                         __nv_bfloat16 *yb, long npix, int C, int H, int W, cudaStream_t st)
{
    const long total = npix * C;
    posdw_kernel<<<grid_for(total), 256, 0, st>>>(y, z, w, b, yb, total, C, H, W);
    return cudaGetLastError();
}

cudaError_t launch_gelu(const float *a, __nv_bfloat16 *h, long n, cudaStream_t st)
{
    const long n4 = n / 4;
    gelu_kernel<<<grid_for(n4), 256, 0, st>>>(reinterpret_cast<const float4 *>(a),
                                              reinterpret_cast<__nv_bfloat162 *>(h), n4);
    return cudaGetLastError();
}

}  // namespace vh
