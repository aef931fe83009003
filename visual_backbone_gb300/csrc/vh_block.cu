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
// The four pointwise layers are GEMMs on bf16 operands with fp32 accumulation
// (vh_gemm_tc.cu: bias, residual and FFN1's GELU in their epilogues).  The kernels here do
// the rest, each one pass over the activations: the three depthwise convolutions with
// their epilogues (CPE, the gated branch, the positional branch with the cast for
// Proj_out) and LN1 and LN2 (one warp per pixel).  bf16 rounding points: LN1's and LN2's
// outputs, Z, Y before Proj_out, FFN1's product (before its bias) and GELU's output.

#include "vh_common.cuh"

namespace vh {

// ------------------------------------------------------------------ kernels

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

// The three 3 x 3 depthwise convolutions of the block (zero padding, bias per channel),
// with their epilogues:
//   kCpe:  out_f32  = src + b + dw(src)             conditional positional encoding
//   kGate: out_bf16 = src + SiLU(b + dw(src))       gated depthwise residual branch
//   kPos:  out_bf16 = res + b + dw(src), src bf16   positional branch, cast for Proj_out
// One CTA per image row; the taps are staged transposed ([tap][channel]) in shared
// memory, and a thread handles four consecutive channels of one pixel (16-byte loads).
enum DwMode { kCpe = 0, kGate = 1, kPos = 2 };

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    static __device__ __forceinline__ float4 load(const float *p) { return *reinterpret_cast<const float4 *>(p); }
};
template <> struct Vec4<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load(const __nv_bfloat16 *p)
    {
        const uint2 r = *reinterpret_cast<const uint2 *>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&r.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
};

template <int kMode, typename TIn>
__global__ void __launch_bounds__(256) dw3_kernel(const TIn *__restrict__ src,
                                                  const float *__restrict__ res,
                                                  const float *__restrict__ w,
                                                  const float *__restrict__ bias,
                                                  void *__restrict__ out, int H, int W, int C)
{
    extern __shared__ float sw[];  // [9][C] taps, then [C] bias
    for (int e = threadIdx.x; e < 9 * C; e += blockDim.x) sw[(e % 9) * C + e / 9] = w[e];
    for (int e = threadIdx.x; e < C; e += blockDim.x) sw[9 * C + e] = bias[e];
    __syncthreads();
    const int row = blockIdx.x;  // b * H + i
    const int i = row % H;
    const int C4 = C >> 2;
    for (int t = threadIdx.x; t < W * C4; t += blockDim.x) {
        const int j = t / C4, c = (t - j * C4) * 4;
        float4 acc = *reinterpret_cast<const float4 *>(sw + 9 * C + c);
#pragma unroll
        for (int di = -1; di <= 1; ++di) {
            if (i + di < 0 || i + di >= H) continue;
#pragma unroll
            for (int dj = -1; dj <= 1; ++dj) {
                if (j + dj < 0 || j + dj >= W) continue;
                const float4 v = Vec4<TIn>::load(src + ((size_t)(row + di) * W + j + dj) * C + c);
                const float4 k = *reinterpret_cast<const float4 *>(sw + ((di + 1) * 3 + dj + 1) * C + c);
                acc.x = fmaf(k.x, v.x, acc.x);
                acc.y = fmaf(k.y, v.y, acc.y);
                acc.z = fmaf(k.z, v.z, acc.z);
                acc.w = fmaf(k.w, v.w, acc.w);
            }
        }
        const size_t e = ((size_t)row * W + j) * C + c;
        if (kMode == kCpe) {
            const float4 x = Vec4<TIn>::load(src + e);
            *reinterpret_cast<float4 *>(static_cast<float *>(out) + e) =
                make_float4(x.x + acc.x, x.y + acc.y, x.z + acc.z, x.w + acc.w);
        } else {
            float4 r;
            if (kMode == kGate) {
                const float4 u = Vec4<TIn>::load(src + e);
                r = make_float4(u.x + acc.x / (1.0f + __expf(-acc.x)),
                                u.y + acc.y / (1.0f + __expf(-acc.y)),
                                u.z + acc.z / (1.0f + __expf(-acc.z)),
                                u.w + acc.w / (1.0f + __expf(-acc.w)));
            } else {
                const float4 y = *reinterpret_cast<const float4 *>(res + e);
                r = make_float4(y.x + acc.x, y.y + acc.y, y.z + acc.z, y.w + acc.w);
            }
            __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(out) + e);
            o[0] = __floats2bfloat162_rn(r.x, r.y);
            o[1] = __floats2bfloat162_rn(r.z, r.w);
        }
    }
}

// ------------------------------------------------------------------ launches

cudaError_t launch_ln(const float *x, const float *g, const float *beta, float eps,
                      __nv_bfloat16 *a, long npix, int D, cudaStream_t st);

namespace {

unsigned grid_for(long threads)
{
    long g = (threads + 255) / 256;
    const long cap = 152L * 16;  // a few waves of resident blocks; grid-stride beyond
    return (unsigned)(g < cap ? (g > 0 ? g : 1) : cap);
}

}  // namespace

// CPE (x0 = x + dw(x) + b, fp32) then LN1 (bf16), two bandwidth-bound passes.
cudaError_t launch_cpe_ln(const float *x, const float *cw, const float *cb, const float *g,
                          const float *beta, float eps, float *x0, __nv_bfloat16 *a, int B, int H,
                          int W, int D, cudaStream_t st)
{
    const size_t sm = (size_t)10 * D * sizeof(float);
    dw3_kernel<kCpe, float><<<B * H, 256, sm, st>>>(x, nullptr, cw, cb, x0, H, W, D);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_ln(x0, g, beta, eps, a, (long)B * H * W, D, st);
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
    const int rows = (int)(npix / W);
    dw3_kernel<kGate, float><<<rows, 256, (size_t)10 * C * sizeof(float), st>>>(u, nullptr, w, b, z,
                                                                              H, W, C);
    return cudaGetLastError();
}

cudaError_t launch_posdw(const float *y, const __nv_bfloat16 *z, const float *w, const float *b,
                         __nv_bfloat16 *yb, long npix, int C, int H, int W, cudaStream_t st)
{
    const int rows = (int)(npix / W);
    dw3_kernel<kPos, __nv_bfloat16><<<rows, 256, (size_t)10 * C * sizeof(float), st>>>(
        z, y, w, b, yb, H, W, C);
    return cudaGetLastError();
}


}  // namespace vh
