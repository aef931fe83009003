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

// v = p1 + p2 + p3 with bf16 pieces, each the rounding of what the previous ones leave
// (24 significant bits: the fp32-intermediate test mode's GEMM operands).
__device__ __forceinline__ void split3_bf16x2(float v0, float v1, __nv_bfloat162 &p1, __nv_bfloat162 &p2,
                                              __nv_bfloat162 &p3)
{
    p1 = __floats2bfloat162_rn(v0, v1);
    const float2 f1 = __bfloat1622float2(p1);
    const float r0 = v0 - f1.x, r1 = v1 - f1.y;
    p2 = __floats2bfloat162_rn(r0, r1);
    const float2 f2 = __bfloat1622float2(p2);
    p3 = __floats2bfloat162_rn(r0 - f2.x, r1 - f2.y);
}

// Per pixel (one warp): a = bf16(LN(x) * g + beta), or with kSplit its three bf16 pieces
// a[pix][c], a[pix][D + c], a[pix][2D + c] (fp32-intermediate test mode).  A lane holds
// channel pairs 2 lane + 64 m (8-byte loads, bf16x2 stores); the scale and shift of its
// channels stay in registers across the pixels it visits.  D even, x 8-byte aligned rows.
template <int MAXP, bool kSplit>
__global__ void __launch_bounds__(256) ln_kernel(const float *__restrict__ x,
                                                 const float *__restrict__ g,
                                                 const float *__restrict__ beta, float eps,
                                                 __nv_bfloat16 *__restrict__ a, long npix, int D)
{
    const int lane = threadIdx.x & 31;
    float2 gv[MAXP], bv[MAXP];
#pragma unroll
    for (int m = 0; m < MAXP; ++m) {
        const int c = 2 * lane + 64 * m;
        gv[m] = c < D ? make_float2(g[c], g[c + 1]) : make_float2(0.0f, 0.0f);
        bv[m] = c < D ? make_float2(beta[c], beta[c + 1]) : make_float2(0.0f, 0.0f);
    }
    for (long pix = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5; pix < npix;
         pix += ((long)gridDim.x * blockDim.x) >> 5) {
        float2 v[MAXP];
        float s = 0.0f;
#pragma unroll
        for (int m = 0; m < MAXP; ++m) {
            const int c = 2 * lane + 64 * m;
            v[m] = c < D ? *reinterpret_cast<const float2 *>(x + pix * D + c) : make_float2(0.0f, 0.0f);
            s += v[m].x + v[m].y;
        }
        const float mu = warp_sum(s) / D;
        float q = 0.0f;
#pragma unroll
        for (int m = 0; m < MAXP; ++m)
            if (2 * lane + 64 * m < D) {
                q = fmaf(v[m].x - mu, v[m].x - mu, q);
                q = fmaf(v[m].y - mu, v[m].y - mu, q);
            }
        const float rs = rsqrtf(warp_sum(q) / D + eps);
#pragma unroll
        for (int m = 0; m < MAXP; ++m) {
            const int c = 2 * lane + 64 * m;
            if (c < D) {
                const float o0 = (v[m].x - mu) * rs * gv[m].x + bv[m].x;
                const float o1 = (v[m].y - mu) * rs * gv[m].y + bv[m].y;
                if (kSplit) {
                    __nv_bfloat162 p1, p2, p3;
                    split3_bf16x2(o0, o1, p1, p2, p3);
                    *reinterpret_cast<__nv_bfloat162 *>(a + pix * 3 * D + c) = p1;
                    *reinterpret_cast<__nv_bfloat162 *>(a + pix * 3 * D + D + c) = p2;
                    *reinterpret_cast<__nv_bfloat162 *>(a + pix * 3 * D + 2 * D + c) = p3;
                } else {
                    *reinterpret_cast<__nv_bfloat162 *>(a + pix * D + c) = __floats2bfloat162_rn(o0, o1);
                }
            }
        }
    }
}

// The three 3 x 3 depthwise convolutions of the block (zero padding, bias per channel),
// with their epilogues:
//   kCpe:  out_f32  = src + b + dw(src)             conditional positional encoding
//   kGate: out_bf16 = src + SiLU(b + dw(src))       gated depthwise residual branch
//   kPos:  out_bf16 = res + b + dw(src), src bf16   positional branch, cast for Proj_out
// and, for the fp32-intermediate test mode, kGateF32 (the gated branch with fp32 out) and
// kPosSplit (src fp32, out the three bf16 pieces of the positional sum, [pixel][3C]).
// One CTA per image row.  A thread takes four consecutive channels (16-byte loads) of NP
// neighbouring pixels: each tap loaded from shared memory serves all of them, and they
// share the columns of their 3 x 3 windows (3 (NP + 2) 16-byte loads for NP outputs
// instead of 9 NP).  The taps are summed in the order (di, dj) = (-1, -1), (-1, 0), ... (1, 1),
// starting from the bias; taps outside the map are skipped.
enum DwMode { kCpe = 0, kGate = 1, kPos = 2, kGateF32 = 3, kPosSplit = 4 };

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

__device__ __forceinline__ void fma4(float4 &acc, const float4 k, const float4 v)
{
    acc.x = fmaf(k.x, v.x, acc.x);
    acc.y = fmaf(k.y, v.y, acc.y);
    acc.z = fmaf(k.z, v.z, acc.z);
    acc.w = fmaf(k.w, v.w, acc.w);
}

template <int kMode, typename TIn>
__device__ __forceinline__ void dw3_store(const TIn *__restrict__ src, const float *__restrict__ res,
                                          void *__restrict__ out, size_t e, float4 acc, int C)
{
    if (kMode == kCpe) {
        const float4 x = Vec4<TIn>::load(src + e);
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + e) =
            make_float4(x.x + acc.x, x.y + acc.y, x.z + acc.z, x.w + acc.w);
    } else if (kMode == kGateF32) {
        const float4 u = Vec4<TIn>::load(src + e);
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + e) =
            make_float4(u.x + acc.x / (1.0f + __expf(-acc.x)), u.y + acc.y / (1.0f + __expf(-acc.y)),
                        u.z + acc.z / (1.0f + __expf(-acc.z)), u.w + acc.w / (1.0f + __expf(-acc.w)));
    } else if (kMode == kPosSplit) {
        // e = pix * C + c: the pieces go to [pix][c], [pix][C + c], [pix][2C + c]
        const float4 y = *reinterpret_cast<const float4 *>(res + e);
        const float4 r = make_float4(y.x + acc.x, y.y + acc.y, y.z + acc.z, y.w + acc.w);
        const size_t pix = e / C, c = e - pix * C;
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out) + pix * 3 * C + c;
        __nv_bfloat162 p1, p2, p3, q1, q2, q3;
        split3_bf16x2(r.x, r.y, p1, p2, p3);
        split3_bf16x2(r.z, r.w, q1, q2, q3);
        reinterpret_cast<__nv_bfloat162 *>(o)[0] = p1;
        reinterpret_cast<__nv_bfloat162 *>(o)[1] = q1;
        reinterpret_cast<__nv_bfloat162 *>(o + C)[0] = p2;
        reinterpret_cast<__nv_bfloat162 *>(o + C)[1] = q2;
        reinterpret_cast<__nv_bfloat162 *>(o + 2 * C)[0] = p3;
        reinterpret_cast<__nv_bfloat162 *>(o + 2 * C)[1] = q3;
    } else {
        float4 r;
        if (kMode == kGate) {
            const float4 u = Vec4<TIn>::load(src + e);
            r = make_float4(u.x + acc.x / (1.0f + __expf(-acc.x)), u.y + acc.y / (1.0f + __expf(-acc.y)),
                            u.z + acc.z / (1.0f + __expf(-acc.z)), u.w + acc.w / (1.0f + __expf(-acc.w)));
        } else {
            const float4 y = *reinterpret_cast<const float4 *>(res + e);
            r = make_float4(y.x + acc.x, y.y + acc.y, y.z + acc.z, y.w + acc.w);
        }
        __nv_bfloat162 *o = reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(out) + e);
        o[0] = __floats2bfloat162_rn(r.x, r.y);
        o[1] = __floats2bfloat162_rn(r.z, r.w);
    }
}

template <int kMode, typename TIn, int NP>
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
    const int C4 = C >> 2, Wp = (W + NP - 1) / NP;
    for (int t = threadIdx.x; t < Wp * C4; t += blockDim.x) {
        const int j = NP * (t / C4), c = (t - (t / C4) * C4) * 4;
        float4 acc[NP];
        acc[0] = *reinterpret_cast<const float4 *>(sw + 9 * C + c);
#pragma unroll
        for (int q = 1; q < NP; ++q) acc[q] = acc[0];
#pragma unroll
        for (int di = -1; di <= 1; ++di) {
            if (i + di < 0 || i + di >= H) continue;
            const TIn *p = src + ((size_t)(row + di) * W + j) * C + c;
            // columns j-1 .. j+NP of this row (those outside the map are not read)
            float4 v[NP + 2];
#pragma unroll
            for (int q = 0; q < NP + 2; ++q) {
                const int jj = j - 1 + q;
                v[q] = (jj >= 0 && jj < W) ? Vec4<TIn>::load(p + (q - 1) * C)
                                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int dj = -1; dj <= 1; ++dj) {
                const float4 k = *reinterpret_cast<const float4 *>(sw + ((di + 1) * 3 + dj + 1) * C + c);
#pragma unroll
                for (int q = 0; q < NP; ++q)
                    if (j + q + dj >= 0 && j + q + dj < W) fma4(acc[q], k, v[q + dj + 1]);
            }
        }
        const size_t e = ((size_t)row * W + j) * C + c;
#pragma unroll
        for (int q = 0; q < NP; ++q)
            if (j + q < W) dw3_store<kMode, TIn>(src, res, out, e + (size_t)q * C, acc[q], C);
    }
}

template <int kMode, typename TIn>
cudaError_t launch_dw3(const TIn *src, const float *res, const float *w, const float *b, void *out,
                       int rows, int H, int W, int C, cudaStream_t st)
{
    // four pixels a thread when that still leaves every thread two or more of them (CPE at
    // 192 channels), else two
    const size_t sm = (size_t)10 * C * sizeof(float);
    if ((C >> 2) * ((W + 3) / 4) >= 2 * 256)
        dw3_kernel<kMode, TIn, 4><<<rows, 256, sm, st>>>(src, res, w, b, out, H, W, C);
    else
        dw3_kernel<kMode, TIn, 2><<<rows, 256, sm, st>>>(src, res, w, b, out, H, W, C);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ launches

cudaError_t launch_ln(const float *x, const float *g, const float *beta, float eps,
                      __nv_bfloat16 *a, long npix, int D, bool split, cudaStream_t st);

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
                          int W, int D, bool split, cudaStream_t st)
{
    cudaError_t e = launch_dw3<kCpe, float>(x, nullptr, cw, cb, x0, B * H, H, W, D, st);
    if (e != cudaSuccess) return e;
    return launch_ln(x0, g, beta, eps, a, (long)B * H * W, D, split, st);
}

// LayerNorm of each pixel's D channels to bf16 (split: its three pieces, [pixel][3D]).
cudaError_t launch_ln(const float *x, const float *g, const float *beta, float eps,
                      __nv_bfloat16 *a, long npix, int D, bool split, cudaStream_t st)
{
    const unsigned grid = grid_for(npix * 32);
    if (D <= 256) {
        if (split)
            ln_kernel<4, true><<<grid, 256, 0, st>>>(x, g, beta, eps, a, npix, D);
        else
            ln_kernel<4, false><<<grid, 256, 0, st>>>(x, g, beta, eps, a, npix, D);
    } else {
        if (split)
            ln_kernel<16, true><<<grid, 256, 0, st>>>(x, g, beta, eps, a, npix, D);
        else
            ln_kernel<16, false><<<grid, 256, 0, st>>>(x, g, beta, eps, a, npix, D);
    }
    return cudaGetLastError();
}

// Z = U + SiLU(DW(U) + b): bf16 Z, or fp32 Z (f32).
cudaError_t launch_dwgate(const float *u, const float *w, const float *b, void *z, long npix, int C,
                          int H, int W, bool f32, cudaStream_t st)
{
    if (f32) return launch_dw3<kGateF32, float>(u, nullptr, w, b, z, (int)(npix / W), H, W, C, st);
    return launch_dw3<kGate, float>(u, nullptr, w, b, z, (int)(npix / W), H, W, C, st);
}

// Y + DW(Z) + b for Proj_out: bf16 from bf16 Z, or (f32) the three bf16 pieces from fp32 Z.
cudaError_t launch_posdw(const float *y, const void *z, const float *w, const float *b, void *yb,
                         long npix, int C, int H, int W, bool f32, cudaStream_t st)
{
    if (f32)
        return launch_dw3<kPosSplit, float>(static_cast<const float *>(z), y, w, b, yb, (int)(npix / W),
                                            H, W, C, st);
    return launch_dw3<kPos, __nv_bfloat16>(static_cast<const __nv_bfloat16 *>(z), y, w, b, yb,
                                           (int)(npix / W), H, W, C, st);
}


}  // namespace vh
