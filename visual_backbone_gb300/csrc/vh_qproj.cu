// vh_qproj.cu -- the VisionHOPE-exact readout's query and skip terms ("VisionHOPE:
// Visual Backbones as Self-Modifying Learning Systems", Sec. 2.1.2 Eq. (14), App. B.5).
//
// 1-4 adjacent threads per (pixel, head): q = W_q z for the head's d output channels (fp32 FMA over
// all Cc input channels, the head's W_q rows staged transposed in shared memory so each
// input channel's d weights are broadcast vector loads),
// L2-normalised within the head with the stabiliser of the key norm, and written as three
// bf16 pieces (p1 + p2 + p3 = the fp32 value) -- the operand form the scan kernels read.
// The same thread seeds out with the channel-wise skip of the enabled routes,
// sum_r lambda_r D_r z (Eq. (26) applied to Y_r = reads + D_r Z_r), before the scans add
// their reads.
#include "vh_common.cuh"

namespace vh {
namespace {

constexpr int QP_KC = 64;   // input channels of W_q staged per pass

// Threads per (pixel, head): each thread forms OUT = min(D, 16) consecutive outputs of the
// head, and the TPH threads of a pixel are adjacent lanes (the head norm is a shuffle sum).
template <int D> struct QpShape {
    static constexpr int OUT = D < 16 ? D : 16;
    static constexpr int TPH = D / OUT;
    static constexpr int PIX = 128 / TPH;  // pixels per 128-thread CTA
};

template <int D, typename XT>
__global__ void __launch_bounds__(128)
    qproj_kernel(const XT *__restrict__ x, const float *__restrict__ wq,
                 const float *__restrict__ skip, const float *__restrict__ dir_scale,
                 unsigned dirs, __nv_bfloat16 *__restrict__ qhat, float *__restrict__ out,
                 int accumulate, long npix, int Cc, float knorm_eps)
{
    using S = QpShape<D>;
    constexpr int OUT = S::OUT, TPH = S::TPH;
    // the head's W_q rows, transposed: wt[j][i] = W_q[h*D + i][j0 + j] for one slice of
    // QP_KC input channels, so each input channel's weights are broadcast vector loads;
    // the CTA's pixel rows of that slice in fp32, row stride QP_KC + 1 (conflict-free)
    __shared__ __align__(16) float wt[QP_KC * D];
    __shared__ float zs[S::PIX * (QP_KC + 1)];
    const int part = threadIdx.x % TPH;   // which OUT outputs of the head
    const long pix = (long)blockIdx.x * S::PIX + threadIdx.x / TPH;
    const int h = blockIdx.y;
    const bool live = pix < npix;
    const XT *z = x + (live ? pix : 0) * Cc;
    const size_t o = (size_t)(live ? pix : 0) * Cc + (size_t)h * D + (size_t)part * OUT;
    if (wq) {
        float q[OUT];
#pragma unroll
        for (int i = 0; i < OUT; ++i) q[i] = 0.0f;
        const float *w = wq + (size_t)h * D * Cc;
        constexpr int EPV = 16 / (int)sizeof(XT);  // input channels per 16-byte load
        const long pix0 = (long)blockIdx.x * S::PIX;
        const int npx = (int)min((long)S::PIX, npix - pix0);
        const float *zrow = zs + (threadIdx.x / TPH) * (QP_KC + 1);
        for (int j0 = 0; j0 < Cc; j0 += QP_KC) {
            const int kc = min(QP_KC, Cc - j0);
            __syncthreads();
            for (int e = threadIdx.x; e < kc * D; e += blockDim.x) {
                const int i = e / kc, j = e % kc;  // coalesced along the W_q row
                wt[j * D + i] = w[(size_t)i * Cc + j0 + j];
            }
            // the CTA's pixel rows of this slice, 16-byte loads running along each row
            const int vpr = kc / EPV;
            for (int e = threadIdx.x; e < npx * vpr; e += blockDim.x) {
                const int pr = e / vpr, v = e % vpr;
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(x + (pix0 + pr) * Cc + j0 + v * EPV));
                const XT *el = reinterpret_cast<const XT *>(&raw);
#pragma unroll
                for (int u = 0; u < EPV; ++u) zs[pr * (QP_KC + 1) + v * EPV + u] = XElem<XT>::to_f(el[u]);
            }
            __syncthreads();
            if (live) {
                for (int j = 0; j < kc; ++j) {
                    const float zj = zrow[j];
                    const float4 *wr = reinterpret_cast<const float4 *>(wt + j * D + part * OUT);
#pragma unroll
                    for (int i4 = 0; i4 < OUT / 4; ++i4) {
                        const float4 wv = wr[i4];
                        q[4 * i4] = fmaf(wv.x, zj, q[4 * i4]);
                        q[4 * i4 + 1] = fmaf(wv.y, zj, q[4 * i4 + 1]);
                        q[4 * i4 + 2] = fmaf(wv.z, zj, q[4 * i4 + 2]);
                        q[4 * i4 + 3] = fmaf(wv.w, zj, q[4 * i4 + 3]);
                    }
                }
            }
        }
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < OUT; ++i) ss = fmaf(q[i], q[i], ss);
#pragma unroll
        for (int m = 1; m < TPH; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (live) {
            const float rq = 1.0f / sqrtf(ss + knorm_eps);
            const size_t plane = (size_t)npix * Cc;
#pragma unroll
            for (int i = 0; i < OUT; i += 8) {
                __align__(16) __nv_bfloat16 p1[8], p2[8], p3[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float v = q[i + e] * rq;
                    p1[e] = __float2bfloat16_rn(v);
                    const float r1 = v - __bfloat162float(p1[e]);
                    p2[e] = __float2bfloat16_rn(r1);
                    p3[e] = __float2bfloat16_rn(r1 - __bfloat162float(p2[e]));
                }
                *reinterpret_cast<uint4 *>(qhat + o + i) = *reinterpret_cast<const uint4 *>(p1);
                *reinterpret_cast<uint4 *>(qhat + plane + o + i) = *reinterpret_cast<const uint4 *>(p2);
                *reinterpret_cast<uint4 *>(qhat + 2 * plane + o + i) = *reinterpret_cast<const uint4 *>(p3);
            }
        }
    }
    if (skip) {
        // sum over the enabled routes of lambda_r D_r for this head's channels, once per CTA
        __shared__ __align__(16) float coef[D];
        if (threadIdx.x < D) {
            const int c = h * D + threadIdx.x;
            float sc = 0.0f;
            for (int r = 0; r < 4; ++r)
                if (dirs & (1u << r))
                    sc = fmaf(dir_scale ? dir_scale[(size_t)r * Cc + c] : 1.0f, skip[(size_t)r * Cc + c], sc);
            coef[threadIdx.x] = sc;
        }
        __syncthreads();
        if (live) {
            constexpr int EPV = 16 / (int)sizeof(XT);
            const XT *zh = z + h * D + part * OUT;
            const float *ch = coef + part * OUT;
            float *oh = out + o;
#pragma unroll
            for (int i = 0; i < OUT; i += EPV) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(zh + i));
                const XT *el = reinterpret_cast<const XT *>(&raw);
#pragma unroll
                for (int u = 0; u < EPV; u += 4) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(ch + i + u);
                    float4 v = make_float4(c4.x * XElem<XT>::to_f(el[u]), c4.y * XElem<XT>::to_f(el[u + 1]),
                                           c4.z * XElem<XT>::to_f(el[u + 2]), c4.w * XElem<XT>::to_f(el[u + 3]));
                    float4 *dst = reinterpret_cast<float4 *>(oh + i + u);
                    if (accumulate) {
                        const float4 a4 = *dst;
                        v.x += a4.x; v.y += a4.y; v.z += a4.z; v.w += a4.w;
                    }
                    *dst = v;
                }
            }
        }
    }
}

template <int D, typename XT>
cudaError_t launch_d(const void *x, const float *wq, const float *skip, const float *dir_scale,
                     unsigned dirs, __nv_bfloat16 *qhat, float *out, int accumulate, long npix,
                     int Cc, float knorm_eps, cudaStream_t st)
{
    const dim3 grid((unsigned)((npix + QpShape<D>::PIX - 1) / QpShape<D>::PIX), (unsigned)(Cc / D));
    qproj_kernel<D, XT><<<grid, 128, 0, st>>>(static_cast<const XT *>(x), wq, skip, dir_scale,
                                               dirs, qhat, out, accumulate, npix, Cc, knorm_eps);
    return cudaGetLastError();
}

}  // namespace

namespace tc {
cudaError_t launch_qproj_tc(const void *x, bool bf16, int d, const float *wq, const float *skip,
                            const float *dir_scale, unsigned dirs, __nv_bfloat16 *qhat, float *out,
                            int accumulate, long npix, int Cc, float knorm_eps, cudaStream_t st,
                            bool *handled);
}

cudaError_t launch_qproj(const void *x, bool bf16, int d, const float *wq, const float *skip,
                         const float *dir_scale, unsigned dirs, __nv_bfloat16 *qhat, float *out,
                         int accumulate, long npix, int Cc, float knorm_eps, cudaStream_t st)
{
    bool handled = false;
    const cudaError_t e = tc::launch_qproj_tc(x, bf16, d, wq, skip, dir_scale, dirs, qhat, out,
                                              accumulate, npix, Cc, knorm_eps, st, &handled);
    if (e != cudaSuccess || handled) return e;
#define VH_QP(DD)                                                                              \
    return bf16 ? launch_d<DD, __nv_bfloat16>(x, wq, skip, dir_scale, dirs, qhat, out,        \
                                               accumulate, npix, Cc, knorm_eps, st)            \
                : launch_d<DD, float>(x, wq, skip, dir_scale, dirs, qhat, out, accumulate,     \
                                      npix, Cc, knorm_eps, st)
    switch (d) {
    case 16: VH_QP(16);
    case 32: VH_QP(32);
    case 64: VH_QP(64);
    }
#undef VH_QP
    return cudaErrorInvalidValue;
}

}  // namespace vh
