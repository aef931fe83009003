// vh_qproj.cu -- the VisionHOPE-exact readout's query and skip terms ("VisionHOPE:
// Visual Backbones as Self-Modifying Learning Systems", Sec. 2.1.2 Eq. (14), App. B.5).
//
// One thread per (pixel, head): q = W_q z for the head's d output channels (fp32 FMA over
// all Cc input channels; the warp shares the head, so W_q rows are broadcast loads),
// L2-normalised within the head with the stabiliser of the key norm, and written as three
// bf16 pieces (p1 + p2 + p3 = the fp32 value) -- the operand form the scan kernels read.
// The same thread seeds out with the channel-wise skip of the enabled routes,
// sum_r lambda_r D_r z (Eq. (26) applied to Y_r = reads + D_r Z_r), before the scans add
// their reads.
#include "vh_common.cuh"

namespace vh {
namespace {

template <int D, typename XT>
__global__ void __launch_bounds__(128)
    qproj_kernel(const XT *__restrict__ x, const float *__restrict__ wq,
                 const float *__restrict__ skip, const float *__restrict__ dir_scale,
                 unsigned dirs, __nv_bfloat16 *__restrict__ qhat, float *__restrict__ out,
                 int accumulate, long npix, int Cc, float knorm_eps)
{
    const long pix = (long)blockIdx.x * blockDim.x + threadIdx.x;
    const int h = blockIdx.y;
    if (pix >= npix) return;
    const XT *z = x + pix * Cc;
    const size_t o = (size_t)pix * Cc + (size_t)h * D;
    if (wq) {
        float q[D];
#pragma unroll
        for (int i = 0; i < D; ++i) q[i] = 0.0f;
        const float *w = wq + (size_t)h * D * Cc;
        for (int j = 0; j < Cc; ++j) {
            const float zj = XElem<XT>::to_f(z[j]);
#pragma unroll
            for (int i = 0; i < D; ++i) q[i] = fmaf(__ldg(w + (size_t)i * Cc + j), zj, q[i]);
        }
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < D; ++i) ss = fmaf(q[i], q[i], ss);
        const float rq = 1.0f / sqrtf(ss + knorm_eps);
        const size_t plane = (size_t)npix * Cc;
#pragma unroll
        for (int i = 0; i < D; i += 8) {
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
    if (skip) {
        for (int i = 0; i < D; ++i) {
            const int c = h * D + i;
            float s = 0.0f;
            for (int r = 0; r < 4; ++r)
                if (dirs & (1u << r))
                    s = fmaf(dir_scale ? dir_scale[(size_t)r * Cc + c] : 1.0f, skip[(size_t)r * Cc + c], s);
            const float v = s * XElem<XT>::to_f(z[c]);
            out[o + i] = accumulate ? out[o + i] + v : v;
        }
    }
}

template <int D, typename XT>
cudaError_t launch_d(const void *x, const float *wq, const float *skip, const float *dir_scale,
                     unsigned dirs, __nv_bfloat16 *qhat, float *out, int accumulate, long npix,
                     int Cc, float knorm_eps, cudaStream_t st)
{
    const dim3 grid((unsigned)((npix + 127) / 128), (unsigned)(Cc / D));
    qproj_kernel<D, XT><<<grid, 128, 0, st>>>(static_cast<const XT *>(x), wq, skip, dir_scale,
                                               dirs, qhat, out, accumulate, npix, Cc, knorm_eps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qproj(const void *x, bool bf16, int d, const float *wq, const float *skip,
                         const float *dir_scale, unsigned dirs, __nv_bfloat16 *qhat, float *out,
                         int accumulate, long npix, int Cc, float knorm_eps, cudaStream_t st)
{
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
