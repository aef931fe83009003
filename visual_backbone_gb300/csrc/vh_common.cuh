// vh_common.cuh -- device helpers shared by the scan kernels of libvh.
//
// Method: "VisionHOPE: Visual Backbones as Self-Modifying Learning Systems"
// (Sec. 2.1-2.3, App. B.3-B.5, App. C.1) with the six-memory set of "Nested
// Learning: The Illusion of Deep Learning Architectures", part 12,
// Eqs. (94)-(96).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "vh.h"

namespace vh {

// Everything a scan kernel needs, by value (kernel parameter space).
struct ScanArgs {
    const void *x;            // [B][H][W][Cc]
    const float *mem0;        // [4][nh][4d^2+2d]
    float *out;               // [B][H][W][Cc] fp32, zeroed before the scan kernels run
    float *mem_out;           // [B][4][nh][4d^2+2d] or nullptr
    const float *dir_scale;   // [4][Cc] or nullptr
    unsigned long long *stats;
    int B, H, W, nh, Cc;
    int dir_list[4];          // enabled routes in ascending order
    int ndirs;
    int chunk;                // 0 = aligned
    // method constants in fp32 (Def. 1, App. B.3, App. C.1)
    float gamma_eta, alpha_logit, eta_bias, eps, knorm_eps;
    float inj_factor;         // 1 - inj_inward
    float spec_factor;        // 1 - spec_inward
    float kk_floor;
    int gate_mode;
    float forced_eta, forced_alpha;
    unsigned control_flags;
    // VisionHOPE-exact readout: normalised outer queries as three bf16 pieces
    // [3][B][H][W][Cc] (piece p at qhat + p * B*H*W*Cc); nullptr = q from M^q
    const __nv_bfloat16 *qhat;
    // backward support: when set, the boundary state of every chunk of scan i is written
    // to ckpt + i * ckpt_stride + chunk * (4d^2 + 2d) (fp32, state layout)
    float *ckpt;
    size_t ckpt_stride;
    // backward support: when set (with ckpt), route token t of scan i leaves its record at
    // rec + i * rec_stride + t * (3d + 8): k, q, delta (normalised, fp32), then
    // |k_raw|^2, s_eta, s_alpha, |k|^2, |delta|^2, |q_raw|^2 and two unused slots
    float *rec;
    size_t rec_stride;
    // bounded waits: cycles before a wait gives up (0 = 2^32); test hook that never issues
    // the first input copy (head_dim 32 tensor-core kernel)
    long long wait_limit;
    int withhold_first_copy;
};

// Checked index of a VH_DEBUG_BOUNDS build: elements [i, i + n) of an array of `total`
// elements.  A failed check is counted in stats[VH_STAT_BOUNDS] (when stats are given) and
// the caller skips the access.  In other builds the check compiles to `true`.
#ifdef VH_DEBUG_BOUNDS
__device__ __forceinline__ bool vh_in_bounds(unsigned long long *stats, size_t i, size_t n,
                                             size_t total)
{
    const bool ok = i <= total && n <= total - i;  // a negative index wraps to a huge i
    if (!ok && stats) atomicAdd(stats + VH_STAT_BOUNDS, 1ull);
    return ok;
}
#define VH_IN(stats, i, n, total) ::vh::vh_in_bounds((stats), (size_t)(i), (size_t)(n), (size_t)(total))
#else
#define VH_IN(stats, i, n, total) true
#endif

// Element counts of the arrays a scan reads and writes (for the checked indices).
__host__ __device__ __forceinline__ size_t map_elems(const ScanArgs &a)
{
    return (size_t)a.B * a.H * a.W * a.Cc;
}
__host__ __device__ __forceinline__ size_t state_elems(const ScanArgs &a, int d)
{
    return (size_t)4 * d * d + 2 * d;
}

// Floats of one token record (layout above); the scalar slots follow the three vectors.
__host__ __device__ constexpr int token_rec_floats(int d) { return 3 * d + 8; }
enum { TR_KK = 0, TR_SE = 1, TR_SA = 2, TR_KN2 = 3, TR_DD = 4, TR_QQ = 5 };

// Arguments of the backward scan kernel.
struct BwdArgs {
    ScanArgs s;                // forward arguments (out, mem_out, stats, qhat unused)
    const float *dout;         // [B][H][W][Cc]
    const float *dmem_final;   // [B][4][nh][4d^2+2d] or nullptr
    float *dx;                 // [B][H][W][Cc], zeroed before the launch
    float *dmem0;              // [4][nh][4d^2+2d], zeroed before the launch
    float *ws;                 // per scan: nck boundary states, lmax gain slices and records
    int nck, lmax;
    int have_ckpt;             // the boundary states are already in ws (tensor-core forward)
                               // s.rec set: so are the token records
};

// fp32 value of element e of the three-piece query planes (the pieces sum exactly).
__device__ __forceinline__ float qhat_at(const __nv_bfloat16 *q, size_t plane, size_t e)
{
    return (__bfloat162float(q[e]) + __bfloat162float(q[e + plane])) +
           __bfloat162float(q[e + 2 * plane]);
}

// Pixel visited at step t of route r on an H x W map (Eq. (24); the route
// orders of the VMamba explainer: row-major, full reversal, transpose then
// flatten, full reversal).
__host__ __device__ __forceinline__ int route_pixel(int r, int t, int H, int W)
{
    const int N = H * W;
    const int s = (r & 1) ? (N - 1 - t) : t;
    return (r < 2) ? s : (s % H) * W + s / H;
}

// Chunk length of route r, Eq. (25) when chunk == 0.
__host__ __device__ __forceinline__ int route_chunk(int r, int chunk, int H, int W)
{
    return chunk > 0 ? chunk : (r < 2 ? W : H);
}

__device__ __forceinline__ float softplus_f(float s)
{
    return fmaxf(s, 0.0f) + log1pf(__expf(-fabsf(s)));
}

// Per-token scalars of the step-size control (Def. 1, Eqs. (19)-(20)) with
// the App. B.3 safeguards: inward factors on both limits, ||k||^2 floored,
// the spectral limit rounded toward zero.  kk = ||k||^2, dd = ||delta||^2.
struct StepOut {
    float eta_tilde;
    bool spec_active;    // spectral limit strictly below the candidate
    bool inj_ratio_gt1;  // raw step above the injection limit
};

// `oma` = 1 - alpha, passed separately so it keeps its relative precision near alpha = 1.
// Quotients use the hardware reciprocal (a few ulp): far inside the fp32 path's error.
// kAbl = false compiles the method as defined (every ablation switch off).
template <bool kAbl = true>
__device__ __forceinline__ StepOut step_control(const ScanArgs &a, float eta, float alpha,
                                                float oma, float kk, float dd)
{
    StepOut o;
    const float r = sqrtf(dd + a.eps * a.eps) + a.eps;
    const float eta_inj = __fdividef(a.inj_factor * oma, r);
    float eta_bar;
    if (kAbl && (a.control_flags & VH_CTRL_NO_INJ_CAP))
        eta_bar = eta;
    else if (kAbl && (a.control_flags & VH_CTRL_HARD_INJ))
        eta_bar = fminf(eta, eta_inj);  // injection clamp (ablation)
    else if (eta_inj > 0.0f)
        eta_bar = eta_inj * (-expm1f(-__fdividef(eta, eta_inj)));
    else
        eta_bar = 0.0f;  // limit of Eq. (19) when the injection limit vanishes
    float spec = __fdividef(a.spec_factor * 2.0f * alpha, fmaxf(kk, a.kk_floor));
    // one step toward zero (spec >= 0): the next representable value below
    if (spec > 0.0f) spec = __int_as_float(__float_as_int(spec) - 1);
    const bool clamp = !(kAbl && (a.control_flags & VH_CTRL_NO_SPEC_CLAMP));
    o.spec_active = clamp && spec < eta_bar;
    if (kAbl && clamp && (a.control_flags & VH_CTRL_SOFT_SPEC))  // soft spectral cap (ablation)
        o.eta_tilde = spec > 0.0f ? spec * (-expm1f(-__fdividef(eta_bar, spec))) : 0.0f;
    else
        o.eta_tilde = o.spec_active ? spec : eta_bar;
    o.inj_ratio_gt1 = eta > eta_inj;
    return o;
}

// Row o of the (4d + 2) x d state (k, v, q, m memories, then the eta and alpha rows) is
// held fixed within the image by an ablation switch.
template <bool kAbl = true>
__device__ __forceinline__ bool frozen_row(const ScanArgs &a, int o, int d)
{
    return kAbl && (((a.control_flags & VH_CTRL_FREEZE_KV) && o < 2 * d) ||
                    ((a.control_flags & VH_CTRL_FREEZE_DYN) && o >= 4 * d));
}

// Raw step and retention from the scalar memory outputs, Eq. (53).
// Also returns oma = 1 - alpha: for the sigmoid, e / (1 + e) = e alpha with
// e = exp(-(s + logit alpha_init)), free of the cancellation in 1 - alpha.
__device__ __forceinline__ void gates(const ScanArgs &a, float s_eta, float s_alpha,
                                      float &eta, float &alpha, float &oma)
{
    if (a.gate_mode == VH_GATE_GENERATED) {
        eta = a.gamma_eta * softplus_f(s_eta + a.eta_bias);
        const float e = __expf(-(s_alpha + a.alpha_logit));
        alpha = __frcp_rn(1.0f + e);
        oma = alpha > 0.0f ? e * alpha : 1.0f;
    } else {
        eta = a.forced_eta;
        alpha = a.forced_alpha;
        oma = 1.0f - a.forced_alpha;
    }
}

template <typename T> struct XElem;
template <> struct XElem<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
};
template <> struct XElem<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
};

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace vh
