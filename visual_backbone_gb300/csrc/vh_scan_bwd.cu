// vh_scan_bwd.cu -- outer gradients of the four-direction VisionHOPE memory scan on
// fp32 CUDA cores: the gradients of <dout, out> + <dmem_final, memories_final> with
// respect to x and memories0.
//
// "VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.1.2: the
// recurrence is explicit and differentiable, so outer gradients pass through the memory
// trajectory without an inner solver.  Sec. 3.4 Eq. (60) budgets the activation storage
// of training as token quantities plus one d x d gain per chunk, head and route; here
// each chunk keeps its boundary state (the state is 4d + 2 rows of the gain's width) and
// the gains are re-formed chunk by chunk in the reverse pass.
//
// One CTA owns one scan (image b, route r, head h).
//  Pass 1 (forward): the state recurrence of the forward kernel without the readout; the
//    boundary state S_b of every chunk goes to the workspace.  Where the tensor-core
//    forward runs (d = 32, bf16, aligned chunks) it writes these states instead, in a
//    launch of its own before this kernel, and pass 1 is skipped.
//  Pass 2 (reverse, from the last chunk), holding dS = dL/dS_end of the chunk (dmem_final,
//    or zero, for the last one):
//    a. S_b is reloaded and the chunk's tokens regenerated tile by tile (Eq. (15),
//       App. C.1 normalisation, Eq. (53) gates, Def. 1 step control), or, after the
//       tensor-core forward, read from the token records it wrote; their quantities are
//       recorded in the workspace and the shared gain (Prop. 2, Eq. (46)) re-advanced,
//       every thread keeping its slice of G_{t-1} for every fourth token and z_t for all;
//    b. the chunk end S_end = S_b G_L gives the gain adjoint P_L = S_b^T dS, and
//       dS <- dS G_L^T;
//    c. with z_t = G_{t-1} k_t + delta_t, G_t = alpha_t G_{t-1} - eta_t z_t k_t^T (which
//       also rebuilds the slices between the stored ones, with no reduction), so the
//       adjoint runs backwards as P_{t-1} = alpha_t P_t - eta_t (P_t k_t) k_t^T and gives,
//       with u_t = P_t k_t,
//         dalpha_t = <P_t, G_{t-1}>,  deta_t = -z_t . u_t,  ddelta_t = -eta_t u_t,
//         dk_t = -eta_t (G_{t-1}^T u_t + P_t^T z_t);
//    d. per token, in parallel: the readout y = M^m_b q (Eq. (16)) with dy = lambda_r dout
//       at the token's pixel, the executed step, the gates, delta = k - v and the two
//       normalisations are differentiated; dx_t collects the generation memories'
//       transposes applied to the generated quantities' adjoints, added at the pixel
//       over the routes (Eq. (26));
//    e. the generation and readout adjoints add their outer products with x_t and q_t to
//       dS, which then holds dL/dS_b: the chunk-end adjoint of the previous chunk.
//  After chunk 0, dS is the gradient of memories0, summed over the batch.
// The branch of the step control (soft injection cap or spectral limit) follows the
// forward's choice; the one-step rounding of the spectral limit passes the gradient of
// the unrounded value.  The method as defined only: no ablation switch, no outer query.
#include "vh_common.cuh"

namespace vh {

// One slice of G_{t-1} is kept per this many tokens of a chunk.
constexpr int kGainGroup = 4;

template <int D>
struct BwdCfg {
    static constexpr int NT = 256;
    static constexpr int NW = NT / 32;
    static constexpr int R = 4 * D + 2;     // rows of the state
    static constexpr int SS = D + 4;        // row stride: 16-byte rows, no two rows in a bank quad
    static constexpr int T = D == 16 ? 64 : 16;   // token tile
    static constexpr int MINB = D == 64 ? 1 : 3;  // resident CTAs per SM (one wave at stage 1)
    static constexpr int JB = 4;                  // tokens per register block (generation)
    static constexpr int GS = kGainGroup;         // tokens per stored slice of the gain
    static constexpr int TPR = NT / D;      // threads per gain row
    static constexpr int CPT = D / TPR;     // gain columns per thread
    static constexpr int RW = 32 / TPR;     // gain rows per warp
    static constexpr int CPL = (D + 31) / 32;
    static constexpr int PS = 3 * D + 4;    // generation outputs k_raw v q_raw s_eta s_alpha
                                            // (16-byte rows)
    static constexpr int NSC = 16;          // scalars per token
    static constexpr int TRS = token_rec_floats(D);  // token record: k q delta, raw scalars
    static constexpr int GRS = D + NSC;              // gain record: G_{t-1} k, scalars
    // scalar slots
    static constexpr int S_NK = 0, S_NQ = 1, S_SE = 2, S_AL = 4, S_OMA = 5, S_ETA = 6,
                         S_ET = 7, S_INJ = 8, S_BAR = 9, S_SPEC = 10, S_R = 11, S_BR = 12,
                         S_KN2 = 13, S_DD = 14, S_PIX = 15;
    static constexpr int OFF_S = 0;
    static constexpr int OFF_DS = OFF_S + R * SS;
    static constexpr int OFF_GT = OFF_DS + R * SS;   // chunk-end gain (pass 1) / its transpose
    static constexpr int OFF_X = OFF_GT + D * D;
    static constexpr int OFF_P = OFF_X + T * D;      // generation outputs / their adjoints
    static constexpr int OFF_K = OFF_P + T * PS;
    static constexpr int OFF_DL = OFF_K + T * D;
    static constexpr int OFF_Q = OFF_DL + T * D;
    static constexpr int OFF_Z = OFF_Q + T * D;      // z = G_{t-1} k + delta
    static constexpr int OFF_SC = OFF_Z + T * D;
    static constexpr int OFF_KG = OFF_SC + T * NSC;  // dk from the gain
    static constexpr int OFF_DG = OFF_KG + T * D;    // ddelta from the gain
    static constexpr int OFF_Y = OFF_DG + T * D;     // dy
    static constexpr int OFF_UV = OFF_Y + T * D;     // per (token, row): u = P k and <p, g>
    static constexpr int OFF_PIX = OFF_UV + 2 * T * D;
    static constexpr int FLOATS = OFF_PIX + T;
    static constexpr size_t BYTES = (size_t)FLOATS * 4;
    static_assert(TPR * CPT == D && TPR <= 32, "gain thread map");
    static_assert(T % GS == 0, "tiles hold whole groups of stored gain slices");
    static_assert(BYTES <= 227 * 1024, "shared memory");
};

// Asynchronous global -> shared copies (16 or 4 bytes) and the wait for all of them.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Column sums over the rows held by one warp, added (times `scale`) to dst[0..D): each
// lane holds v[0..CPT) for columns gc0.. of its row.  Every level halves the value set
// (a lane keeps one half and receives its partner's copy of it), so a lane ends with the
// warp's sums of CPT / RW columns; when CPT < RW the last levels add duplicates, and
// only one lane of each duplicate set writes.
template <int D>
__device__ __forceinline__ void col_sums_add(float (&v)[BwdCfg<D>::CPT], int lane, int gc0,
                                             float *dst, float scale)
{
    using C = BwdCfg<D>;
    int off = 0;
    unsigned dup = 0;
#pragma unroll
    for (int lvl = 0; (C::TPR << lvl) < 32; ++lvl) {
        const int o = C::TPR << lvl;
        const int n = C::CPT >> lvl;
        const bool up = (lane & o) != 0;
        if (n >= 2) {
            const int hh = n / 2;
#pragma unroll
            for (int i = 0; i < hh; ++i) {
                const float send = up ? v[i] : v[hh + i];
                const float keep = up ? v[hh + i] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
            off += up ? hh : 0;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
            dup |= (unsigned)o;
        }
    }
    constexpr int NF = (C::CPT / C::RW) > 0 ? C::CPT / C::RW : 1;
    if ((lane & dup) == 0) {
#pragma unroll
        for (int i = 0; i < NF; ++i) atomicAdd(dst + gc0 + off + i, scale * v[i]);
    }
}

// The scalars of one token (slots of BwdCfg) from its norms, raw gate inputs and squared
// norms: gates (Eq. (53)) and the executed step with its intermediates, formed as the
// forward kernels' step control forms them (Def. 1, App. B.3), so the branch matches.
template <int D>
__device__ __forceinline__ void token_scalars(const ScanArgs &a, float *sc, float nk, float nq,
                                              float se, float sa, float kn2, float dd, int pix)
{
    using C = BwdCfg<D>;
    float eta, alpha, oma;
    gates(a, se, sa, eta, alpha, oma);
    const float rr = sqrtf(dd + a.eps * a.eps) + a.eps;
    const float einj = __fdividef(a.inj_factor * oma, rr);
    const float ebar = einj > 0.0f ? einj * (-expm1f(-__fdividef(eta, einj))) : 0.0f;
    float spec = __fdividef(a.spec_factor * 2.0f * alpha, fmaxf(kn2, a.kk_floor));
    if (spec > 0.0f) spec = __int_as_float(__float_as_int(spec) - 1);
    const bool sp = spec < ebar;
    const bool forced = a.gate_mode == VH_GATE_FORCED_EXEC;
    sc[C::S_NK] = nk;
    sc[C::S_NQ] = nq;
    sc[C::S_SE] = se + a.eta_bias;
    sc[3] = sa;
    sc[C::S_AL] = alpha;
    sc[C::S_OMA] = oma;
    sc[C::S_ETA] = eta;
    sc[C::S_ET] = forced ? a.forced_eta : (sp ? spec : ebar);
    sc[C::S_INJ] = einj;
    sc[C::S_BAR] = ebar;
    sc[C::S_SPEC] = spec;
    sc[C::S_R] = rr;
    sc[C::S_BR] = (!forced && sp) ? 1.0f : 0.0f;
    sc[C::S_KN2] = kn2;
    sc[C::S_DD] = dd;
    sc[C::S_PIX] = __int_as_float(pix);
}

template <int D, typename XT>
__global__ void __launch_bounds__(256, BwdCfg<D>::MINB) scan_bwd_kernel(const BwdArgs ba)
{
    using C = BwdCfg<D>;
    const ScanArgs &a = ba.s;
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    float *S = sm + C::OFF_S, *dS = sm + C::OFF_DS, *GT = sm + C::OFF_GT;
    float *X = sm + C::OFF_X, *P = sm + C::OFF_P, *K = sm + C::OFF_K, *DL = sm + C::OFF_DL;
    float *Q = sm + C::OFF_Q, *Z = sm + C::OFF_Z, *SC = sm + C::OFF_SC, *KG = sm + C::OFF_KG;
    float *DG = sm + C::OFF_DG, *Y = sm + C::OFF_Y, *UV = sm + C::OFF_UV;
    int *PIX = reinterpret_cast<int *>(sm + C::OFF_PIX);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int id = blockIdx.x;
    const int h = id % a.nh;
    id /= a.nh;
    const int r = a.dir_list[id % a.ndirs];
    const int b = id / a.ndirs;
    const int H = a.H, W = a.W, N = H * W, Cc = a.Cc;
    const size_t SZ = (size_t)C::R * D;
    const int Cr = route_chunk(r, a.chunk, H, W);
    const int nchunks = (N + Cr - 1) / Cr;
    const int ngs = (ba.lmax + C::GS - 1) / C::GS;    // stored gain slices per chunk
    float *ckpt = ba.ws + (size_t)blockIdx.x * ((size_t)ba.nck * SZ + (size_t)ngs * D * D +
                                                (size_t)ba.lmax * (C::TRS + C::GRS));
    float *gsc = ckpt + (size_t)ba.nck * SZ;          // [ngs][NT][CPT]: slices of G_{t-1}
    float *trl = gsc + (size_t)ngs * D * D;           // [lmax][TRS]: token records of the chunk
    float *grec = trl + (size_t)ba.lmax * C::TRS;     // [lmax][GRS]
    // token records of the whole scan, when the tensor-core forward wrote them
    const float *trg = a.rec ? a.rec + (size_t)blockIdx.x * a.rec_stride : nullptr;
    const XT *xb = static_cast<const XT *>(a.x) + (size_t)b * N * Cc + (size_t)h * D;
    const float *lam = a.dir_scale ? a.dir_scale + (size_t)r * Cc + (size_t)h * D : nullptr;
    const float *gob = ba.dout + (size_t)b * N * Cc + (size_t)h * D;
    float *dxb = ba.dx + (size_t)b * N * Cc + (size_t)h * D;
    const int grow = tid / C::TPR, gc0 = (tid % C::TPR) * C::CPT;

    const float *m0 = a.mem0 + ((size_t)r * a.nh + h) * SZ;
    for (int e = tid; e < C::R * D; e += C::NT) S[(e / D) * C::SS + (e % D)] = m0[e];
    float G[C::CPT];

    // ---- a tile of a chunk, forward.  gen_tile: gather, generation and the per-token
    // step into X, K, DL, Q, SC.  load_tile: K, DL and SC from the token records the
    // tensor-core forward wrote.  gain_tile: with `record` the token quantities go to the
    // chunk's records; then the shared gain over the tile's tokens, with `record` each
    // token's slice of G_{t-1} and G_{t-1} k saved.
    // this thread's CPT key entries of tile token j (columns gc0..)
    auto ld_key = [&](int j, float (&kv)[C::CPT]) {
        const float *kj = K + j * D + gc0;
        if constexpr (C::CPT % 4 == 0) {
#pragma unroll
            for (int c = 0; c < C::CPT; c += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(kj + c);
                kv[c] = f.x; kv[c + 1] = f.y; kv[c + 2] = f.z; kv[c + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int c = 0; c < C::CPT; ++c) kv[c] = kj[c];
        }
    };
    auto gather_x = [&](int c0, int t0, int Lt) {
        constexpr int EPV = 16 / (int)sizeof(XT);
        constexpr int VPT = D / EPV;
        for (int e = tid; e < Lt * VPT; e += C::NT) {
            const int j = e / VPT, v = e % VPT;
            const int pix = route_pixel(r, c0 + t0 + j, H, W);
            const uint4 raw = VH_IN(a.stats, ((size_t)b * N + pix) * Cc + (size_t)h * D + v * EPV, EPV, map_elems(a))
                                  ? __ldg(reinterpret_cast<const uint4 *>(xb + (size_t)pix * Cc + v * EPV))
                                  : make_uint4(0u, 0u, 0u, 0u);
            const XT *el = reinterpret_cast<const XT *>(&raw);
#pragma unroll
            for (int u = 0; u < EPV; ++u) X[j * D + v * EPV + u] = XElem<XT>::to_f(el[u]);
        }
    };
    auto gen_tile = [&](int c0, int t0, int Lt) {
        __syncthreads();  // earlier users of the tile buffers are done
        if (tid < Lt) PIX[tid] = route_pixel(r, c0 + t0 + tid, H, W);
        gather_x(c0, t0, Lt);
        __syncthreads();
        // generation from the boundary state, Eq. (15): rows 0..3d-1 (k, v, q), then the
        // eta and alpha rows (4d, 4d + 1)
        // (lane = output row, JB tokens per item: one state load serves JB tokens)
        {
            constexpr int NG = 3 * D + 2;
            constexpr int OB = (NG + 31) / 32;
            const int nJB = (Lt + C::JB - 1) / C::JB;
            for (int item = warp; item < OB * nJB; item += C::NW) {
                const int o = (item % OB) * 32 + lane;
                const int j0 = (item / OB) * C::JB;
                if (o < NG) {
                    const float *srow = S + (o < 3 * D ? o : o + D) * C::SS;
                    float acc[C::JB];
#pragma unroll
                    for (int jj = 0; jj < C::JB; ++jj) acc[jj] = 0.0f;
#pragma unroll 2
                    for (int i = 0; i < D; i += 4) {
                        const float4 sv = *reinterpret_cast<const float4 *>(srow + i);
#pragma unroll
                        for (int jj = 0; jj < C::JB; ++jj) {
                            const float4 xv = *reinterpret_cast<const float4 *>(X + (j0 + jj) * D + i);
                            acc[jj] = fmaf(sv.x, xv.x, acc[jj]);
                            acc[jj] = fmaf(sv.y, xv.y, acc[jj]);
                            acc[jj] = fmaf(sv.z, xv.z, acc[jj]);
                            acc[jj] = fmaf(sv.w, xv.w, acc[jj]);
                        }
                    }
#pragma unroll
                    for (int jj = 0; jj < C::JB; ++jj)
                        if (j0 + jj < Lt) P[(j0 + jj) * C::PS + o] = acc[jj];
                }
            }
        }
        __syncthreads();
        // per-token step, one warp per token
        for (int j = warp; j < Lt; j += C::NW) {
            const float *pr = P + j * C::PS;
            float kr[C::CPL], vv[C::CPL], qr[C::CPL];
            float kk = 0.0f, qq = 0.0f;
#pragma unroll
            for (int m = 0; m < C::CPL; ++m) {
                const int c = lane + 32 * m;
                const bool ok = c < D;
                kr[m] = ok ? pr[c] : 0.0f;
                vv[m] = ok ? pr[D + c] : 0.0f;
                qr[m] = ok ? pr[2 * D + c] : 0.0f;
                kk = fmaf(kr[m], kr[m], kk);
                qq = fmaf(qr[m], qr[m], qq);
            }
            kk = warp_sum(kk);
            qq = warp_sum(qq);
            const float nk = sqrtf(kk + a.knorm_eps), nq = sqrtf(qq + a.knorm_eps);
            float kn2 = 0.0f, dd = 0.0f;
#pragma unroll
            for (int m = 0; m < C::CPL; ++m) {
                kr[m] = kr[m] / nk;
                qr[m] = qr[m] / nq;
                vv[m] = kr[m] - vv[m];
                kn2 = fmaf(kr[m], kr[m], kn2);
                dd = fmaf(vv[m], vv[m], dd);
            }
            kn2 = warp_sum(kn2);
            dd = warp_sum(dd);
#pragma unroll
            for (int m = 0; m < C::CPL; ++m) {
                const int c = lane + 32 * m;
                if (c < D) {
                    K[j * D + c] = kr[m];
                    DL[j * D + c] = vv[m];
                    Q[j * D + c] = qr[m];
                }
            }
            if (lane == 0)
                token_scalars<D>(a, SC + j * C::NSC, nk, nq, pr[3 * D], pr[3 * D + 1], kn2, dd, PIX[j]);
        }
        __syncthreads();
    };
    auto load_tile = [&](int c0, int t0, int Lt) {
        __syncthreads();  // earlier users of the tile buffers are done
        const float *tr = trg + (size_t)(c0 + t0) * C::TRS;
        for (int e = tid; e < Lt * (D / 4); e += C::NT) {
            const int j = e / (D / 4), f = (e % (D / 4)) * 4;
            const float *tk = tr + (size_t)j * C::TRS;
            cp_async16(K + j * D + f, tk + f);
            cp_async16(DL + j * D + f, tk + 2 * D + f);
        }
        if (tid < Lt) {
            const float *ts = tr + (size_t)tid * C::TRS + 3 * D;
            token_scalars<D>(a, SC + tid * C::NSC, sqrtf(ts[TR_KK] + a.knorm_eps),
                             sqrtf(ts[TR_QQ] + a.knorm_eps), ts[TR_SE], ts[TR_SA], ts[TR_KN2],
                             ts[TR_DD], route_pixel(r, c0 + t0 + tid, H, W));
        }
        cp_async_wait_all();
        __syncthreads();
    };
    auto gain_tile = [&](int t0, int Lt, bool record) {
        if (record) {
            if (!trg) {
                for (int e = tid; e < Lt * (3 * D); e += C::NT) {
                    const int j = e / (3 * D), f = e % (3 * D);
                    const float v = f < D ? K[j * D + f] : (f < 2 * D ? Q[j * D + f - D] : DL[j * D + f - 2 * D]);
                    trl[(size_t)(t0 + j) * C::TRS + f] = v;
                }
            }
            for (int e = tid; e < Lt * C::NSC; e += C::NT)
                grec[(size_t)(t0 + e / C::NSC) * C::GRS + D + e % C::NSC] = SC[e];
        }
        // thread (grow, gc0) holds G[grow][gc0..]
        for (int j = 0; j < Lt; ++j) {
            float kj[C::CPT];
            ld_key(j, kj);
            float part = 0.0f;
#pragma unroll
            for (int c = 0; c < C::CPT; ++c) part = fmaf(G[c], kj[c], part);
#pragma unroll
            for (int o = C::TPR / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (record) {
                if ((j % C::GS) == 0) {  // a group's first slice of G_{t-1}
                    float *gd = gsc + ((size_t)(t0 + j) / C::GS * C::NT + tid) * C::CPT;
                    if constexpr (C::CPT % 4 == 0) {
#pragma unroll
                        for (int c = 0; c < C::CPT; c += 4)
                            *reinterpret_cast<float4 *>(gd + c) = make_float4(G[c], G[c + 1], G[c + 2], G[c + 3]);
                    } else {
#pragma unroll
                        for (int c = 0; c < C::CPT; ++c) gd[c] = G[c];
                    }
                }
                if (gc0 == 0) grec[(size_t)(t0 + j) * C::GRS + grow] = part;
            }
            const float et = SC[j * C::NSC + C::S_ET], al = SC[j * C::NSC + C::S_AL];
            const float s = et * (part + DL[j * D + grow]);
#pragma unroll
            for (int c = 0; c < C::CPT; ++c) G[c] = fmaf(-s, kj[c], al * G[c]);
        }
    };

    // Row transform M[o][:] <- sum_l M[o][l] GT[l][:] of the R rows of M (stride SS), in
    // place, one warp per row; for d <= 32 each lane keeps its column of GT in registers.
    auto rows_times = [&](float *M) {
        if constexpr (D <= 32) {
            float gcol[D];
#pragma unroll
            for (int l = 0; l < D; ++l) gcol[l] = lane < D ? GT[l * D + lane] : 0.0f;
            for (int o = warp; o < C::R; o += C::NW) {
                const float *mrow = M + o * C::SS;
                float acc = 0.0f;
#pragma unroll
                for (int l = 0; l < D; l += 4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(mrow + l);
                    acc = fmaf(m4.x, gcol[l], acc);
                    acc = fmaf(m4.y, gcol[l + 1], acc);
                    acc = fmaf(m4.z, gcol[l + 2], acc);
                    acc = fmaf(m4.w, gcol[l + 3], acc);
                }
                __syncwarp();
                if (lane < D) M[o * C::SS + lane] = acc;
                __syncwarp();
            }
        } else {
            for (int o = warp; o < C::R; o += C::NW) {
                const float *mrow = M + o * C::SS;
                float acc[C::CPL];
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) acc[m] = 0.0f;
#pragma unroll 8
                for (int l = 0; l < D; ++l) {
                    const float s = mrow[l];
#pragma unroll
                    for (int m = 0; m < C::CPL; ++m) acc[m] = fmaf(s, GT[l * D + lane + 32 * m], acc[m]);
                }
                __syncwarp();
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) M[o * C::SS + lane + 32 * m] = acc[m];
                __syncwarp();
            }
        }
    };

    // ---- pass 1: forward, checkpointing each chunk's boundary state (skipped when the
    // tensor-core forward has written them)
    for (int c = 0; c < (ba.have_ckpt ? 0 : nchunks); ++c) {
        const int c0 = c * Cr, L = min(Cr, N - c0);
        __syncthreads();
        float *ck = ckpt + (size_t)c * SZ;
        for (int e = tid; e < C::R * D; e += C::NT) ck[e] = S[(e / D) * C::SS + (e % D)];
        if (c == nchunks - 1) break;  // the last chunk's end state is not needed
#pragma unroll
        for (int q = 0; q < C::CPT; ++q) G[q] = (grow == gc0 + q) ? 1.0f : 0.0f;
        for (int t0 = 0; t0 < L; t0 += C::T) {
            gen_tile(c0, t0, min(C::T, L - t0));
            gain_tile(t0, min(C::T, L - t0), false);
        }
        // chunk end: S <- S_b G, row by row
        __syncthreads();
#pragma unroll
        for (int q = 0; q < C::CPT; ++q) GT[grow * D + gc0 + q] = G[q];
        __syncthreads();
        rows_times(S);  // GT holds G: S <- S G
    }

    // ---- pass 2: reverse
    __syncthreads();
    {
        const float *dmf = ba.dmem_final ? ba.dmem_final + (((size_t)b * 4 + r) * a.nh + h) * SZ : nullptr;
        for (int e = tid; e < C::R * D; e += C::NT) dS[(e / D) * C::SS + (e % D)] = dmf ? dmf[e] : 0.0f;
    }
    for (int c = nchunks - 1; c >= 0; --c) {
        const int c0 = c * Cr, L = min(Cr, N - c0);
        __syncthreads();
        {
            // the boundary state, every load issued before the stores
            const float4 *ck4 = reinterpret_cast<const float4 *>(ckpt + (size_t)c * SZ);
            constexpr int NS4 = (C::R * D / 4 + C::NT - 1) / C::NT;
            float4 v[NS4];
#pragma unroll
            for (int i = 0; i < NS4; ++i)
                if (tid + i * C::NT < C::R * D / 4) v[i] = ck4[tid + i * C::NT];
#pragma unroll
            for (int i = 0; i < NS4; ++i) {
                const int e = tid + i * C::NT;
                if (e < C::R * D / 4)
                    *reinterpret_cast<float4 *>(S + (e / (D / 4)) * C::SS + (e % (D / 4)) * 4) = v[i];
            }
        }
#pragma unroll
        for (int q = 0; q < C::CPT; ++q) G[q] = (grow == gc0 + q) ? 1.0f : 0.0f;
        // a. regenerate the chunk (or read its token records), recording
        for (int t0 = 0; t0 < L; t0 += C::T) {
            if (trg) load_tile(c0, t0, min(C::T, L - t0));
            else gen_tile(c0, t0, min(C::T, L - t0));
            gain_tile(t0, min(C::T, L - t0), true);
        }
        const float *tr = trg ? trg + (size_t)c0 * C::TRS : trl;  // this chunk's token records
        // b. chunk end: P_L = S_b^T dS (this thread's slice), then dS <- dS G_L^T
        __syncthreads();
#pragma unroll
        for (int q = 0; q < C::CPT; ++q) GT[(gc0 + q) * D + grow] = G[q];
        float Pg[C::CPT];
#pragma unroll
        for (int q = 0; q < C::CPT; ++q) Pg[q] = 0.0f;
        for (int o = 0; o < C::R; ++o) {
            const float sv = S[o * C::SS + grow];
            const float *dr = dS + o * C::SS + gc0;
            if constexpr (C::CPT % 4 == 0) {
#pragma unroll
                for (int q = 0; q < C::CPT; q += 4) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dr + q);
                    Pg[q] = fmaf(sv, d4.x, Pg[q]);
                    Pg[q + 1] = fmaf(sv, d4.y, Pg[q + 1]);
                    Pg[q + 2] = fmaf(sv, d4.z, Pg[q + 2]);
                    Pg[q + 3] = fmaf(sv, d4.w, Pg[q + 3]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < C::CPT; ++q) Pg[q] = fmaf(sv, dr[q], Pg[q]);
            }
        }
        __syncthreads();
        rows_times(dS);  // GT holds G^T: dS <- dS G^T
        // c-e. tiles, last first
        const int ntiles = (L + C::T - 1) / C::T;
        for (int ti = ntiles - 1; ti >= 0; --ti) {
            const int t0 = ti * C::T, Lt = min(C::T, L - t0);
            __syncthreads();
            // staging by asynchronous copies, all in flight together: the token records
            // (k, q, delta), G_{t-1} k into Z and the scalars from the gain records, x at the
            // tokens' pixels (fp32 straight into X; bf16 through the P buffer, which is free
            // until the per-token adjoints) and dout at the pixels into Y
            {
                constexpr int EPV = 16 / (int)sizeof(XT), VPT = D / EPV;
                unsigned char *xraw = sizeof(XT) == 4 ? reinterpret_cast<unsigned char *>(X)
                                                      : reinterpret_cast<unsigned char *>(P);
                for (int e = tid; e < Lt * (D / 4); e += C::NT) {
                    const int j = e / (D / 4), f = (e % (D / 4)) * 4;
                    const float *tk = tr + (size_t)(t0 + j) * C::TRS + f;
                    cp_async16(K + j * D + f, tk);
                    cp_async16(Q + j * D + f, tk + D);
                    cp_async16(DL + j * D + f, tk + 2 * D);
                    cp_async16(Z + j * D + f, grec + (size_t)(t0 + j) * C::GRS + f);
                }
                for (int e = tid; e < Lt * (C::NSC / 4); e += C::NT)
                    cp_async16(SC + 4 * e, grec + (size_t)(t0 + e / (C::NSC / 4)) * C::GRS + D + (e % (C::NSC / 4)) * 4);
                for (int e = tid; e < Lt * VPT; e += C::NT) {
                    const int pix = route_pixel(r, c0 + t0 + e / VPT, H, W);
                    if (VH_IN(a.stats, ((size_t)b * N + pix) * Cc + (size_t)h * D + (e % VPT) * EPV, EPV,
                              map_elems(a)))
                        cp_async16(xraw + (size_t)e * 16, xb + (size_t)pix * Cc + (e % VPT) * EPV);
                }
                for (int e = tid; e < Lt * D; e += C::NT) {
                    const int pix = route_pixel(r, c0 + t0 + e / D, H, W);
                    if (VH_IN(a.stats, ((size_t)b * N + pix) * Cc + (size_t)h * D + e % D, 1, map_elems(a)))
                        cp_async4(Y + e, gob + (size_t)pix * Cc + e % D);
                }
                cp_async_wait_all();
                __syncthreads();
                // z = G_{t-1} k + delta; the dk share of the gain starts at zero; x to fp32
                for (int e = tid; e < Lt * (D / 4); e += C::NT) {
                    float4 *z4 = reinterpret_cast<float4 *>(Z) + e;
                    const float4 d4 = reinterpret_cast<const float4 *>(DL)[e];
                    const float4 g4 = *z4;
                    *z4 = make_float4(g4.x + d4.x, g4.y + d4.y, g4.z + d4.z, g4.w + d4.w);
                    reinterpret_cast<float4 *>(KG)[e] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
                if (lam)  // dy = lambda_r dout
                    for (int e = tid; e < Lt * D; e += C::NT) Y[e] *= lam[e % D];
                if constexpr (sizeof(XT) != 4) {
                    for (int e = tid; e < Lt * VPT; e += C::NT) {
                        const uint4 raw = *reinterpret_cast<const uint4 *>(xraw + (size_t)e * 16);
                        const XT *el = reinterpret_cast<const XT *>(&raw);
                        float *xd = X + e * EPV;
#pragma unroll
                        for (int u = 0; u < EPV; ++u) xd[u] = XElem<XT>::to_f(el[u]);
                    }
                }
            }
            __syncthreads();
            // c. gain adjoint, last token first, by groups of GS tokens.  A group's first
            // slice of G_{t-1} is in the workspace (fetched one group ahead); the others
            // follow forward from it, G_t = alpha_t G_{t-1} - eta_t z_t k_t^T with the
            // recorded z_t, exactly as the recompute formed them.
            auto ld_slice = [&](int j, float (&g)[C::CPT]) {
                const float *gs = gsc + ((size_t)(t0 + j) / C::GS * C::NT + tid) * C::CPT;
                if constexpr (C::CPT % 4 == 0) {
#pragma unroll
                    for (int q = 0; q < C::CPT; q += 4) {
                        const float4 f = *reinterpret_cast<const float4 *>(gs + q);
                        g[q] = f.x; g[q + 1] = f.y; g[q + 2] = f.z; g[q + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < C::CPT; ++q) g[q] = gs[q];
                }
            };
            float nxt[C::CPT];
            const int ngrp = (Lt + C::GS - 1) / C::GS;
            ld_slice((ngrp - 1) * C::GS, nxt);
            for (int gi = ngrp - 1; gi >= 0; --gi) {
                const int m0 = gi * C::GS;
                float ring[C::GS][C::CPT];
#pragma unroll
                for (int q = 0; q < C::CPT; ++q) ring[0][q] = nxt[q];
                if (gi > 0) ld_slice(m0 - C::GS, nxt);
#pragma unroll
                for (int i = 1; i < C::GS; ++i) {
                    const int jp = min(m0 + i - 1, Lt - 1);  // past the tile's end: unused
                    float kp[C::CPT];
                    ld_key(jp, kp);
                    const float sp = SC[jp * C::NSC + C::S_ET] * Z[jp * D + grow];
                    const float ap = SC[jp * C::NSC + C::S_AL];
#pragma unroll
                    for (int q = 0; q < C::CPT; ++q) ring[i][q] = fmaf(-sp, kp[q], ap * ring[i - 1][q]);
                }
#pragma unroll
                for (int i = C::GS - 1; i >= 0; --i) {
                    const int j = m0 + i;
                    if (j >= Lt) continue;
                    float kj[C::CPT];
                    ld_key(j, kj);
                    // u = P_t k_t and this row's share of <P_t, G_{t-1}>, reduced together
                    float u = 0.0f, sa = 0.0f;
#pragma unroll
                    for (int q = 0; q < C::CPT; ++q) {
                        u = fmaf(Pg[q], kj[q], u);
                        sa = fmaf(Pg[q], ring[i][q], sa);
                    }
#pragma unroll
                    for (int o = C::TPR / 2; o > 0; o >>= 1) {
                        u += __shfl_xor_sync(0xffffffffu, u, o);
                        sa += __shfl_xor_sync(0xffffffffu, sa, o);
                    }
                    const float zr = Z[j * D + grow];
                    const float al = SC[j * C::NSC + C::S_AL], et = SC[j * C::NSC + C::S_ET];
                    float cp[C::CPT];
#pragma unroll
                    for (int q = 0; q < C::CPT; ++q) cp[q] = fmaf(ring[i][q], u, Pg[q] * zr);
                    if (gc0 == 0) {
                        DG[j * D + grow] = -et * u;
                        UV[j * D + grow] = u;
                        UV[(C::T + j) * D + grow] = sa;
                    }
#pragma unroll
                    for (int q = 0; q < C::CPT; ++q) Pg[q] = fmaf(-et * u, kj[q], al * Pg[q]);
                    col_sums_add<D>(cp, lane, gc0, KG + j * D, -et);
                }
            }
            __syncthreads();
            // d. per-token adjoints; a warp takes two tokens at a time (j and j + NW) so
            // that every load of the state serves both
            for (int j0 = warp; j0 < Lt; j0 += 2 * C::NW) {
                const bool two = j0 + C::NW < Lt;
                const int jt[2] = {j0, two ? j0 + C::NW : j0};
                // readout adjoint: dq = M^m_b^T dy
                float dq[2][C::CPL];
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) {
                    const int c = lane + 32 * m;
                    float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
                    if (c < D) {
#pragma unroll 4
                        for (int i = 0; i < D; i += 4) {
                            const float4 ya = *reinterpret_cast<const float4 *>(Y + jt[0] * D + i);
                            const float4 yb = *reinterpret_cast<const float4 *>(Y + jt[1] * D + i);
                            const float *sm0 = S + (3 * D + i) * C::SS + c;
                            const float s0 = sm0[0], s1 = sm0[C::SS], s2 = sm0[2 * C::SS], s3 = sm0[3 * C::SS];
                            a0 = fmaf(s0, ya.x, a0);
                            a1 = fmaf(s1, ya.y, a1);
                            a0 = fmaf(s2, ya.z, a0);
                            a1 = fmaf(s3, ya.w, a1);
                            b0 = fmaf(s0, yb.x, b0);
                            b1 = fmaf(s1, yb.y, b1);
                            b0 = fmaf(s2, yb.z, b0);
                            b1 = fmaf(s3, yb.w, b1);
                        }
                    }
                    dq[0][m] = a0 + a1;
                    dq[1][m] = b0 + b1;
                }
                int pixt[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int j = jt[u];
                    const float *sc = SC + j * C::NSC;
                    pixt[u] = __float_as_int(sc[C::S_PIX]);
                    float kk[C::CPL], qv[C::CPL], dl[C::CPL];
#pragma unroll
                    for (int m = 0; m < C::CPL; ++m) {
                        const int c = lane + 32 * m;
                        const bool ok = c < D;
                        kk[m] = ok ? K[j * D + c] : 0.0f;
                        qv[m] = ok ? Q[j * D + c] : 0.0f;
                        dl[m] = ok ? DL[j * D + c] : 0.0f;
                    }
                    // the gain's step and retention adjoints: deta_t = -z_t . u_t,
                    // dalpha_t = <P_t, G_{t-1}> (row shares summed)
                    float det = 0.0f, dag = 0.0f;
#pragma unroll
                    for (int m = 0; m < C::CPL; ++m) {
                        const int c = lane + 32 * m;
                        if (c < D) {
                            det = fmaf(-Z[j * D + c], UV[j * D + c], det);
                            dag += UV[(C::T + j) * D + c];
                        }
                    }
                    det = warp_sum(det);
                    dag = warp_sum(dag);
                    // executed step and gates
                    float deta = 0.0f, dalpha = dag, dkn2 = 0.0f, ddd = 0.0f;
                    if (a.gate_mode != VH_GATE_FORCED_EXEC) {
                        if (sc[C::S_BR] != 0.0f) {  // spectral limit executed
                            const float kn2 = sc[C::S_KN2];
                            const float fl = fmaxf(kn2, a.kk_floor);
                            dalpha += det * a.spec_factor * 2.0f / fl;
                            if (kn2 > a.kk_floor) dkn2 -= det * sc[C::S_SPEC] / kn2;
                        } else if (sc[C::S_INJ] > 0.0f) {  // soft injection cap
                            const float einj = sc[C::S_INJ], eta = sc[C::S_ETA], rr = sc[C::S_R];
                            const float x = eta / einj;
                            const float ex = expf(-x);
                            deta += det * ex;
                            const float dinj = det * (-expm1f(-x) - x * ex);
                            dalpha -= dinj * a.inj_factor / rr;  // eta_inj falls with alpha
                            const float dr = -dinj * einj / rr;
                            ddd += dr / (2.0f * sqrtf(sc[C::S_DD] + a.eps * a.eps));
                        }
                    }
                    float dse = 0.0f, dsa = 0.0f;
                    if (a.gate_mode == VH_GATE_GENERATED) {
                        dse = deta * a.gamma_eta / (1.0f + expf(-sc[C::S_SE]));  // softplus' = sigmoid
                        dsa = dalpha * sc[C::S_AL] * sc[C::S_OMA];
                    }
                    // delta = k - v, the two normalisations
                    float dk[C::CPL], ddl[C::CPL];
                    float kdk = 0.0f, qdq = 0.0f;
#pragma unroll
                    for (int m = 0; m < C::CPL; ++m) {
                        const int c = lane + 32 * m;
                        const bool ok = c < D;
                        ddl[m] = ok ? fmaf(2.0f * ddd, dl[m], DG[j * D + c]) : 0.0f;
                        dk[m] = ok ? fmaf(2.0f * dkn2, kk[m], KG[j * D + c]) + ddl[m] : 0.0f;
                        kdk = fmaf(kk[m], dk[m], kdk);
                        qdq = fmaf(qv[m], dq[u][m], qdq);
                    }
                    kdk = warp_sum(kdk);
                    qdq = warp_sum(qdq);
                    const float nk = sc[C::S_NK], nq = sc[C::S_NQ];
                    float *gv = P + j * C::PS;  // generation adjoints dk_raw | dv | dq_raw | dse dsa
                    if (u == 0 || two) {
#pragma unroll
                        for (int m = 0; m < C::CPL; ++m) {
                            const int c = lane + 32 * m;
                            if (c < D) {
                                gv[c] = (dk[m] - kk[m] * kdk) / nk;
                                gv[D + c] = -ddl[m];
                                gv[2 * D + c] = (dq[u][m] - qv[m] * qdq) / nq;
                            }
                        }
                        if (lane == 0) {
                            gv[3 * D] = dse;
                            gv[3 * D + 1] = dsa;
                        }
                    }
                }
                __syncwarp();
                // dx_t = M^k^T dk_raw + M^v^T dv + M^q^T dq_raw + m^eta dse + m^alpha dsa
                const float *ga = P + jt[0] * C::PS, *gb = P + jt[1] * C::PS;
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) {
                    const int c = lane + 32 * m;
                    if (c < D) {
                        const float se = S[(4 * D) * C::SS + c], sl = S[(4 * D + 1) * C::SS + c];
                        float a0 = fmaf(se, ga[3 * D], sl * ga[3 * D + 1]), a1 = 0.0f, a2 = 0.0f;
                        float b0 = fmaf(se, gb[3 * D], sl * gb[3 * D + 1]), b1 = 0.0f, b2 = 0.0f;
#pragma unroll 2
                        for (int i = 0; i < D; i += 4) {
                            const float4 ka = *reinterpret_cast<const float4 *>(ga + i);
                            const float4 va = *reinterpret_cast<const float4 *>(ga + D + i);
                            const float4 qa = *reinterpret_cast<const float4 *>(ga + 2 * D + i);
                            const float4 kb = *reinterpret_cast<const float4 *>(gb + i);
                            const float4 vb = *reinterpret_cast<const float4 *>(gb + D + i);
                            const float4 qb = *reinterpret_cast<const float4 *>(gb + 2 * D + i);
                            const float kaa[4] = {ka.x, ka.y, ka.z, ka.w}, vaa[4] = {va.x, va.y, va.z, va.w};
                            const float qaa[4] = {qa.x, qa.y, qa.z, qa.w}, kba[4] = {kb.x, kb.y, kb.z, kb.w};
                            const float vba[4] = {vb.x, vb.y, vb.z, vb.w}, qba[4] = {qb.x, qb.y, qb.z, qb.w};
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const float sk = S[(i + w) * C::SS + c];
                                const float sv = S[(D + i + w) * C::SS + c];
                                const float sq = S[(2 * D + i + w) * C::SS + c];
                                a0 = fmaf(sk, kaa[w], a0);
                                a1 = fmaf(sv, vaa[w], a1);
                                a2 = fmaf(sq, qaa[w], a2);
                                b0 = fmaf(sk, kba[w], b0);
                                b1 = fmaf(sv, vba[w], b1);
                                b2 = fmaf(sq, qba[w], b2);
                            }
                        }
                        if (VH_IN(a.stats, ((size_t)b * N + pixt[0]) * Cc + (size_t)h * D + c, 1, map_elems(a)))
                            atomicAdd(dxb + (size_t)pixt[0] * Cc + c, (a0 + a1) + a2);
                        if (two &&
                            VH_IN(a.stats, ((size_t)b * N + pixt[1]) * Cc + (size_t)h * D + c, 1, map_elems(a)))
                            atomicAdd(dxb + (size_t)pixt[1] * Cc + c, (b0 + b1) + b2);
                    }
                }
                __syncwarp();
            }
            __syncthreads();
            // e. generation and readout adjoints into dL/dS_b, four columns per item
            for (int e = tid; e < C::R * (D / 4); e += C::NT) {
                const int o = e / (D / 4), j4 = (e % (D / 4)) * 4;
                float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
                const bool rd = o >= 3 * D && o < 4 * D;  // content memory: dy q^T
                const float *vs = rd ? Y + (o - 3 * D) : P + (o < 3 * D ? o : o - D);
                const int vstride = rd ? D : C::PS;
                const float *us = (rd ? Q : X) + j4;
                for (int t = 0; t < Lt; ++t) {
                    const float g = vs[t * vstride];
                    const float4 u = *reinterpret_cast<const float4 *>(us + t * D);
                    a0 = fmaf(g, u.x, a0);
                    a1 = fmaf(g, u.y, a1);
                    a2 = fmaf(g, u.z, a2);
                    a3 = fmaf(g, u.w, a3);
                }
                float *dd = dS + o * C::SS + j4;
                dd[0] += a0;
                dd[1] += a1;
                dd[2] += a2;
                dd[3] += a3;
            }
        }
    }
    __syncthreads();
    float *dm = ba.dmem0 + ((size_t)r * a.nh + h) * SZ;
    if (VH_IN(a.stats, ((size_t)r * a.nh + h) * SZ, SZ, (size_t)4 * a.nh * SZ))
        for (int e = tid; e < C::R * D; e += C::NT) atomicAdd(dm + e, dS[(e / D) * C::SS + (e % D)]);
}

template <int D, typename XT>
static cudaError_t launch_bwd_t(const BwdArgs &ba, cudaStream_t st)
{
    using C = BwdCfg<D>;
    auto kern = scan_bwd_kernel<D, XT>;
    static int attr_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const unsigned grid = (unsigned)(ba.s.B * ba.s.ndirs * ba.s.nh);
    kern<<<grid, C::NT, C::BYTES, st>>>(ba);
    return cudaGetLastError();
}

// Floats of workspace one CTA (scan) needs: boundary states, gain slices and records.
size_t bwd_floats_per_scan(int d, int nck, int lmax)
{
    const size_t sz = (size_t)(4 * d + 2) * d;
    return (size_t)nck * sz + (size_t)(lmax + kGainGroup - 1) / kGainGroup * d * d +
           (size_t)lmax * (token_rec_floats(d) + d + 16);
}

cudaError_t launch_scan_bwd(const BwdArgs &ba, int d, bool bf16, cudaStream_t st)
{
    switch (d) {
    case 16: return bf16 ? launch_bwd_t<16, __nv_bfloat16>(ba, st) : launch_bwd_t<16, float>(ba, st);
    case 32: return bf16 ? launch_bwd_t<32, __nv_bfloat16>(ba, st) : launch_bwd_t<32, float>(ba, st);
    case 64: return bf16 ? launch_bwd_t<64, __nv_bfloat16>(ba, st) : launch_bwd_t<64, float>(ba, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace vh
