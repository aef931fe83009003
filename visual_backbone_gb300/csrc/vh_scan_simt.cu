// vh_scan_simt.cu -- fp32 CUDA-core kernel of the four-direction VisionHOPE
// memory scan.
//
// One CTA owns one scan (image b, route r, head h) for its whole length and
// keeps the six memories of that scan in shared memory.  Per chunk
// ("VisionHOPE", Sec. 2.1.3 Eqs. (15)-(16)) it
//   1. gathers the chunk's tokens along the route (Eq. (24)),
//   2. generates k_raw, v, q_raw, s^eta, s^alpha from the boundary state,
//   3. normalises k and q (App. C.1, App. B.5) and applies the step-size
//      control of Def. 1 per token (Eqs. (19)-(20), App. B.3 safeguards),
//   4. reads out y_t = M^m_b q_t and adds lambda_r * y_t at the token's
//      pixel (Eq. (26)),
//   5. advances the shared gain G_t = G_{t-1} A_t + B_t = alpha_t G_{t-1}
//      - eta_t (G_{t-1} k_t + delta_t) k_t^T (App. B.4, Prop. 2, Eq. (46)),
//      whose rows evolve independently,
//   6. at the chunk end replaces every memory by M_b G (Eq. (46)).
// Long chunks are processed in token tiles; the gain carries across tiles.
// All arithmetic is fp32 on CUDA cores; this kernel is the general path (any
// head_dim in {16,32,64}, any chunk length) and the A/B reference for the
// tensor-core kernel.  At d = 64, where it is the only kernel, the phases are
// shaped for its 16-token tile: register-tiled generation and chunk-end update
// over 16-byte state rows, every warp in the readout, half a warp per token in
// the step control.
#include "vh_common.cuh"

namespace vh {

// Packed fp32 pairs for fma.rn.f32x2: lane 0 in the low word.
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// d = a * b + d on both lanes, each an fp32 fma rounded to nearest
__device__ __forceinline__ void fma_f32x2(unsigned long long &d, unsigned long long a, unsigned long long b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

template <int D>
struct SimtCfg {
    static constexpr int NT = 256;
    static constexpr int NW = NT / 32;
    static constexpr int R = 4 * D + 2;    // rows of the state: k, v, q, m (d each), eta, alpha
    static constexpr int RG = 3 * D + 2;   // rows used by the generation: k, v, q, eta, alpha
    // padded row stride of the state: d + 1 keeps column walks over lane-distinct rows
    // conflict-free; at d = 64 the rows are 16-byte aligned instead (d + 4), so every phase
    // reads along a row with 16-byte vectors
    static constexpr int SS = (D == 64) ? D + 4 : D + 1;
    static constexpr int T = (D == 64) ? 16 : 64;  // token tile (d = 64: two CTAs per SM)
    static constexpr int PS = RG + 1;      // row stride of the generation outputs
    static constexpr int TPR = NT / D;     // threads per gain row
    static constexpr int CPT = D / TPR;    // gain columns per thread
    static constexpr int JB = 8;           // tokens per register block
    static constexpr int CPL = (D + 31) / 32;  // vector components per lane
    static constexpr int OFF_S = 0;
    static constexpr int OFF_X = OFF_S + R * SS;
    static constexpr int OFF_P = OFF_X + T * D;
    static constexpr int OFF_K = OFF_P + T * PS;
    static constexpr int OFF_DL = OFF_K + T * D;
    static constexpr int OFF_Q = OFF_DL + T * D;
    static constexpr int OFF_SC = OFF_Q + T * D;
    static constexpr int OFF_PIX = OFF_SC + 2 * T;
    static constexpr int FLOATS = OFF_PIX + T;
    // the chunk-end copy of G starts at the first 16-byte boundary of the generation buffer
    // and may run on into the key buffer (d = 64), never into the delta buffer
    static constexpr int GS_PAD = (4 - OFF_P % 4) % 4;
    static_assert(OFF_P + GS_PAD + D * D <= OFF_DL, "chunk-end G copy");
    static_assert(D != 64 || (SS % 4 == 0 && OFF_X % 4 == 0 && OFF_P % 4 == 0 && OFF_Q % 4 == 0),
                  "16-byte rows at d = 64");
    static constexpr size_t BYTES = (size_t)FLOATS * 4;
    static_assert(T % JB == 0, "tile must hold whole register blocks");
    static_assert(D * D <= T * PS + T * D && OFF_K == OFF_P + T * PS,
                  "gain must fit in the generation and key buffers it reuses");
    static_assert(TPR * CPT == D && TPR <= 32, "gain thread map");
};

template <int D, typename XT>
__device__ __forceinline__ void scan_simt_body(const ScanArgs &a)
{
    using C = SimtCfg<D>;
    extern __shared__ float4 smem_f4[];
    float *sm = reinterpret_cast<float *>(smem_f4);
    float *S = sm + C::OFF_S;
    float *X = sm + C::OFF_X;
    float *P = sm + C::OFF_P;
    float *K = sm + C::OFF_K;
    float *DL = sm + C::OFF_DL;
    float *Q = sm + C::OFF_Q;
    float *SC = sm + C::OFF_SC;
    int *PIX = reinterpret_cast<int *>(sm + C::OFF_PIX);
    __shared__ unsigned long long st_cnt[3];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int id = blockIdx.x;
    const int h = id % a.nh;
    id /= a.nh;
    const int r = a.dir_list[id % a.ndirs];
    const int b = id / a.ndirs;
    const int H = a.H, W = a.W, N = H * W, Cc = a.Cc;
    const size_t SZ = (size_t)C::R * D;

    if (tid < 3) st_cnt[tid] = 0;
    // checked indices (VH_DEBUG_BOUNDS builds; `true` otherwise): this scan's slices of
    // memories0 and memories_out; every pixel index of the gather, the queries and the adds
    const size_t mem_base = ((size_t)r * a.nh + h) * SZ;
    const float *m0 = a.mem0 + (VH_IN(a.stats, mem_base, SZ, (size_t)4 * a.nh * SZ) ? mem_base : 0);
    for (int e = tid; e < C::R * D; e += C::NT) S[(e / D) * C::SS + (e % D)] = m0[e];

    const float dgd = (a.control_flags & VH_CTRL_NO_DGD) ? 0.0f : 1.0f;
    const bool intra = (a.control_flags & VH_CTRL_INTRA_READ) != 0;
    const int grow = tid / C::TPR;
    const int gc0 = (tid % C::TPR) * C::CPT;
    // column of this thread's c-th gain entry: a contiguous slice, or at d = 64 four
    // 4-column groups 4 TPR apart, so a row's lanes read their 16-byte key pieces from
    // distinct banks
    auto gcol = [&](int c) {
        return C::CPT >= 8 ? 4 * (tid % C::TPR) + 4 * C::TPR * (c >> 2) + (c & 3) : gc0 + c;
    };
    float G[C::CPT];

    const int Cr = route_chunk(r, a.chunk, H, W);
    const XT *xb = static_cast<const XT *>(a.x) + (size_t)b * N * Cc + (size_t)h * D;
    float *ob = a.out + (size_t)b * N * Cc + (size_t)h * D;
    const float *lam = a.dir_scale ? a.dir_scale + (size_t)r * Cc + (size_t)h * D : nullptr;
    unsigned n_spec = 0, n_inj = 0, n_nf = 0;

    for (int c0 = 0; c0 < N; c0 += Cr) {
        const int L = min(Cr, N - c0);
#pragma unroll
        for (int c = 0; c < C::CPT; ++c) G[c] = (grow == gcol(c)) ? 1.0f : 0.0f;

        for (int t0 = 0; t0 < L; t0 += C::T) {
            const int Lt = min(C::T, L - t0);
            __syncthreads();  // previous tile / chunk-end update finished with X, P, K, S
            // 1. gather the tile along the route, 16-byte vectors
            constexpr int EPV = 16 / (int)sizeof(XT);
            constexpr int VPT = D / EPV;
            if (tid < Lt) PIX[tid] = route_pixel(r, c0 + t0 + tid, H, W);
            for (int e = tid; e < Lt * VPT; e += C::NT) {
                const int j = e / VPT, v = e % VPT;
                const int pix = route_pixel(r, c0 + t0 + j, H, W);
                const bool in = VH_IN(a.stats, ((size_t)b * N + pix) * Cc + (size_t)h * D + v * EPV, EPV,
                                      map_elems(a));
                const uint4 raw = in ? __ldg(reinterpret_cast<const uint4 *>(xb + (size_t)pix * Cc + v * EPV))
                                     : make_uint4(0u, 0u, 0u, 0u);
                const XT *el = reinterpret_cast<const XT *>(&raw);
#pragma unroll
                for (int u = 0; u < EPV; ++u) X[j * D + v * EPV + u] = XElem<XT>::to_f(el[u]);
            }
            __syncthreads();

            // 2. generation from the boundary state: P[j][o] = sum_i S[o][i] x_j[i]
            if constexpr (D == 64) {
                // register tiles of 4 tokens x 4 outputs: thread (tg, og) takes tokens
                // 4 tg..4 tg+3 and outputs og + 49 k (k, v, q rows and the two gate rows),
                // so one 16-byte load of x serves four outputs and one of the state four
                // tokens; consecutive og read rows 16 bytes apart in the bank space
                constexpr int OG = (C::RG + 3) / 4;  // 49 output groups
                static_assert(4 * 4 == C::T && 4 * OG >= C::RG && 4 * OG <= C::NT, "tiles");
                if (tid < 4 * OG) {
                    const int tg = tid / OG, og = tid % OG;
                    int srow[4];  // state row offsets
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int o = min(og + OG * k, C::RG - 1);  // a padding output reads a real row
                        srow[k] = (o < 3 * D ? o : o + D) * C::SS;
                    }
                    float acc[4][4];
#pragma unroll
                    for (int t = 0; t < 4; ++t)
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[t][k] = 0.0f;
#pragma unroll 1
                    for (int i = 0; i < D; i += 4) {
                        float4 sv[4], xv[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) sv[k] = *reinterpret_cast<const float4 *>(S + srow[k] + i);
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            xv[t] = *reinterpret_cast<const float4 *>(X + (4 * tg + t) * D + i);
#pragma unroll
                        for (int t = 0; t < 4; ++t)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                acc[t][k] = fmaf(sv[k].w, xv[t].w,
                                                 fmaf(sv[k].z, xv[t].z,
                                                      fmaf(sv[k].y, xv[t].y, fmaf(sv[k].x, xv[t].x, acc[t][k]))));
                    }
#pragma unroll
                    for (int t = 0; t < 4; ++t)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int o = og + OG * k, j = 4 * tg + t;
                            if (o < C::RG && j < Lt) P[j * C::PS + o] = acc[t][k];
                        }
                }
            } else {
                constexpr int OB = (C::RG + 31) / 32;
                const int nJB = (Lt + C::JB - 1) / C::JB;
                for (int item = warp; item < OB * nJB; item += C::NW) {
                    const int o = (item % OB) * 32 + lane;
                    const int j0 = (item / OB) * C::JB;
                    if (o < C::RG) {
                        float acc[C::JB];
#pragma unroll
                        for (int jj = 0; jj < C::JB; ++jj) acc[jj] = 0.0f;
                        // outputs 0..3d-1 are k, v, q (state rows 0..3d-1); outputs 3d, 3d+1
                        // are s^eta, s^alpha (state rows 4d, 4d+1, after the content memory)
                        const float *srow = S + (o < 3 * D ? o : o + D) * C::SS;
#pragma unroll 8
                        for (int i = 0; i < D; ++i) {
                            const float s = srow[i];
#pragma unroll
                            for (int jj = 0; jj < C::JB; ++jj)
                                acc[jj] = fmaf(s, X[(j0 + jj) * D + i], acc[jj]);
                        }
#pragma unroll
                        for (int jj = 0; jj < C::JB; ++jj)
                            if (j0 + jj < Lt) P[(j0 + jj) * C::PS + o] = acc[jj];
                    }
                }
            }
            __syncthreads();

            // 3. per-token normalisation and step control, one warp per token (half a warp
            // at d = 64, so the 16-token tile takes one pass)
            constexpr int LPT = (D == 64) ? 16 : 32;  // lanes per token
            constexpr int TPW = 32 / LPT;             // tokens per warp and pass
            const int sub = lane / LPT, sl = lane % LPT;
            const unsigned smask = (LPT == 32) ? 0xffffffffu : (0xffffu << (16 * sub));
            auto tsum = [&](float v) {
                if constexpr (LPT == 32) {
                    return warp_sum(v);
                } else {
#pragma unroll
                    for (int o = LPT / 2; o > 0; o >>= 1) v += __shfl_xor_sync(smask, v, o);
                    return v;
                }
            };
            constexpr int CPT3 = (D + LPT - 1) / LPT;  // components per lane
            for (int j = warp * TPW + sub; j < Lt; j += C::NW * TPW) {
                const float *pr = P + j * C::PS;
                float kr[CPT3], vv[CPT3], qr[CPT3];
                float kk = 0.0f, qq = 0.0f;
                // VisionHOPE-exact readout: the query of the token's pixel, already
                // normalised, from the outer projection's planes
                const size_t qplane = (size_t)a.B * N * Cc;
                const size_t qo = (a.qhat && VH_IN(a.stats, ((size_t)b * N + PIX[j]) * Cc + (size_t)h * D, D,
                                                   qplane))
                                      ? ((size_t)b * N + PIX[j]) * Cc + (size_t)h * D
                                      : 0;
#pragma unroll
                for (int m = 0; m < CPT3; ++m) {
                    const int c = sl + LPT * m;
                    const bool ok = c < D;
                    kr[m] = ok ? pr[c] : 0.0f;
                    vv[m] = ok ? pr[D + c] : 0.0f;
                    qr[m] = ok ? (a.qhat ? qhat_at(a.qhat, qplane, qo + c) : pr[2 * D + c]) : 0.0f;
                    kk = fmaf(kr[m], kr[m], kk);
                    qq = fmaf(qr[m], qr[m], qq);
                }
                kk = tsum(kk);
                qq = tsum(qq);
                // stabilised norms as correctly rounded reciprocal square roots (one
                // multiply per component instead of a division)
                const float rk = __frsqrt_rn(kk + a.knorm_eps);
                const float rq = a.qhat ? 1.0f : __frsqrt_rn(qq + a.knorm_eps);
                float kn2 = 0.0f, dd = 0.0f;
#pragma unroll
                for (int m = 0; m < CPT3; ++m) {
                    kr[m] *= rk;
                    qr[m] *= rq;
                    vv[m] = kr[m] - vv[m];  // delta = k - v
                    kn2 = fmaf(kr[m], kr[m], kn2);
                    dd = fmaf(vv[m], vv[m], dd);
                }
                kn2 = tsum(kn2);
                dd = tsum(dd);
                float eta, alpha, oma;
                gates(a, pr[3 * D], pr[3 * D + 1], eta, alpha, oma);
                float eta_t;
                if (a.gate_mode == VH_GATE_FORCED_EXEC) {
                    eta_t = a.forced_eta;
                } else {
                    const StepOut so = step_control(a, eta, alpha, oma, kn2, dd);
                    eta_t = so.eta_tilde;
                    n_spec += (sl == 0 && so.spec_active);
                    n_inj += (sl == 0 && so.inj_ratio_gt1);
                }
#pragma unroll
                for (int m = 0; m < CPT3; ++m) {
                    const int c = sl + LPT * m;
                    if (c < D) {
                        K[j * D + c] = kr[m];
                        DL[j * D + c] = vv[m];
                        Q[j * D + c] = qr[m];
                    }
                }
                if (sl == 0) {
                    SC[2 * j] = alpha;
                    SC[2 * j + 1] = eta_t;
                }
            }
            __syncthreads();

            // 4. readout y_j = M^m_b q_j and the fused restore/sum of Eq. (26); with the
            // intra-chunk readout (ablation) the query is replaced by u_j = G_{j-1} q_j,
            // formed in the gain loop, and the readout follows it
            auto readout = [&](const float *Qv) {
                if constexpr (D == 64) {
                    // every warp: thread = output channel i, tokens tg, tg + TG, ...
                    constexpr int TG = C::NT / D, JT = C::T / TG;
                    const int i = tid % D, tg = tid / D;
                    float acc[JT];
#pragma unroll
                    for (int jj = 0; jj < JT; ++jj) acc[jj] = 0.0f;
                    const float *mrow = S + (3 * D + i) * C::SS;
#pragma unroll 2
                    for (int l = 0; l < D; l += 4) {
                        const float4 mv = *reinterpret_cast<const float4 *>(mrow + l);
#pragma unroll
                        for (int jj = 0; jj < JT; ++jj) {
                            const float4 qv = *reinterpret_cast<const float4 *>(Qv + (tg + TG * jj) * D + l);
                            acc[jj] = fmaf(mv.w, qv.w, fmaf(mv.z, qv.z, fmaf(mv.y, qv.y, fmaf(mv.x, qv.x, acc[jj]))));
                        }
                    }
                    const float lm = lam ? lam[i] : 1.0f;
#pragma unroll
                    for (int jj = 0; jj < JT; ++jj) {
                        const int j = tg + TG * jj;
                        if (j < Lt && VH_IN(a.stats, ((size_t)b * N + PIX[j]) * Cc + (size_t)h * D + i, 1,
                                            map_elems(a))) {
                            n_nf += !isfinite(acc[jj]);
                            atomicAdd(ob + (size_t)PIX[j] * Cc + i, lm * acc[jj]);
                        }
                    }
                } else {
                    const int nJB = (Lt + C::JB - 1) / C::JB;
                    for (int jb = warp; jb < nJB; jb += C::NW) {
                        const int j0 = jb * C::JB;
#pragma unroll
                        for (int m = 0; m < C::CPL; ++m) {
                            const int i = lane + 32 * m;
                            if (i < D) {
                                float acc[C::JB];
#pragma unroll
                                for (int jj = 0; jj < C::JB; ++jj) acc[jj] = 0.0f;
                                const float *mrow = S + (3 * D + i) * C::SS;
#pragma unroll 8
                                for (int l = 0; l < D; ++l) {
                                    const float mv = mrow[l];
#pragma unroll
                                    for (int jj = 0; jj < C::JB; ++jj)
                                        acc[jj] = fmaf(mv, Qv[(j0 + jj) * D + l], acc[jj]);
                                }
                                const float lm = lam ? lam[i] : 1.0f;
#pragma unroll
                                for (int jj = 0; jj < C::JB; ++jj) {
                                    if (j0 + jj < Lt &&
                                        VH_IN(a.stats, ((size_t)b * N + PIX[j0 + jj]) * Cc + (size_t)h * D + i, 1,
                                              map_elems(a))) {
                                        n_nf += !isfinite(acc[jj]);
                                        atomicAdd(ob + (size_t)PIX[j0 + jj] * Cc + i, lm * acc[jj]);
                                    }
                                }
                            }
                        }
                    }
                }
            };
            if (!intra) readout(Q);

            // 5. shared gain over the tile's tokens (rows are independent); without the
            // DGD correction (ablation) the G k term drops: G <- alpha G - eta delta k^T.
            // The intra-chunk readout's u_j = G_{j-1} q_j goes to P (free after step 3).
            float *U = P;
            // d = 64 (and no intra-chunk readout): the next token's key slice, delta entry
            // and scalars are loaded while the current token is applied
            const bool prefetch_loop = C::CPT >= 8 && !intra;
            if constexpr (C::CPT >= 8) {
                if (prefetch_loop) {
                    float kc[C::CPT], kn[C::CPT];
                    auto ldk = [&](int j, float (&kv)[C::CPT]) {
#pragma unroll
                        for (int c = 0; c < C::CPT; c += 4) {
                            const float4 f = *reinterpret_cast<const float4 *>(K + j * D + gcol(c));
                            kv[c] = f.x; kv[c + 1] = f.y; kv[c + 2] = f.z; kv[c + 3] = f.w;
                        }
                    };
                    ldk(0, kc);
                    float dlc = DL[grow];
                    float2 scc = *reinterpret_cast<const float2 *>(SC);
                    for (int j = 0; j < Lt; ++j) {
                        const int jn = min(j + 1, Lt - 1);
                        ldk(jn, kn);
                        const float dln = DL[jn * D + grow];
                        const float2 scn = *reinterpret_cast<const float2 *>(SC + 2 * jn);
                        float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int c = 0; c < C::CPT; ++c) p4[c & 3] = fmaf(G[c], kc[c], p4[c & 3]);
                        float part = (p4[0] + p4[1]) + (p4[2] + p4[3]);
#pragma unroll
                        for (int o = C::TPR / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                        const float sg = scc.y * (part * dgd + dlc);
#pragma unroll
                        for (int c = 0; c < C::CPT; ++c) G[c] = fmaf(-sg, kc[c], scc.x * G[c]);
#pragma unroll
                        for (int c = 0; c < C::CPT; ++c) kc[c] = kn[c];
                        dlc = dln;
                        scc = scn;
                    }
                }
            }
            for (int j = 0; j < Lt && !prefetch_loop; ++j) {
                const float *kj = K + j * D;
                float part = 0.0f;
                if constexpr (C::CPT >= 8) {  // four partial sums: a short dependent chain
                    float p4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int c = 0; c < C::CPT; ++c) p4[c & 3] = fmaf(G[c], kj[gcol(c)], p4[c & 3]);
                    part = (p4[0] + p4[1]) + (p4[2] + p4[3]);
                } else {
#pragma unroll
                    for (int c = 0; c < C::CPT; ++c) part = fmaf(G[c], kj[gcol(c)], part);
                }
#pragma unroll
                for (int o = C::TPR / 2; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if (intra) {
                    const float *qj = Q + j * D;
                    float u = 0.0f;
#pragma unroll
                    for (int c = 0; c < C::CPT; ++c) u = fmaf(G[c], qj[gcol(c)], u);
#pragma unroll
                    for (int o = C::TPR / 2; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
                    if (gc0 == 0) U[j * D + grow] = u;
                }
                const float s = SC[2 * j + 1] * (part * dgd + DL[j * D + grow]);
                const float al = SC[2 * j];
#pragma unroll
                for (int c = 0; c < C::CPT; ++c) G[c] = fmaf(-s, kj[gcol(c)], al * G[c]);
            }
            if (intra) {
                __syncthreads();  // U complete
                readout(U);
                __syncthreads();  // U read before P is reused
            }
        }

        // 6. chunk end: every memory becomes M_b G (G in the generation buffer and, for
        // d = 64, the key buffer after it, which the gain loop reads until its last token)
        if constexpr (D * D > C::T * C::PS) __syncthreads();
        float *Gs = P + C::GS_PAD;
#pragma unroll
        for (int c = 0; c < C::CPT; ++c) Gs[grow * D + gcol(c)] = G[c];
        __syncthreads();
        int row_first = 0;  // state rows left to the four-row passes below
        if constexpr (D == 64) {
            // the four d x d memories in 8 x 8 register tiles: warp w owns rows 32w..32w+31,
            // lane = (row group lane / 8) x (column group lane % 8); the row group takes the
            // rows 4 apart and the column group columns 4 cg..4 cg+3 and 32 + 4 cg..+3, so
            // the vector reads of the state and of G hit distinct banks.  Every loaded entry
            // of G serves eight rows and every state entry eight columns.
            const int r0 = warp * 32 + (lane >> 3), c0 = (lane & 7) * 4;
            // pairs of adjacent columns accumulate in packed fp32x2 FMAs (each half an fp32
            // fma rounded to nearest, as fmaf), half the FMA issue slots of scalar FMAs
            unsigned long long acc2[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int m = 0; m < 4; ++m) acc2[i][m] = 0ull;
#pragma unroll 1
            for (int l = 0; l < D; l += 2) {
                float2 s2[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) s2[i] = *reinterpret_cast<const float2 *>(S + (r0 + 4 * i) * C::SS + l);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const float4 g0 = *reinterpret_cast<const float4 *>(Gs + (l + u) * D + c0);
                    const float4 g1 = *reinterpret_cast<const float4 *>(Gs + (l + u) * D + 32 + c0);
                    const unsigned long long gp[4] = {pack_f32x2(g0.x, g0.y), pack_f32x2(g0.z, g0.w),
                                                      pack_f32x2(g1.x, g1.y), pack_f32x2(g1.z, g1.w)};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float sv = u == 0 ? s2[i].x : s2[i].y;
                        const unsigned long long sp = pack_f32x2(sv, sv);
#pragma unroll
                        for (int m = 0; m < 4; ++m) fma_f32x2(acc2[i][m], sp, gp[m]);
                    }
                }
            }
            float acc[8][8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int m = 0; m < 4; ++m) unpack_f32x2(acc2[i][m], acc[i][2 * m], acc[i][2 * m + 1]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (frozen_row(a, r0 + 4 * i, D)) continue;
#pragma unroll
                for (int m = 0; m < 8; ++m) S[(r0 + 4 * i) * C::SS + (m < 4 ? c0 + m : 28 + c0 + m)] = acc[i][m];
            }
            // the eta and alpha rows on warps 0-3, one output each (row 4d + tid / d, column
            // tid % d); every read of the two rows precedes every write (named barrier 1
            // spans those four warps)
            if (tid < 2 * D) {
                const int row = 4 * D + tid / D, col = tid % D;
                float ea = 0.0f;
#pragma unroll 8
                for (int l = 0; l < D; ++l) ea = fmaf(S[row * C::SS + l], Gs[l * D + col], ea);
                asm volatile("bar.sync 1, %0;" ::"n"(2 * D) : "memory");
                if (!frozen_row(a, row, D)) S[row * C::SS + col] = ea;
            }
            row_first = C::R;
        }
        // four state rows per warp and pass: each loaded column entry of G serves four rows
        constexpr int RB = 4;
        for (int o0 = row_first + warp * RB; o0 < C::R; o0 += C::NW * RB) {
            float acc[RB][C::CPL];
#pragma unroll
            for (int rr = 0; rr < RB; ++rr)
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) acc[rr][m] = 0.0f;
            const int nr = min(RB, C::R - o0);
#pragma unroll 4
            for (int l = 0; l < D; ++l) {
                float gl[C::CPL];
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) {
                    const int i = lane + 32 * m;
                    gl[m] = i < D ? Gs[l * D + i] : 0.0f;
                }
#pragma unroll
                for (int rr = 0; rr < RB; ++rr) {
                    if (rr < nr) {
                        const float sv = S[(o0 + rr) * C::SS + l];
#pragma unroll
                        for (int m = 0; m < C::CPL; ++m) acc[rr][m] = fmaf(sv, gl[m], acc[rr][m]);
                    }
                }
            }
            __syncwarp();
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) {
                // a memory held fixed by an ablation switch keeps its boundary value
                if (rr >= nr || frozen_row(a, o0 + rr, D)) continue;
#pragma unroll
                for (int m = 0; m < C::CPL; ++m) {
                    const int i = lane + 32 * m;
                    if (i < D) S[(o0 + rr) * C::SS + i] = acc[rr][m];
                }
            }
            __syncwarp();
        }
    }
    __syncthreads();

    if (a.mem_out &&
        VH_IN(a.stats, (((size_t)b * 4 + r) * a.nh + h) * SZ, SZ, (size_t)a.B * 4 * a.nh * SZ)) {
        float *mo = a.mem_out + (((size_t)b * 4 + r) * a.nh + h) * SZ;
        for (int e = tid; e < C::R * D; e += C::NT) mo[e] = S[(e / D) * C::SS + (e % D)];
    }
    if (a.stats) {
        if (n_spec) atomicAdd(&st_cnt[0], (unsigned long long)n_spec);
        if (n_inj) atomicAdd(&st_cnt[1], (unsigned long long)n_inj);
        if (n_nf) atomicAdd(&st_cnt[2], (unsigned long long)n_nf);
        __syncthreads();
        if (tid == 0) {
            atomicAdd(a.stats + VH_STAT_TOKENS, (unsigned long long)N);
            if (st_cnt[0]) atomicAdd(a.stats + VH_STAT_SPEC_ACTIVE, st_cnt[0]);
            if (st_cnt[1]) atomicAdd(a.stats + VH_STAT_INJ_RATIO_GT1, st_cnt[1]);
            if (st_cnt[2]) atomicAdd(a.stats + VH_STAT_NONFINITE, st_cnt[2]);
        }
    }
}

template <int D, typename XT>
__global__ void __launch_bounds__(256) scan_simt_kernel(const ScanArgs a)
{
    scan_simt_body<D, XT>(a);
}

// d = 64: two CTAs per SM (their shared memory fits twice), registers capped to match
template <typename XT>
__global__ void __launch_bounds__(256, 2) scan_simt_kernel_d64(const ScanArgs a)
{
    scan_simt_body<64, XT>(a);
}

template <int D, typename XT>
static cudaError_t launch_simt_t(const ScanArgs &a, cudaStream_t st)
{
    using C = SimtCfg<D>;
    void (*kern)(const ScanArgs);
    if constexpr (D == 64)
        kern = scan_simt_kernel_d64<XT>;
    else
        kern = scan_simt_kernel<D, XT>;
    static int attr_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const unsigned grid = (unsigned)(a.B * a.ndirs * a.nh);
    kern<<<grid, C::NT, C::BYTES, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_scan_simt(const ScanArgs &a, int d, bool bf16, cudaStream_t st)
{
    switch (d) {
    case 16: return bf16 ? launch_simt_t<16, __nv_bfloat16>(a, st) : launch_simt_t<16, float>(a, st);
    case 32: return bf16 ? launch_simt_t<32, __nv_bfloat16>(a, st) : launch_simt_t<32, float>(a, st);
    case 64: return bf16 ? launch_simt_t<64, __nv_bfloat16>(a, st) : launch_simt_t<64, float>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace vh
