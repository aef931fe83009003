// vh_scan_tc64.cu -- tensor-core (tcgen05 + TMA) kernel of the four-direction VisionHOPE
// memory scan for head_dim 64, bf16 feature maps and chunks aligned with rows/columns
// ("VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.3 Eq. (25);
// App. C.1 gives the third stage its 14-token chunks).
//
// One CTA (eight warps) owns one scan (image b, route r, head h); one CTA per SM.  The
// 4d + 2 = 258 state rows in three bf16 pieces (the operand form, s = s1 + s2 + s3 to
// 2^-27 relative) take 104 KB of shared memory, and the chunk-end update's two 128-row
// tiles with the gain's pieces stacked along N take 384 of the 512 TMEM columns.  Per
// 32-token sub-tile of a chunk (a chunk is one image row or column):
//   TMA    eight 8-channel x 32-token boxes of the NHWC map land as the K-major operand;
//          reverse routes load the same boxes and index them backwards.
//   MMA 1  generation, Eq. (15): [s_eta s_alpha 0.. | k_raw | v | q_raw] = x (s1+s2+s3)^T,
//          M = 128 (the tokens land in TMEM lanes 0..31), N = 208, one MMA per piece and
//          K step (x is exact in bf16).
//   SIMT   lane = token, warps 0 and 4 sharing the lanes: stabilised L2 norms of k and q
//          (App. C.1, App. B.5), delta = k - v, the queries' operand pieces; then the
//          Eq. (53) gates and Def. 1 step control with the App. B.3 safeguards (warp 1)
//          beside the Gram entries of four-token blocks (warps 2 and 3).
//   MMA 2  readout, Eq. (16): y = q M^m_b^T, six split cross terms, N = 64, issued before
//          the gain and added to out (lambda_r y at the token's pixel, Eq. (26)) after it.
//   GAIN   the shared gain of Prop. 2, Eq. (46), in one of two forms:
//          - recurrence (chunks longer than a sub-tile): G_t = alpha_t G_{t-1} -
//            eta_t (G_{t-1} k_t + delta_t) k_t^T on all 256 threads, four lanes per row of
//            G, sixteen columns each, in the scaled form G = gamma Ghat, blocks of four
//            tokens;
//          - WY (every chunk within one sub-tile, the stage-3 shape): Eq. (46) unrolled
//            over the chunk gives G = gamma_L I + sum_j sigma_j w_j k_j^T with
//            w_j = -eta_j (r_j + sum_{i<j} c(i,j) w_i), r_j = gamma_{j-1} k_j + delta_j and
//            c(i,j) = (prod_{i<s<j} alpha_s) k_i.k_j, retention products only; the Gram
//            entries and this triangular system run on CUDA cores (warps 0 and 1, one
//            row of G per thread), and G = gamma_L I + W' K^T is one tensor-core
//            assembly (three to six MMAs, keys as the MN-major A operand).
//   MMA 3  at the chunk end every memory <- M_b G: the k, v memories and the q, m memories
//          as two M = 128 tiles; per K step one MMA per piece of M_b against G's pieces
//          stacked along N (192, 128, 64 columns), the six cross terms in three column
//          blocks; G - I instead of G when the chunk retains at least half of the state
//          (the epilogue adds M_b in fp32).  The 1 x d eta and alpha rows on CUDA cores.
// Every mbarrier wait is bounded (clock64); on expiry the kernel records VH_STAT_TIMEOUT
// (when stats are given), issues no further asynchronous work and runs to its end.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "vh_tc_ptx.cuh"

namespace vh {
namespace tc64 {

using namespace vh::tc;

constexpr int D = 64;                    // head dim of this kernel
constexpr int TT = 32;                   // tokens per sub-tile
constexpr int NT = 256;                  // eight warps
constexpr int LBO = 128;                 // K-direction core-matrix stride of a K = 64 operand
constexpr int SBO = 8 * D * 2;           // 8-row group stride of a K = 64 operand (1 KB)
constexpr int ROW_MEM = 16;              // rows 0, 1: eta, alpha; 2..15 zero; then k, v, q, m
constexpr int S_ROWS = ROW_MEM + 4 * D;  // 272
constexpr int S_PIECE = S_ROWS / 8 * SBO;
constexpr int N_GEN = ROW_MEM + 3 * D;   // generation columns: eta, alpha, zeros, k, v, q
constexpr int LBO_X = TT * 16;           // K-direction stride of the TMA-loaded x tile
constexpr int SBO_X = 128;
constexpr int Q_PIECE = TT / 8 * SBO;    // queries: rows = tokens, K = 64
// The gain as the update's B operand is MN-major (N contiguous): element (n, k) of piece p
// at (k/8) G_KSTR + (8p + n/8) 128 + (k%8) 16 + (n%8) 2, so the pieces stack along N.
constexpr int G_NSTR = 128, G_KSTR = 3 * (D / 8) * G_NSTR;
constexpr int G_BYTES = D / 8 * G_KSTR;
constexpr int KS = D + 4;                // fp32 row stride of the key / delta tiles
constexpr int GFS = D + 4;               // fp32 row stride of the gain rows
constexpr int NB = 4;                    // tokens per block of the gain recurrence

constexpr int OFF_S = 0;
constexpr int OFF_X = 3 * S_PIECE;
constexpr int OFF_Q = OFF_X + TT * D * 2;
constexpr int OFF_G = OFF_Q + 3 * Q_PIECE;
constexpr int OFF_GF = OFF_G + G_BYTES;
constexpr int OFF_KF = OFF_GF + D * GFS * 4;
constexpr int OFF_DL = OFF_KF + TT * KS * 4;
constexpr int OFF_SEA = OFF_DL + TT * KS * 4;
constexpr int OFF_SC = OFF_SEA + 2 * D * 4;
constexpr int OFF_GT = OFF_SC + TT * 16;
// WY form (chunks of at most one sub-tile): the keys' operand pieces (MN-major A of the
// gain assembly: element (column b, token j, piece p) at (j/8) KP_KSTR + (8p + b/8) 128 +
// (j%8) 16 + (b%8) 2), the solution's pieces W' (K-major B: row n = 64p + a, K = token,
// element at (n/8) WP_SBO + (j/8) 128 + (n%8) 16 + (j%8) 2) and the Gram entries (fp32).
constexpr int KP_KSTR = 3 * (D / 8) * 128;
constexpr int OFF_KP = OFF_GT + TT / NB * 8 * 4;
constexpr int WP_SBO = TT / 8 * 128;
constexpr int OFF_WP = OFF_KP + TT / 8 * KP_KSTR;
constexpr int GRS = TT + 4;
constexpr int OFF_GR = OFF_WP + 3 * D / 8 * WP_SBO;
constexpr int OFF_BAR = OFF_GR + TT * GRS * 4;
constexpr int SMEM_BYTES = OFF_BAR + 128;
static_assert(OFF_KP + TT / 8 * KP_KSTR + 2048 <= SMEM_BYTES, "assembly operand rows stay in shared memory");
static_assert(SMEM_BYTES <= 227 * 1024, "one CTA per SM");
static_assert(OFF_X % 1024 == 0, "x tile aligned");
// the M = 128 operands read past their data: rows 32..127 of the x tile and the queries
static_assert(OFF_X + 7 * LBO_X + 16 * SBO_X <= OFF_G, "x operand rows stay in shared memory");
static_assert(OFF_Q + 2 * Q_PIECE + 16 * SBO <= SMEM_BYTES, "query operand rows stay in shared memory");
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: the generation at 0..207, the update's two tiles at 0..191 and 192..383
// (issued after the generation is consumed), the readout at 448..511.
constexpr int COL_GEN = 0, COL_K = ROW_MEM, COL_V = ROW_MEM + D, COL_QR = ROW_MEM + 2 * D;
constexpr int COL_UPD = 0, UPD_TILE = 3 * D, COL_RO = 448;

// Byte offset of row `row`, K-group g (8 elements) in a K = 64 K-major operand.
__device__ __forceinline__ int op64(int row, int g) { return (row >> 3) * SBO + g * LBO + (row & 7) * 16; }

// 64 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld64(uint32_t ta, float (&v)[64])
{
    float a[32], b[32];
    tmem_ld32(ta, a);
    tmem_ld32(ta + 32, b);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = a[i];
        v[32 + i] = b[i];
    }
}

__device__ __forceinline__ float sumsq64(const float (&v)[64])
{
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = v[e] * v[e];
#pragma unroll
    for (int e = 8; e < 64; ++e) a[e & 7] = fmaf(v[e], v[e], a[e & 7]);
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// The chunk's triangular system for gain row a (lane = a), as in the d = 32 kernel's WY
// form ("VisionHOPE", App. B.4 Prop. 2, Eqs. (46), (49) unrolled):
//   G = gamma_L I + sum_j sigma_j w_j k_j^T,  w_j = -eta_j (r_j + sum_{i<j} c(i, j) w_i),
//   r_j = gamma_{j-1} k_j + delta_j,  c(i, j) = (prod_{i<s<j} alpha_s) k_i . k_j,
// every factor a product of retentions.  With at most 32 tokens the coefficients are
// formed on the fly from the Gram entries (a running product along each row).  Then
// W' = sigma_j w_j goes out as the assembly's B operand (row a of each piece, K = token,
// zero past LP).
template <int LP>
__device__ __forceinline__ void wy64_solve(const float *__restrict__ dl, const float *__restrict__ gr,
                                           const float *__restrict__ alp, const float *__restrict__ eta,
                                           const float *__restrict__ sig, unsigned char *wp, int a)
{
    float acc[LP];
#pragma unroll
    for (int j = 0; j < LP; ++j) acc[j] = dl[j * KS + a];
#pragma unroll
    for (int i = 0; i < LP; ++i) {
        const float w = -eta[i] * acc[i];
        acc[i] = w;
        float rat = 1.0f;
#pragma unroll
        for (int j4 = (i + 1) & ~3; j4 < LP; j4 += 4) {
            const float4 g4 = *reinterpret_cast<const float4 *>(gr + i * GRS + j4);
            const float4 a4 = *reinterpret_cast<const float4 *>(alp + j4);
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (j4 + u > i) {
                    acc[j4 + u] = fmaf(rat * gv[u], w, acc[j4 + u]);
                    rat *= av[u];
                }
            }
        }
    }
#pragma unroll
    for (int g = 0; g < TT / 8; ++g) {
        float v8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v8[u] = (8 * g + u < LP) ? sig[8 * g + u] * acc[(8 * g + u) % LP] : 0.0f;
        store_split8(wp + (a >> 3) * WP_SBO + g * 128 + (a & 7) * 16, 8 * WP_SBO, v8);
    }
}

// kWY: the shared gain in WY form (every chunk within one sub-tile); otherwise the blocked
// recurrence on all 256 threads.
template <bool kWY>
__global__ void __launch_bounds__(NT, 1)
    scan_tc64_kernel(const ScanArgs a, const __grid_constant__ CUtensorMap tm_row,
                     const __grid_constant__ CUtensorMap tm_col)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int id = blockIdx.x;
    const int h = id % a.nh;
    id /= a.nh;
    const int r = a.dir_list[id % a.ndirs];
    const int b = id / a.ndirs;
    const int H = a.H, W = a.W, Cc = a.Cc;
    const bool rowr = r < 2, rev = (r & 1) != 0;
    const int Lline = rowr ? W : H;            // chunk length (Eq. (25))
    const int nlines = rowr ? H : W;           // chunks per route
    const int nsub = (Lline + TT - 1) / TT;    // sub-tiles per chunk
    const CUtensorMap *tm = rowr ? &tm_row : &tm_col;
    const size_t SZ = (size_t)4 * D * D + 2 * D;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    const uint32_t mb_x = smem_u32(&bars[0]), mb_gen = smem_u32(&bars[1]);
    const uint32_t mb_ro = smem_u32(&bars[2]), mb_upd = smem_u32(&bars[3]);
    const uint32_t mb_drain = smem_u32(sm + OFF_BAR + 112);  // end of a CTA that gave up
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 64);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_BAR + 72);
    volatile int *delta_form = reinterpret_cast<volatile int *>(sm + OFF_BAR + 80);
    volatile int *vote = reinterpret_cast<volatile int *>(sm + OFF_BAR + 96);
    const Waiter wt{abort_flag, a.stats, a.wait_limit > 0 ? a.wait_limit : (1ll << 32)};

    unsigned char *sX = sm + OFF_X, *sS = sm + OFF_S, *sQ = sm + OFF_Q, *sG = sm + OFF_G;
    float *Kf = reinterpret_cast<float *>(sm + OFF_KF);
    float *DLf = reinterpret_cast<float *>(sm + OFF_DL);
    float *Gf = reinterpret_cast<float *>(sm + OFF_GF);
    float *Sea = reinterpret_cast<float *>(sm + OFF_SEA);
    float4 *SC = reinterpret_cast<float4 *>(sm + OFF_SC);
    float *GT = reinterpret_cast<float *>(sm + OFF_GT);

    // ---- set-up: barriers, TMEM, first TMA, initial state
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(mb_x, 1);
        mbar_init(mb_gen, 1);
        mbar_init(mb_ro, 1);
        mbar_init(mb_upd, 1);
        mbar_init(mb_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    auto line_of = [&](int c) { return rev ? nlines - 1 - c : c; };
    auto box_start = [&](int s) { return rev ? Lline - (s + 1) * TT : s * TT; };
    // x copies issued and completions observed (issuing thread); at most one copy is in
    // flight, so after an abort the drain waits for completion number nx_iss - 1
    uint32_t nx_iss = 0, nx_obs = 0;
    auto issue_x = [&](int c, int s) {
        ++nx_iss;
        mbar_expect_tx(mb_x, TT * D * 2);
#pragma unroll
        for (int q = 0; q < D / 8; ++q)
            tma_load_4d(smem_u32(sX + q * LBO_X), tm, h * D + 8 * q, box_start(s), line_of(c), b, mb_x);
    };
    __syncthreads();  // barriers initialised, TMEM address written
    const bool issuer = warp == 3 && lane == 0;  // MMA and TMA issue; no token work
    if (issuer) issue_x(0, 0);
    // checked indices (VH_DEBUG_BOUNDS builds; `true` otherwise): this scan's slices of
    // memories0 and memories_out, checked once for their whole extent
    const size_t mem_base = ((size_t)r * a.nh + h) * SZ;
    const bool mo_ok = !a.mem_out ||
                       VH_IN(a.stats, (((size_t)b * 4 + r) * a.nh + h) * SZ, SZ, (size_t)a.B * 4 * a.nh * SZ);
    {
        const float *m0 = a.mem0 + (VH_IN(a.stats, mem_base, SZ, (size_t)4 * a.nh * SZ) ? mem_base : 0);
        // memory rows 0..255 (k, v, q, m) -> operand rows 16..271: thread = row
        float v[64];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(m0 + (size_t)tid * D) + e);
            v[4 * e] = f.x; v[4 * e + 1] = f.y; v[4 * e + 2] = f.z; v[4 * e + 3] = f.w;
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) store_split8(sS + op64(ROW_MEM + tid, g), S_PIECE, v + 8 * g);
        // eta / alpha rows: fp32 copy and operand rows 0, 1; rows 2..15 are zero
        if (tid < 2 * D) Sea[tid] = m0[4 * D * D + tid];
        if (tid < ROW_MEM) {
            float z[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) {
#pragma unroll
                for (int e = 0; e < 8; ++e) z[e] = tid < 2 ? m0[4 * D * D + tid * D + 8 * g + e] : 0.0f;
                store_split8(sS + op64(tid, g), S_PIECE, z);
            }
        }
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t lrow = ((uint32_t)(warp & 3) * 32u) << 16;  // this warp's TMEM lane quarter

    const float *lam = a.dir_scale ? a.dir_scale + (size_t)r * Cc + (size_t)h * D : nullptr;
    float *ob = a.out + (size_t)b * H * W * Cc + (size_t)h * D;
    unsigned n_spec = 0, n_inj = 0, n_nf = 0;
    uint32_t ph_x = 0, ph_gen = 0, ph_ro = 0, ph_upd = 0;

    // gain state: thread t owns row t/4 of G = gam * ghat, columns 16(t%4)..+15
    const int grow = tid >> 2, gq = tid & 3;
    float gh[16];
    float gam = 1.0f, inv_gam = 1.0f;
    // the token of this thread's TMEM lane (warps 0 and 4: box row = lane)
    const bool tokw = (warp & 3) == 0;

    // the 1 x d eta and alpha rows advanced by G on CUDA cores, in fp32 (one warp, lane =
    // column pair): eta <- eta G, alpha <- alpha G, with their operand rows re-split
    auto eta_alpha_rows = [&]() {
                    float ne0 = 0.0f, na0 = 0.0f, ne1 = 0.0f, na1 = 0.0f;
#pragma unroll 8
                    for (int l = 0; l < D; ++l) {
                        const float g0 = Gf[l * GFS + lane], g1 = Gf[l * GFS + 32 + lane];
                        ne0 = fmaf(Sea[l], g0, ne0);
                        na0 = fmaf(Sea[D + l], g0, na0);
                        ne1 = fmaf(Sea[l], g1, ne1);
                        na1 = fmaf(Sea[D + l], g1, na1);
                    }
                    __syncwarp();
                    Sea[lane] = ne0;
                    Sea[32 + lane] = ne1;
                    Sea[D + lane] = na0;
                    Sea[D + 32 + lane] = na1;
                    const float vals[4] = {ne0, ne1, na0, na1};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int row = k >> 1, col = lane + 32 * (k & 1);
                        __nv_bfloat16 p1, p2, p3;
                        split3(vals[k], p1, p2, p3);
                        unsigned char *d0 = sS + op64(ROW_MEM * 0 + row, col >> 3) + 2 * (col & 7);
                        *reinterpret_cast<__nv_bfloat16 *>(d0) = p1;
                        *reinterpret_cast<__nv_bfloat16 *>(d0 + S_PIECE) = p2;
                        *reinterpret_cast<__nv_bfloat16 *>(d0 + 2 * S_PIECE) = p3;
                    }
                    };
    // new state rows after the update MMA: thread = memory row (TMEM lane of its tile), the
    // three column blocks summed, re-split into the operand pieces; in the increment form M_b
    // is recovered exactly from its three pieces and added in fp32
    int c = 0;
    auto resplit = [&]() {
                const int tl = warp >> 2;
                const int mrow = ROW_MEM + 128 * tl + 32 * (warp & 3) + lane;
                float v[64];
                {
                    float w2[64];
                    tmem_ld64(tbase + lrow + COL_UPD + UPD_TILE * tl, v);
                    tmem_ld64(tbase + lrow + COL_UPD + UPD_TILE * tl + D, w2);
#pragma unroll
                    for (int e = 0; e < 64; ++e) v[e] += w2[e];
                    tmem_ld64(tbase + lrow + COL_UPD + UPD_TILE * tl + 2 * D, w2);
#pragma unroll
                    for (int e = 0; e < 64; ++e) v[e] += w2[e];
                }
                const bool add_mb = *delta_form != 0;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    unsigned char *src = sS + op64(mrow, g);
                    if (add_mb) {
                        const uint4 u1 = *reinterpret_cast<const uint4 *>(src);
                        const uint4 u2 = *reinterpret_cast<const uint4 *>(src + S_PIECE);
                        const uint4 u3 = *reinterpret_cast<const uint4 *>(src + 2 * S_PIECE);
                        const uint32_t *w1 = &u1.x, *x2 = &u2.x, *x3 = &u3.x;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            v[8 * g + 2 * i] += (bf16_lo(w1[i]) + bf16_lo(x2[i])) + bf16_lo(x3[i]);
                            v[8 * g + 2 * i + 1] += (bf16_hi(w1[i]) + bf16_hi(x2[i])) + bf16_hi(x3[i]);
                        }
                    }
                    store_split8(src, S_PIECE, v + 8 * g);
                }
                if (c == nlines - 1 && a.mem_out && mo_ok) {
                    float *mo = a.mem_out + (((size_t)b * 4 + r) * a.nh + h) * SZ;
                    float4 *d4 = reinterpret_cast<float4 *>(mo + (size_t)(mrow - ROW_MEM) * D);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                }
                };

    for (c = 0; c < nlines; ++c) {
        const int Lidx = line_of(c);
        for (int s = 0; s < nsub; ++s) {
            const int t0 = s * TT;
            const int Lt = min(TT, Lline - t0);
            const bool last = s == nsub - 1;
            const int p = box_start(s) + lane;  // position along the line (token warps)
            const int jr = (rev ? Lline - 1 - p : p) - t0;  // route-ordered index in the sub-tile
            const bool jr_in = !tokw || VH_IN(a.stats, jr, 1, TT);  // (token warps' row index)
            const bool valid = tokw && p >= 0 && p < Lline && jr_in;
            // ---- MMA 1: generation from the boundary state, Eq. (15)
            if (issuer) {
                tc_after();
                const bool got_x = wt.wait(mb_x, ph_x);
                nx_obs += got_x;
                if (got_x && !*abort_flag) {
                    const uint64_t dx = sdesc(smem_u32(sX), LBO_X, SBO_X);
                    const uint64_t ds = sdesc(smem_u32(sS), LBO, SBO);
#pragma unroll
                    for (int pc = 0; pc < 3; ++pc)
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            mma(tbase + COL_GEN, dadd(dx, ks * 2 * LBO_X), dadd(ds, pc * S_PIECE + ks * 2 * LBO),
                                idesc_bf16(128, N_GEN), (pc | ks) != 0);
                    mma_commit(mb_gen);
                }
            }
            ph_x ^= 1;
            wt.wait(mb_gen, ph_gen);
            ph_gen ^= 1;
            tc_after();
            // the x tile is free again: fetch the next sub-tile while this one is processed
            if (issuer && !*abort_flag) {
                const int ns = (s + 1 < nsub) ? s + 1 : 0;
                const int nc = (s + 1 < nsub) ? c : c + 1;
                if (nc < nlines) issue_x(nc, ns);
            }
            if constexpr (kWY) {
            // ================= WY form of the shared gain (one sub-tile per chunk) =========
            float *ALP = reinterpret_cast<float *>(SC), *ETA = ALP + TT, *GPRE = ETA + TT, *SIG = GPRE + TT;
            float *GR = reinterpret_cast<float *>(sm + OFF_GR);
            unsigned char *sKP = sm + OFF_KP, *sWP = sm + OFF_WP;
            float *gam_slot = reinterpret_cast<float *>(sm + OFF_BAR + 84);
            const int Lp = Lt <= 16 ? 16 : 32;  // size of the triangular system (tokens past Lt are zero)
            // ---- per-token step.  Warp 0 (lane = token): norms, delta, gates and step control,
            // the retention products along the route, the shifted deltas r_j, the fp32 keys
            // (for the Gram warps) and the keys' operand pieces.  Warp 4: the queries, handed
            // to the issuer for the readout MMA.  Warps 1, 2, 5, 6: the Gram entries once the
            // keys are written.
            if (warp == 0) {
                float kr[64], vv[64];
                tmem_ld64(tbase + lrow + COL_K, kr);
                tmem_ld64(tbase + lrow + COL_V, vv);
                float se, sa;
                tmem_ld2(tbase + lrow + COL_GEN, se, sa);
                const float kkr = sumsq64(kr);
                const float rk = __frsqrt_rn(kkr + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    kr[e] *= rk;            // k
                    vv[e] = kr[e] - vv[e];  // delta = k - v
                }
                const float kn2 = sumsq64(kr), dd2 = sumsq64(vv);
                if (!valid) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) kr[e] = 0.0f;
                }
                if (jr_in) {
                    float4 *kd = reinterpret_cast<float4 *>(Kf + jr * KS);
#pragma unroll
                    for (int e = 0; e < 16; ++e) kd[e] = make_float4(kr[4 * e], kr[4 * e + 1], kr[4 * e + 2], kr[4 * e + 3]);
                }
                __threadfence_block();
                named_arrive(1, 5 * 32);  // keys written: the Gram warps may start
                float alpha = 1.0f, eta_t = 0.0f;
                if (valid) {
                    float eta, oma;
                    gates(a, se, sa, eta, alpha, oma);
                    if (a.gate_mode == VH_GATE_FORCED_EXEC) {
                        eta_t = a.forced_eta;
                    } else {
                        const StepOut so = step_control<false>(a, eta, alpha, oma, kn2, dd2);
                        eta_t = so.eta_tilde;
                        n_spec += so.spec_active;
                        n_inj += so.inj_ratio_gt1;
                    }
                }
                if (jr_in) {
                    ALP[jr] = alpha;
                    ETA[jr] = eta_t;
                }
                __syncwarp();
                // prefix and suffix products of the retentions in route order (lane = route index)
                float pre = ALP[lane], suf = pre;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t1 = __shfl_up_sync(0xffffffffu, pre, o);
                    const float t2 = __shfl_down_sync(0xffffffffu, suf, o);
                    if (lane >= o) pre *= t1;
                    if (lane + o < 32) suf *= t2;
                }
                float gp = __shfl_up_sync(0xffffffffu, pre, 1), sg = __shfl_down_sync(0xffffffffu, suf, 1);
                if (lane == 0) gp = 1.0f;
                if (lane == 31) sg = 1.0f;
                GPRE[lane] = gp;
                SIG[lane] = sg;
                if (lane == Lt - 1) *gam_slot = pre;  // gamma_L
                __syncwarp();
                // r_j = gamma_{j-1} k_j + delta_j (zero past the chunk)
                const float gj = jr_in ? GPRE[jr] : 0.0f;
                float4 *dr = reinterpret_cast<float4 *>(DLf + (jr_in ? jr : 0) * KS);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (jr_in) dr[e] = valid ? make_float4(fmaf(gj, kr[4 * e], vv[4 * e]), fmaf(gj, kr[4 * e + 1], vv[4 * e + 1]),
                                                fmaf(gj, kr[4 * e + 2], vv[4 * e + 2]), fmaf(gj, kr[4 * e + 3], vv[4 * e + 3]))
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            } else if (warp == 4) {
                float qr[64];
                tmem_ld64(tbase + lrow + COL_QR, qr);
                const float rq = __frsqrt_rn(sumsq64(qr) + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 64; ++e) qr[e] *= rq;
#pragma unroll
                for (int g = 0; g < 8; ++g) store_split8(sQ + op64(lane, g), Q_PIECE, qr + 8 * g);
                fence_async_smem();
                tc_before();
                named_arrive(2, 64);  // queries written: the issuer may start the readout
            } else if (warp == 3) {
                named_sync(2, 64);
                tc_after();
                // MMA 2: readout y = q M^m_b^T, Eq. (16), six split cross terms
                if (issuer && !*abort_flag) {
                    constexpr int pa[6] = {0, 0, 1, 0, 2, 1};
                    constexpr int pb[6] = {0, 1, 0, 2, 0, 1};
                    const uint64_t da = sdesc(smem_u32(sQ), LBO, SBO);
                    const uint64_t db = sdesc(smem_u32(sS) + (ROW_MEM + 3 * D) / 8 * SBO, LBO, SBO);
#pragma unroll
                    for (int t = 0; t < 6; ++t)
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            mma(tbase + COL_RO, dadd(da, pa[t] * Q_PIECE + ks * 2 * LBO),
                                dadd(db, pb[t] * S_PIECE + ks * 2 * LBO), idesc_bf16(128, D), (t | ks) != 0);
                    mma_commit(mb_ro);
                }
            } else if (warp == 1 || warp == 2 || warp == 5 || warp == 6) {
                // the keys' operand pieces (MN-major: 8 consecutive columns b per 16-byte run;
                // zero rows past the chunk) and the Gram entries k_i . k_j, i < j < Lp (zero past
                // the chunk), route order
                named_sync(1, 5 * 32);
                const int gt = (warp == 1 ? 0 : warp == 2 ? 1 : warp == 5 ? 2 : 3) * 32 + lane;
#pragma unroll
                for (int u = 0; u < TT * (D / 8) / 128; ++u) {
                    const int item = gt + 128 * u, j = item >> 3, g = item & 7;
                    const float4 f0 = *reinterpret_cast<const float4 *>(Kf + j * KS + 8 * g);
                    const float4 f1 = *reinterpret_cast<const float4 *>(Kf + j * KS + 8 * g + 4);
                    const float v8[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
                    store_split8(sKP + (j >> 3) * KP_KSTR + g * 128 + (j & 7) * 16, 1024, v8);
                }
                const int npair = Lp * (Lp - 1) / 2;
                for (int pr = gt; pr < npair; pr += 128) {
                    // pair index -> (i, j), i < j: row i holds Lp - 1 - i pairs
                    int i = 0, rem = pr;
                    while (rem >= Lp - 1 - i) { rem -= Lp - 1 - i; ++i; }
                    const int j = i + 1 + rem;
                    float g = 0.0f;
                    if (j < Lt) {
                        const float4 *ka = reinterpret_cast<const float4 *>(Kf + i * KS);
                        const float4 *kb = reinterpret_cast<const float4 *>(Kf + j * KS);
                        float g4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float4 fa = ka[e], fb = kb[e];
                            g4[0] = fmaf(fa.x, fb.x, g4[0]);
                            g4[1] = fmaf(fa.y, fb.y, g4[1]);
                            g4[2] = fmaf(fa.z, fb.z, g4[2]);
                            g4[3] = fmaf(fa.w, fb.w, g4[3]);
                        }
                        g = (g4[0] + g4[1]) + (g4[2] + g4[3]);
                    }
                    GR[i * GRS + j] = g;
                }
            }
            fence_async_smem();
            tc_before();
            __syncthreads();
            tc_after();
            // ---- the solve (warps 0, 1: lane = gain row) while warp 4 adds the readout to out
            if (warp < 2) {
                if (Lp == 16)
                    wy64_solve<16>(DLf, GR, ALP, ETA, SIG, sWP, 32 * warp + lane);
                else
                    wy64_solve<32>(DLf, GR, ALP, ETA, SIG, sWP, 32 * warp + lane);
                fence_async_smem();
            } else if (warp == 4) {
                wt.wait(mb_ro, ph_ro);
                tc_after();
                float y[32], y2[32];
                tmem_ld32(tbase + lrow + COL_RO, y);
                tmem_ld32(tbase + lrow + COL_RO + 32, y2);
                const int pix = rowr ? Lidx * W + p : p * W + Lidx;
                if (valid && VH_IN(a.stats, ((size_t)b * H * W + pix) * Cc + (size_t)h * D, D, map_elems(a))) {
                    float *dst = ob + (size_t)pix * Cc;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float *yy = e < 8 ? y : y2;
                        const int k = 4 * (e & 7);
                        float4 v4 = make_float4(yy[k], yy[k + 1], yy[k + 2], yy[k + 3]);
                        if (lam) {
                            v4.x *= lam[4 * e]; v4.y *= lam[4 * e + 1];
                            v4.z *= lam[4 * e + 2]; v4.w *= lam[4 * e + 3];
                        }
                        n_nf += !isfinite(v4.x) + !isfinite(v4.y) + !isfinite(v4.z) + !isfinite(v4.w);
                        red_add_v4(dst + 4 * e, v4);
                    }
                }
            }
            ph_ro ^= 1;
            tc_before();
            __syncthreads();
            tc_after();
            // ---- G^T = gamma_L I + K W'^T on the tensor core: the keys' pieces as the MN-major A
            // operand (rows = columns b of G), W' as B with its pieces stacked along N
            // (192, 128, 64): the six cross terms in three column blocks of 64
            if (issuer && !*abort_flag) {
                const uint64_t dk = sdesc(smem_u32(sKP), KP_KSTR, 128);
                const uint64_t dw = sdesc(smem_u32(sWP), 128, WP_SBO);
                for (int ks = 0; ks < Lp / 16; ++ks)
#pragma unroll
                    for (int pc = 0; pc < 3; ++pc)
                        mma(tbase + COL_UPD, dadd(dk, pc * 1024 + ks * 2 * KP_KSTR), dadd(dw, ks * 256),
                            idesc_bf16(128, 3 * D - D * pc, false, true), (ks | pc) != 0);
                mma_commit(mb_upd);
            }
            if ((warp & 3) < 2) {
                // column b = this lane's TMEM row of G; warps 0, 1 hold rows a = 0..31 of their
                // columns, warps 4, 5 rows 32..63: fp32 rows for the eta / alpha rows and the
                // update's B operand (K-major: row n = b, K = a; G - I when the chunk retains at
                // least half of the state)
                wt.wait(mb_upd, ph_upd);
                tc_after();
                const int bcol = 32 * (warp & 3) + lane, half = warp >> 2;
                float v[32], w2[32];
                tmem_ld32(tbase + lrow + COL_UPD + 32 * half, v);
                tmem_ld32(tbase + lrow + COL_UPD + D + 32 * half, w2);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] += w2[e];
                tmem_ld32(tbase + lrow + COL_UPD + 2 * D + 32 * half, w2);
                const float gL = *gam_slot;
                const bool use_delta = gL >= 0.5f;
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = (v[e] + w2[e]) + (32 * half + e == bcol ? gL : 0.0f);
#pragma unroll
                for (int e = 0; e < 32; ++e) Gf[(32 * half + e) * GFS + bcol] = v[e];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float v8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        v8[u] = v[8 * g + u] - ((use_delta && 32 * half + 8 * g + u == bcol) ? 1.0f : 0.0f);
                    store_split8(sG + (bcol >> 3) * SBO + (4 * half + g) * LBO + (bcol & 7) * 16, 8 * SBO, v8);
                }
                if (warp == 0 && lane == 0) *delta_form = use_delta ? 1 : 0;
                fence_async_smem();
            }
            ph_upd ^= 1;
            tc_before();
            __syncthreads();  // G and its fp32 rows written
            tc_after();
            // ---- MMA 3 (chunk end): every d x d memory <- M_b G, with G's pieces K-major
            if (issuer && !*abort_flag) {
                const uint64_t db = sdesc(smem_u32(sG), LBO, SBO);
#pragma unroll
                for (int tl = 0; tl < 2; ++tl) {
                    const uint64_t da = sdesc(smem_u32(sS) + (ROW_MEM / 8 + 16 * tl) * SBO, LBO, SBO);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t ka = ks * 2 * LBO;
#pragma unroll
                        for (int pc = 0; pc < 3; ++pc)
                            mma(tbase + COL_UPD + UPD_TILE * tl, dadd(da, pc * S_PIECE + ka), dadd(db, ka),
                                idesc_bf16(128, 3 * D - D * pc), (ks | pc) != 0);
                    }
                }
                mma_commit(mb_upd);
            }
            if (warp == 2) eta_alpha_rows();
            wt.wait(mb_upd, ph_upd);
            ph_upd ^= 1;
            tc_after();
            resplit();
            } else {
            // ---- per-token step (lane = token).  Warp 0: stabilised norm of k, delta = k - v,
            // the token's fp32 rows and raw scalars.  Warp 4: the query, normalised and split
            // into the readout's A operand (row = box row).
            if (warp == 0) {
                float kr[64], vv[64];
                tmem_ld64(tbase + lrow + COL_K, kr);
                tmem_ld64(tbase + lrow + COL_V, vv);
                float se, sa;
                tmem_ld2(tbase + lrow + COL_GEN, se, sa);
                const float kkr = sumsq64(kr);
                const float rk = __frsqrt_rn(kkr + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    kr[e] *= rk;            // k
                    vv[e] = kr[e] - vv[e];  // delta = k - v
                }
                const float kn2 = sumsq64(kr), dd2 = sumsq64(vv);
                if (valid) {
                    float4 *kd = reinterpret_cast<float4 *>(Kf + jr * KS);
                    float4 *dd4 = reinterpret_cast<float4 *>(DLf + jr * KS);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        kd[e] = make_float4(kr[4 * e], kr[4 * e + 1], kr[4 * e + 2], kr[4 * e + 3]);
                        dd4[e] = make_float4(vv[4 * e], vv[4 * e + 1], vv[4 * e + 2], vv[4 * e + 3]);
                    }
                    SC[jr] = make_float4(se, sa, kn2, dd2);
                }
            } else if (warp == 4) {
                float qr[64];
                tmem_ld64(tbase + lrow + COL_QR, qr);
                const float rq = __frsqrt_rn(sumsq64(qr) + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 64; ++e) qr[e] *= rq;
#pragma unroll
                for (int g = 0; g < 8; ++g) store_split8(sQ + op64(lane, g), Q_PIECE, qr + 8 * g);
            }
            fence_async_smem();
            tc_before();
            __syncthreads();
            tc_after();
            // ---- MMA 2: readout y = q M^m_b^T, Eq. (16), six split cross terms; it runs while
            // the gates and the gain are formed
            if (issuer && !*abort_flag) {
                constexpr int pa[6] = {0, 0, 1, 0, 2, 1};
                constexpr int pb[6] = {0, 1, 0, 2, 0, 1};
                const uint64_t da = sdesc(smem_u32(sQ), LBO, SBO);
                const uint64_t db = sdesc(smem_u32(sS) + (ROW_MEM + 3 * D) / 8 * SBO, LBO, SBO);
#pragma unroll
                for (int t = 0; t < 6; ++t)
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma(tbase + COL_RO, dadd(da, pa[t] * Q_PIECE + ks * 2 * LBO),
                            dadd(db, pb[t] * S_PIECE + ks * 2 * LBO), idesc_bf16(128, D), (t | ks) != 0);
                mma_commit(mb_ro);
            }
            if (warp == 1) {
                // gates and step control of route-ordered token jg = lane; the coefficients
                // of the gain recurrence replace the scalars: (alpha, eta/alpha, 1/alpha, eta)
                // for the scaled form, (alpha, 0, 0, eta) where alpha is too small to divide by
                const int jg = lane;
                const bool tv = jg < Lt;
                float alpha = 1.0f;
                if (tv) {
                    const float4 sc = SC[jg];
                    float eta, oma;
                    gates(a, sc.x, sc.y, eta, alpha, oma);
                    float eta_t;
                    if (a.gate_mode == VH_GATE_FORCED_EXEC) {
                        eta_t = a.forced_eta;
                    } else {
                        const StepOut so = step_control<false>(a, eta, alpha, oma, sc.z, sc.w);
                        eta_t = so.eta_tilde;
                        n_spec += so.spec_active;
                        n_inj += so.inj_ratio_gt1;
                    }
                    const bool keep = alpha >= 1e-6f;
                    SC[jg] = make_float4(alpha, keep ? __fdividef(eta_t, alpha) : 0.0f,
                                         keep ? __frcp_rn(alpha) : 0.0f, eta_t);
                }
                const unsigned small = __ballot_sync(0xffffffffu, tv && !(alpha >= 0.01f));
                if (lane == 0) vote[0] = small != 0u;
            } else if (warp == 2 || warp == 3) {
                // Gram entries k_a . k_b, a < b, of each block of NB route-ordered tokens:
                // pair i of block q goes to thread 6q + i
                const int pr = tid - 64;
                if (pr < TT / NB * 6) {
                    const int q = pr / 6, pi = pr - 6 * q;
                    const int ia = pi < 3 ? 0 : (pi < 5 ? 1 : 2);
                    const int ib = pi < 3 ? pi + 1 : (pi < 5 ? pi - 1 : 3);
                    const float4 *ka = reinterpret_cast<const float4 *>(Kf + (NB * q + ia) * KS);
                    const float4 *kb = reinterpret_cast<const float4 *>(Kf + (NB * q + ib) * KS);
                    float g4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float4 fa = ka[e], fb = kb[e];
                        g4[0] = fmaf(fa.x, fb.x, g4[0]);
                        g4[1] = fmaf(fa.y, fb.y, g4[1]);
                        g4[2] = fmaf(fa.z, fb.z, g4[2]);
                        g4[3] = fmaf(fa.w, fb.w, g4[3]);
                    }
                    GT[q * 8 + pi] = (g4[0] + g4[1]) + (g4[2] + g4[3]);
                }
            }
            __syncthreads();
            // ---- shared gain over this sub-tile's tokens, in route order, on every thread:
            // G = gam * ghat with ghat <- ghat - (eta/alpha) (ghat k + delta / gam) k^T,
            // gam <- alpha gam, a pure scaling of G_j = alpha G_{j-1} - eta (G_{j-1} k + delta)
            // k^T.  When every alpha of the sub-tile is >= 0.01 the tokens go in blocks of NB
            // (the NB dot products independent, an NB-step scalar solve with the blocks' Gram
            // entries, one rank-NB update) and the scale is folded back when it falls below
            // 1e-20; otherwise token by token, a token with alpha < 1e-6 applied to G directly.
            {
                if (s == 0) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) gh[e] = (16 * gq + e == grow) ? 1.0f : 0.0f;
                    gam = 1.0f;
                    inv_gam = 1.0f;
                }
                const bool careful = vote[0] != 0;
                auto fold = [&]() {
#pragma unroll
                    for (int e = 0; e < 16; ++e) gh[e] *= gam;
                    gam = 1.0f;
                    inv_gam = 1.0f;
                };
                auto reduce4 = [](float v) {
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    return v + __shfl_xor_sync(0xffffffffu, v, 2);
                };
                auto apply1 = [&](int j, bool chk) {
                    float kk[16];
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const float4 f = *reinterpret_cast<const float4 *>(Kf + j * KS + 16 * gq + e);
                        kk[e] = f.x; kk[e + 1] = f.y; kk[e + 2] = f.z; kk[e + 3] = f.w;
                    }
                    const float4 cf = SC[j];
                    const float dj = DLf[j * KS + grow];
                    float p0 = gh[0] * kk[0], p1 = gh[1] * kk[1];
#pragma unroll
                    for (int e = 2; e < 16; e += 2) {
                        p0 = fmaf(gh[e], kk[e], p0);
                        p1 = fmaf(gh[e + 1], kk[e + 1], p1);
                    }
                    const float dot = reduce4(p0 + p1);
                    if (!chk || cf.z != 0.0f) {
                        const float sc = -cf.y * fmaf(dj, inv_gam, dot);
#pragma unroll
                        for (int e = 0; e < 16; ++e) gh[e] = fmaf(sc, kk[e], gh[e]);
                        gam *= cf.x;
                        inv_gam *= cf.z;
                        if (chk && gam < 1e-20f) fold();
                    } else {  // G_j = alpha G_{j-1} - eta (G_{j-1} k + delta) k^T, unscaled
                        const float sc = -cf.w * fmaf(gam, dot, dj);
                        const float ag = cf.x * gam;
#pragma unroll
                        for (int e = 0; e < 16; ++e) gh[e] = fmaf(sc, kk[e], ag * gh[e]);
                        gam = 1.0f;
                        inv_gam = 1.0f;
                    }
                };
                if (careful) {
                    for (int j = 0; j < Lt; ++j) apply1(j, true);
                } else {
                    int j = 0;
                    for (; j + NB <= Lt; j += NB) {
                        float kb[NB][16];
                        float4 cb[NB];
                        float db[NB];
#pragma unroll
                        for (int t = 0; t < NB; ++t) {
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const float4 f =
                                    *reinterpret_cast<const float4 *>(Kf + (j + t) * KS + 16 * gq + e);
                                kb[t][e] = f.x; kb[t][e + 1] = f.y; kb[t][e + 2] = f.z; kb[t][e + 3] = f.w;
                            }
                            cb[t] = SC[j + t];
                            db[t] = DLf[(j + t) * KS + grow];
                        }
                        const float4 g0 = *reinterpret_cast<const float4 *>(GT + (j / NB) * 8);
                        const float2 g1 = *reinterpret_cast<const float2 *>(GT + (j / NB) * 8 + 4);
                        float av[NB];
#pragma unroll
                        for (int t = 0; t < NB; ++t) {
                            float p0 = gh[0] * kb[t][0], p1 = gh[1] * kb[t][1];
#pragma unroll
                            for (int e = 2; e < 16; e += 2) {
                                p0 = fmaf(gh[e], kb[t][e], p0);
                                p1 = fmaf(gh[e + 1], kb[t][e + 1], p1);
                            }
                            av[t] = p0 + p1;
                        }
#pragma unroll
                        for (int t = 0; t < NB; ++t) av[t] += __shfl_xor_sync(0xffffffffu, av[t], 1);
#pragma unroll
                        for (int t = 0; t < NB; ++t) av[t] += __shfl_xor_sync(0xffffffffu, av[t], 2);
                        float iv = inv_gam;
                        const float s0 = -cb[0].y * fmaf(db[0], iv, av[0]);
                        iv *= cb[0].z;
                        const float s1 = -cb[1].y * (fmaf(db[1], iv, av[1]) + s0 * g0.x);
                        iv *= cb[1].z;
                        const float s2 = -cb[2].y * (fmaf(db[2], iv, av[2]) + fmaf(s1, g0.w, s0 * g0.y));
                        iv *= cb[2].z;
                        const float s3 =
                            -cb[3].y * (fmaf(db[3], iv, av[3]) + fmaf(s2, g1.y, fmaf(s1, g1.x, s0 * g0.z)));
                        iv *= cb[3].z;
                        inv_gam = iv;
                        gam *= (cb[0].x * cb[1].x) * (cb[2].x * cb[3].x);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            gh[e] = fmaf(s3, kb[3][e],
                                         fmaf(s2, kb[2][e], fmaf(s1, kb[1][e], fmaf(s0, kb[0][e], gh[e]))));
                        if (gam < 1e-20f) fold();
                    }
                    for (; j < Lt; ++j) apply1(j, false);
                    if (gam < 1e-20f) fold();
                }
            }
            if (last) {
                // G = gam * ghat: fp32 rows for the eta / alpha rows, and the update's B operand
                // in three bf16 pieces (G - I when the chunk retains at least half of the state)
                const bool use_delta = gam >= 0.5f;
                float gv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) gv[e] = gam * gh[e];
                float4 *gd = reinterpret_cast<float4 *>(Gf + grow * GFS + 16 * gq);
#pragma unroll
                for (int e = 0; e < 4; ++e) gd[e] = make_float4(gv[4 * e], gv[4 * e + 1], gv[4 * e + 2], gv[4 * e + 3]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float v8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        v8[i] = gv[8 * hh + i] - ((use_delta && 16 * gq + 8 * hh + i == grow) ? 1.0f : 0.0f);
                    store_split8(sG + (grow >> 3) * G_KSTR + (2 * gq + hh) * G_NSTR + (grow & 7) * 16,
                                 8 * G_NSTR, v8);
                }
                if (tid == 0) *delta_form = use_delta ? 1 : 0;
                fence_async_smem();
                tc_before();
                __syncthreads();  // G and its fp32 rows written
                tc_after();
                // ---- MMA 3 (chunk end): every d x d memory <- M_b G (Eq. (46)): two M = 128 tiles
                // (rows 16..143: k, v memories; 144..271: q, m), per K step one MMA per piece of
                // M_b against the pieces of G stacked along N:
                //   cols [0,64): a1 b1 + a2 b1 + a3 b1,  [64,128): a1 b2 + a2 b2,  [128,192): a1 b3.
                if (issuer && !*abort_flag) {
                    const uint64_t db = sdesc(smem_u32(sG), G_KSTR, G_NSTR);
#pragma unroll
                    for (int tl = 0; tl < 2; ++tl) {
                        const uint64_t da = sdesc(smem_u32(sS) + (ROW_MEM / 8 + 16 * tl) * SBO, LBO, SBO);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t ka = ks * 2 * LBO, kb = ks * 2 * G_KSTR;
#pragma unroll
                            for (int pc = 0; pc < 3; ++pc)
                                mma(tbase + COL_UPD + UPD_TILE * tl, dadd(da, pc * S_PIECE + ka), dadd(db, kb),
                                    idesc_bf16(128, 3 * D - D * pc, true), (ks | pc) != 0);
                        }
                    }
                    mma_commit(mb_upd);
                }
            }
            // readout epilogue: lambda_r y added at the token's pixel (Eq. (26)); warp 0 holds
            // channels 0..31 of its lane's token, warp 4 channels 32..63
            if (tokw) {
                wt.wait(mb_ro, ph_ro);
                tc_after();
                const int half = warp >> 2;
                float y[32];
                tmem_ld32(tbase + lrow + COL_RO + 32 * half, y);
                const int pix = rowr ? Lidx * W + p : p * W + Lidx;
                if (valid && VH_IN(a.stats, ((size_t)b * H * W + pix) * Cc + (size_t)h * D + 32 * half, 32,
                                   map_elems(a))) {
                    float *dst = ob + (size_t)pix * Cc + 32 * half;
                    const float *lm = lam ? lam + 32 * half : nullptr;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float4 v4 = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
                        if (lm) {
                            v4.x *= lm[4 * e]; v4.y *= lm[4 * e + 1];
                            v4.z *= lm[4 * e + 2]; v4.w *= lm[4 * e + 3];
                        }
                        n_nf += !isfinite(v4.x) + !isfinite(v4.y) + !isfinite(v4.z) + !isfinite(v4.w);
                        red_add_v4(dst + 4 * e, v4);
                    }
                }
            }
            ph_ro ^= 1;
            if (last) {
                // the 1 x d eta and alpha rows on CUDA cores, in fp32 (lane = column pair);
                // their operand rows are read by no pending MMA
                if (warp == 1) eta_alpha_rows();
                wt.wait(mb_upd, ph_upd);
                ph_upd ^= 1;
                tc_after();
                resplit();
            }
            }  // recurrence form
            fence_async_smem();
            tc_before();
            __syncthreads();  // end of sub-tile: operands rewritten, TMEM consumed
            tc_after();
        }
    }

    if (a.mem_out && mo_ok && tid < 2 * D) {
        float *mo = a.mem_out + (((size_t)b * 4 + r) * a.nh + h) * SZ;
        mo[4 * D * D + tid] = Sea[tid];
    }
    if (a.stats) {
        unsigned long long *st = a.stats;
        unsigned cs = n_spec, ci = n_inj, cn = n_nf;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            cs += __shfl_xor_sync(0xffffffffu, cs, o);
            ci += __shfl_xor_sync(0xffffffffu, ci, o);
            cn += __shfl_xor_sync(0xffffffffu, cn, o);
        }
        if (lane == 0) {
            if (cs) atomicAdd(st + VH_STAT_SPEC_ACTIVE, (unsigned long long)cs);
            if (ci) atomicAdd(st + VH_STAT_INJ_RATIO_GT1, (unsigned long long)ci);
            if (cn) atomicAdd(st + VH_STAT_NONFINITE, (unsigned long long)cn);
        }
        if (tid == 0) atomicAdd(st + VH_STAT_TOKENS, (unsigned long long)H * W);
    }
    // A CTA that gave up lets its own asynchronous work land (bounded) before TMEM is freed
    // and its shared memory released: every MMA it issued (one more commit tracks them all)
    // and the x copy in flight.
    if (issuer && *abort_flag) {
        mma_commit(mb_drain);
        drain_wait(mb_drain, 0);
        if (nx_obs < nx_iss) drain_wait(mb_x, (nx_iss - 1) & 1);
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                     "r"(TMEM_COLS)
                     : "memory");
}

// 4-D view of x [B][H][W][Cc] bf16 with dims (channel, position along the line, line,
// image); a box is 8 channels x TT positions.
bool make_map64(CUtensorMap *m, const void *x, int B, int H, int W, int Cc, bool rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t e = 2;
    cuuint64_t dims[4], strides[3];
    dims[0] = (cuuint64_t)Cc;
    dims[1] = (cuuint64_t)(rows ? W : H);
    dims[2] = (cuuint64_t)(rows ? H : W);
    dims[3] = (cuuint64_t)B;
    strides[0] = rows ? (cuuint64_t)Cc * e : (cuuint64_t)W * Cc * e;
    strides[1] = rows ? (cuuint64_t)W * Cc * e : (cuuint64_t)Cc * e;
    strides[2] = (cuuint64_t)H * W * Cc * e;
    const cuuint32_t box[4] = {8, (cuuint32_t)TT, 1, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc64

// Tensor-core path for head_dim 64: bf16 x, row/column-aligned chunks, the method as
// defined (no control flags, no outer queries, no backward records).  Sets *handled =
// false (and returns success) for any other call.  `gain` (VH_IMPL_*) picks the gain form:
// VH_IMPL_TC_WY the WY form (cudaErrorNotSupported unless every chunk fits one sub-tile),
// VH_IMPL_TC_RECUR the blocked recurrence, otherwise WY where it applies.
cudaError_t launch_scan_tc64(const ScanArgs &a, int d, bool bf16, cudaStream_t st, bool *handled,
                             int gain)
{
    *handled = false;
    const bool aligned = a.chunk == 0 || (a.chunk == a.W && a.chunk == a.H);
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (d != tc64::D || !bf16 || !aligned || (a.Cc % 8) != 0 || a.control_flags || a.ckpt ||
        a.qhat || !a.out || !a16(a.mem0) || (a.mem_out && !a16(a.mem_out)))
        return cudaSuccess;
    CUtensorMap mr, mc;
    if (!tc64::make_map64(&mr, a.x, a.B, a.H, a.W, a.Cc, true) ||
        !tc64::make_map64(&mc, a.x, a.B, a.H, a.W, a.Cc, false))
        return cudaErrorInvalidValue;
    static int attr_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(tc64::scan_tc64_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc64::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc64::scan_tc64_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc64::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const unsigned grid = (unsigned)(a.B * a.ndirs * a.nh);
    // the WY form where every chunk fits one sub-tile (both orientations), else the recurrence
    const bool wy_ok = a.H <= tc64::TT && a.W <= tc64::TT;
    if ((gain == VH_IMPL_TC_WY && !wy_ok) || gain == VH_IMPL_TC_PIPE) return cudaErrorNotSupported;
    if (wy_ok && gain != VH_IMPL_TC_RECUR)
        tc64::scan_tc64_kernel<true><<<grid, tc64::NT, tc64::SMEM_BYTES, st>>>(a, mr, mc);
    else
        tc64::scan_tc64_kernel<false><<<grid, tc64::NT, tc64::SMEM_BYTES, st>>>(a, mr, mc);
    *handled = true;
    return cudaGetLastError();
}

}  // namespace vh
