// vh_scan_tc.cu -- tensor-core (tcgen05 + TMA) kernel of the four-direction
// VisionHOPE memory scan for head_dim 32, bf16 feature maps and chunks aligned
// with rows/columns ("VisionHOPE: Visual Backbones as Self-Modifying Learning
// Systems", Sec. 2.3 Eq. (25)).
//
// One CTA (one warpgroup, 128 threads) owns one scan (image b, route r, head h).
// The six memories stay on chip for the whole scan: the fp32 state leaves the
// update MMA in TMEM and is kept in shared memory
// cut into three bf16 pieces (s = s1 + s2 + s3 exactly to 2^-27 relative),
// the operand form of the tensor core; products of two such operands take the
// six cross terms of total order <= 2.  Per 64-token sub-tile of a chunk (a chunk is one image row or
// column):
//   TMA    four 16-byte x 64-token boxes of the NHWC map land as the canonical
//          K-major no-swizzle operand (core matrices 8 tokens x 16 bytes);
//          reverse routes load the same boxes and index them backwards.
//   MMA 1  generation, Eq. (15): [k_raw v q_raw | s_eta s_alpha] = x (s1+s2+s3)^T
//          (x is exact in bf16, so three passes give fp32-accurate products).
//   SIMT   one thread per token (TMEM lane = token): stabilised L2 norms of k
//          and q (App. C.1, App. B.5), delta = k - v, Eq. (53) gates, Def. 1
//          step control with the App. B.3 safeguards.
//   MMA 2  readout, Eq. (16): y = q M^m_b^T (six split cross terms);
//          the epilogue adds lambda_r y at the token's pixel (Eq. (26)).
//   SIMT   shared gain G_t = alpha_t G_{t-1} - eta_t (G_{t-1} k_t + delta_t) k_t^T
//          (Prop. 2, Eq. (46)), one lane per gain row, in the scaled form
//          G = gamma * Ghat so each token costs one FMA per element.
//   MMA 3  at the chunk end, every memory <- M_b G (Eq. (46)) for the k, v, q and
//          content memories (M = 128 rows) as M_b + M_b (G - I): the MMA forms the
//          increment and the epilogue adds M_b in fp32, so the tensor core's
//          accumulation error is relative to the per-chunk change; the 1 x d eta
//          and alpha rows are advanced on CUDA cores in fp32.
// Every mbarrier wait is bounded (clock64); on expiry the kernel records
// VH_STAT_TIMEOUT (when stats are given), stops issuing asynchronous work and
// runs to its end without blocking.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "vh_tc_ptx.cuh"

namespace vh {
namespace tc {

constexpr int D = 32;        // head dim of this kernel
constexpr int TT = 64;       // tokens per sub-tile (M of the generation/readout MMAs)
constexpr int NT = 128;      // one warpgroup
constexpr int ROW_B = D * 2;         // bytes of one bf16 operand row (64)
constexpr int SBO_K32 = 8 * ROW_B;   // 8-row group stride of a K = 32 operand (512 B)
constexpr int LBO_K32 = 128;         // K-direction core-matrix stride of a K = 32 operand
constexpr int LBO_X = TT * 16;       // K-direction stride of the TMA-loaded x tile (1 KB)
constexpr int SBO_X = 128;
constexpr int KS = D + 4;            // fp32 row stride of the key / delta tiles (padded so the
                                     // per-token row stores of eight lanes hit distinct banks)
// One bf16 piece of the state operand, 144 rows: eta, alpha, 14 zero rows, then the k, v,
// q and content memories (32 rows each).  The generation reads rows 0..111 as one B
// operand, the update rows 16..143 as one A operand, the readout rows 112..143.
constexpr int ROW_ETA = 0, ROW_MEM = 16, S_ROWS = ROW_MEM + 4 * D;
constexpr int S_PIECE = S_ROWS / 8 * SBO_K32;
constexpr int Q_PIECE = TT * ROW_B;
// VisionHOPE-exact readout: the outer queries' three pieces arrive by TMA, one box per
// 8-channel group holding [piece][64 tokens][16 bytes]: K-group stride 3 KB, 8-row stride
// 128 B, piece stride 1 KB (same 12 KB region as the in-kernel query pieces).
constexpr int QX_LBO = 3 * TT * 16, QX_PIECE = TT * 16;
constexpr int G_PIECE = D * ROW_B;
// The gain as the update's B operand is MN-major (N contiguous): element (n, k) of piece p
// at (4p + n/8) * 128 + (k/8) * G_KSTR + (k%8) * 16 + (n%8) * 2, so the three pieces stack
// along N (rows n of piece p are operand rows 32p + n) and a gain row's 16 consecutive
// columns are two 16-byte runs.
constexpr int G_NSTR = 128, G_KSTR = 3 * (D / 8) * G_NSTR;
static_assert(D / 8 * G_KSTR == 3 * G_PIECE, "gain operand size");

// The M = 128 generation and readout MMAs address their operand 1 KB (x) or 4 KB (each
// query piece) below the data, so a readable region precedes both.
constexpr int OFF_S = 0;                                      // 3 pieces of the state operand
constexpr int OFF_X = (3 * S_PIECE + 1023) / 1024 * 1024;     // TT x D bf16 (4 boxes of 1 KB)
constexpr int OFF_Q = OFF_X + TT * D * 2;                     // 3 pieces x TT x D bf16 queries
constexpr int OFF_G = OFF_Q + 3 * Q_PIECE;        // 3 pieces x D x D bf16 gain (B operand)
constexpr int GFS = D + 4;                        // fp32 row stride of the gain rows
constexpr int OFF_GF = OFF_G + 3 * G_PIECE;       // D x GFS fp32 gain rows
constexpr int OFF_KF = OFF_GF + D * GFS * 4;      // TT x KS fp32 keys, route order
constexpr int OFF_DL = OFF_KF + TT * KS * 4;      // TT x KS fp32 delta, route order
constexpr int OFF_SEA = OFF_DL + TT * KS * 4;     // 2 x D fp32 eta / alpha rows of the state
constexpr int OFF_SC = OFF_SEA + 2 * D * 4;       // TT x {alpha, eta/alpha, 1/alpha, eta}
constexpr int NB = 4;                             // tokens per block of the gain recurrence
static_assert(NB == 4 && TT % 16 == 0, "the block solve is written out for four tokens");
constexpr int OFF_GT = OFF_SC + TT * 16;          // per block: k_a . k_b, a < b (6 of 8 slots)
constexpr int OFF_BAR = OFF_GT + TT / NB * 8 * 4; // mbarriers, TMEM base, flags
constexpr int SMEM_BYTES = OFF_BAR + 128;
static_assert(SMEM_BYTES <= 75 * 1024, "three CTAs per SM");
// Pipelined form for lines of several sub-tiles: a second set of the key, delta, scalar and
// Gram tiles past the default layout, so the token pair prepares sub-tile s + 1 in one set
// while the gain pair runs sub-tile s from the other.  Launched with this larger size (two
// CTAs per SM).
constexpr int OFF_KF2 = (SMEM_BYTES + 15) / 16 * 16;
constexpr int OFF_DL2 = OFF_KF2 + TT * KS * 4;
constexpr int OFF_SC2 = OFF_DL2 + TT * KS * 4;
constexpr int OFF_GT2 = OFF_SC2 + TT * 16;
constexpr int SMEM_PIPE = OFF_GT2 + TT / NB * 8 * 4;
static_assert(SMEM_PIPE <= 113 * 1024, "two CTAs per SM");
// Intra-chunk readout (ablation), past the default layout: fp32 normalised queries in
// route order, and per block of NB tokens the cross entries k_a . q_b, a < b (6 of 8).
// Launched with this larger size, the kernel runs two CTAs per SM.
constexpr int OFF_QF = (SMEM_BYTES + 15) / 16 * 16;
constexpr int OFF_CQ = OFF_QF + TT * KS * 4;
constexpr int SMEM_INTRA = OFF_CQ + TT / NB * 8 * 4;
// WY form of the shared gain (chunks of at most one sub-tile, the method as defined):
// the keys' Gram matrix on the tensor core, the chunk's triangular system solved on one
// warp, and G assembled on the tensor core from the solution.  The update then reads G's
// pieces K-major (row n = column of G), pieces G_PIECE apart.
//  * key pieces: the keys of the sub-tile in three bf16 pieces, element (token j, column b,
//    piece p) at (j/8) KP_GSTR + (4p + b/8) 128 + (j%8) 16 + (b%8) 2.  Read K-major (rows j,
//    K = b; piece p at +512 B) by the Gram MMA and MN-major (N = 32p + b stacks the pieces,
//    K = j) by the assembly MMA.
//  * W' pieces: the assembly's B operand, rows = gain rows a, K = tokens (64, zero past the
//    chunk), element (a, j) at (a/8) WP_SBO + (j/8) 128 + (a%8) 16 + (j%8) 2, pieces WP_PIECE
//    apart (so N = 32p + a stacks them).
//  * packed coefficients: row i holds c(i, j) for j = j0(i) .. Lp - 1, j0(i) = 4 floor((i+1)/4)
//    (16-byte aligned rows; entries j <= i are zero).
constexpr int KP_GSTR = 3 * (D / 8) * 128;
constexpr int KP_BYTES = TT / 8 * KP_GSTR;
constexpr int WP_SBO = (TT / 8) * 128;
constexpr int WP_PIECE = D / 8 * WP_SBO;
// The recurrence layout above; the WY layout moves the key and delta tiles behind the key
// pieces, which overlay the gain operand and rows (those are written only after the
// assembly has read the keys).  The coefficients overlay the key tile once the shifted
// deltas are formed, and W' overlays both tiles once the solve has read them.
template <bool kWY> struct Lay {
    static constexpr int KF = OFF_KF, DL = OFF_DL, SEA = OFF_SEA, SC = OFF_SC, BAR = OFF_BAR;
    static constexpr int BYTES = SMEM_BYTES;
};
template <> struct Lay<true> {
    static constexpr int KP = OFF_G;
    static constexpr int KF = KP + KP_BYTES, DL = KF + TT * KS * 4, SEA = DL + TT * KS * 4;
    static constexpr int SC = SEA + 2 * D * 4, BAR = SC + TT * 16, BYTES = BAR + 128;
    static constexpr int CP = KF, WP = KF;
};
static_assert(Lay<true>::BYTES <= 75 * 1024, "three CTAs per SM");
static_assert(OFF_GF + D * GFS * 4 <= Lay<true>::KF, "gain rows inside the key pieces");
static_assert(Lay<true>::WP + 3 * WP_PIECE <= Lay<true>::SEA, "W' inside the key and delta tiles");
static_assert(Lay<true>::KP - 8 * KP_GSTR >= 0 && Lay<true>::KP + 16 * KP_GSTR <= Lay<true>::BYTES,
              "Gram operand rows 0..127 stay in shared memory");
static_assert(Lay<true>::KP - 1024 >= 0 && Lay<true>::KP + KP_BYTES + 2048 <= Lay<true>::BYTES,
              "assembly operand rows 0..127 (key columns, MN-major) stay in shared memory");
static_assert((TT * TT / 2 + 2 * TT) * 4 <= TT * KS * 4, "packed coefficients inside the key tile");
constexpr uint32_t TMEM_COLS = 128;
// TMEM columns (all M = 128): the generation [s_eta s_alpha 0.. | k_raw | v | q_raw] at
// 0..111 (COL_K, COL_V, COL_QR relative), then the readout over the consumed gate and
// key columns and the update's three 32-column blocks over the rest.
constexpr int COL_GEN = 0, COL_K = ROW_MEM, COL_V = ROW_MEM + D, COL_QR = ROW_MEM + 2 * D;
constexpr int COL_RO = 0, COL_UPD = 32;
// WY form: the Gram matrix over the consumed generation columns, the readout beside it,
// the assembly's three column blocks over both once they are read.
constexpr int COL_GRAM = 0, COL_RO_WY = 64, COL_ASM = 0;
static_assert(OFF_X >= LBO_X && OFF_Q >= 8 * SBO_K32, "operand rows 0..63 stay in shared memory");
static_assert(OFF_Q + 4 * Q_PIECE <= OFF_BAR, "operand rows 64..127 stay in shared memory");

// ------------------------------------------------- kernel-specific helpers

// Record of route token t of this CTA's scan (backward support).
__device__ __forceinline__ float *rec_at(const ScanArgs &a, int t)
{
    return a.rec + (size_t)blockIdx.x * a.rec_stride + (size_t)t * token_rec_floats(D);
}

// k_raw (32 columns at +COL_K), v (32 at +COL_V) and s_eta, s_alpha (2 at +0) of this
// thread's lane, with a single wait.
__device__ __forceinline__ void tmem_ld_kvs(uint32_t ta, float (&k)[32], float (&v)[32], float &se,
                                            float &sa)
{
    uint32_t r[32], q[32], s0, s1;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,"
        "%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%67];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%64,%65}, [%68];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
          "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]),
          "=r"(q[14]), "=r"(q[15]), "=r"(q[16]), "=r"(q[17]), "=r"(q[18]), "=r"(q[19]),
          "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]), "=r"(q[24]), "=r"(q[25]),
          "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31]),
          "=r"(s0), "=r"(s1)
        : "r"(ta + COL_K), "r"(ta + COL_V), "r"(ta)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        k[i] = __uint_as_float(r[i]);
        v[i] = __uint_as_float(q[i]);
    }
    se = __uint_as_float(s0);
    sa = __uint_as_float(s1);
}

// Byte offset of row `row`, K-group g (8 elements) in a K = 32 K-major operand.
__device__ __forceinline__ int op_off(int row, int g)
{
    return (row >> 3) * SBO_K32 + g * LBO_K32 + (row & 7) * 16;
}

// ------------------------------------------------------------------ kernel

// Issue the six cross terms (a_i, b_j), i + j <= 2 (pieces counted from 0), of two
// three-piece K = 32 operands into one accumulator: the product of the 24-bit
// splits up to terms below 2^-24 relative.
template <uint32_t A_STRIDE, uint32_t B_STRIDE>
__device__ __forceinline__ void mma_split6(uint32_t dt, uint32_t a0, uint32_t b0, uint32_t idesc)
{
    constexpr int pa[6] = {0, 0, 1, 0, 2, 1};
    constexpr int pb[6] = {0, 1, 0, 2, 0, 1};
    const uint64_t da = sdesc(a0, LBO_K32, SBO_K32), db = sdesc(b0, LBO_K32, SBO_K32);
#pragma unroll
    for (int t = 0; t < 6; ++t)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
            mma(dt, dadd(da, pa[t] * A_STRIDE + ks * 2 * LBO_K32),
                dadd(db, pb[t] * B_STRIDE + ks * 2 * LBO_K32), idesc, (t | ks) != 0);
}


// ---------------------------------------------------------------- WY form

// Start of row i of the packed coefficients (16-byte aligned), and its offset for a
// system of size lp: sum over earlier rows of lp - j0(r).
__host__ __device__ constexpr int wy_j0(int i) { return 4 * ((i + 1) / 4); }
__host__ __device__ constexpr int wy_off(int lp, int i)
{
    // sum_{m=1..i} floor(m/4) = 2 q (q - 1) + q (s + 1) for i = 4q + s
    return i * lp - 4 * (2 * (i / 4) * (i / 4 - 1) + (i / 4) * (i % 4 + 1));
}

// The chunk's triangular system for gain row a (lane = a), with the shared gain written as
//   G = gamma_L I + sum_j sigma_j w_j k_j^T,   w_j = -eta_j z_j,
//   z_j = G_{j-1} k_j + delta_j = r_j + sum_{i<j} c(i, j) w_i,
//   r_j = gamma_{j-1} k_j + delta_j,  c(i, j) = (prod_{i<s<j} alpha_s) k_i . k_j,
// gamma_j = prod_{s<=j} alpha_s and sigma_j = prod_{s>j} alpha_s ("VisionHOPE", App. B.4
// Prop. 2, Eqs. (46), (49): the recurrence unrolled; every factor is a product of
// retentions, so nothing is divided).  Right-looking: w_i is final once the earlier tokens
// have been added to its accumulator; each then adds c(i, j) w_i to every later token.
// The accumulators live in registers (lp of them); the coefficients are read as 16-byte
// broadcasts.  Then W' = sigma_j w_j goes out as the assembly's A operand, three bf16 pieces.
template <int LP>
__device__ __forceinline__ void wy_solve(const float *__restrict__ dl, const float *__restrict__ cpk,
                                         const float *__restrict__ eta, const float *__restrict__ sig,
                                         unsigned char *wp, int a)
{
    float acc[LP];
#pragma unroll
    for (int j = 0; j < LP; ++j) acc[j] = dl[j * KS + a];
    float4 e4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < LP; ++i) {
        if ((i & 3) == 0) e4 = *reinterpret_cast<const float4 *>(eta + i);
        const float ei = (i & 3) == 0 ? e4.x : (i & 3) == 1 ? e4.y : (i & 3) == 2 ? e4.z : e4.w;
        const float w = -ei * acc[i];
        acc[i] = w;
        const int j0 = wy_j0(i), o = wy_off(LP, i);
#pragma unroll
        for (int j4 = j0; j4 < LP; j4 += 4) {
            const float4 cv = *reinterpret_cast<const float4 *>(cpk + o + (j4 - j0));
            if (j4 + 0 > i) acc[j4 + 0] = fmaf(cv.x, w, acc[j4 + 0]);
            if (j4 + 1 > i) acc[j4 + 1] = fmaf(cv.y, w, acc[j4 + 1]);
            if (j4 + 2 > i) acc[j4 + 2] = fmaf(cv.z, w, acc[j4 + 2]);
            if (j4 + 3 > i) acc[j4 + 3] = fmaf(cv.w, w, acc[j4 + 3]);
        }
    }
#pragma unroll
    for (int g = 0; g < TT / 8; ++g) {
        float v8[8];
        if (8 * g < LP) {
            const float4 s0 = *reinterpret_cast<const float4 *>(sig + 8 * g);
            const float4 s1 = *reinterpret_cast<const float4 *>(sig + 8 * g + 4);
            const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
            for (int u = 0; u < 8; ++u) v8[u] = (8 * g + u < LP) ? sv[u] * acc[(8 * g + u) % LP] : 0.0f;
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) v8[u] = 0.0f;
        }
        store_split8(wp + (a >> 3) * WP_SBO + g * 128 + (a & 7) * 16, WP_PIECE, v8);
    }
}

// kAbl: the ablation switches of the step control and the memories are compiled in
// (false for the method as defined, so its hot loops carry no test of them).
// kWY: the shared gain in WY form (chunks of one sub-tile, the method as defined: kAbl
// false, no outer queries); otherwise the blocked recurrence.
// kPipe: the blocked recurrence with the sub-tiles of a line pipelined across the two warp
// pairs (the method as defined, no outer queries); the same arithmetic in the same order.
template <bool kAbl, bool kWY, bool kPipe = false>
__global__ void __launch_bounds__(NT, 3)
    scan_tc_kernel(const ScanArgs a, const __grid_constant__ CUtensorMap tm_row,
                   const __grid_constant__ CUtensorMap tm_col,
                   const __grid_constant__ CUtensorMap tq_row,
                   const __grid_constant__ CUtensorMap tq_col)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    using LY = Lay<kWY>;
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

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::BAR);
    const uint32_t mb_x = smem_u32(&bars[0]), mb_gen = smem_u32(&bars[1]);
    const uint32_t mb_ro = smem_u32(&bars[2]), mb_upd = smem_u32(&bars[3]);
    const uint32_t mb_g = smem_u32(&bars[4]);
    const uint32_t mb_q = smem_u32(&bars[5]);
    const uint32_t mb_gram = smem_u32(&bars[6]), mb_asm = smem_u32(&bars[7]);
    const uint32_t mb_drain = smem_u32(sm + LY::BAR + 112);  // end of a CTA that gave up
    const bool exact = a.qhat != nullptr;  // queries from the outer projection
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + LY::BAR + 64);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + LY::BAR + 72);
    volatile int *role_slot = reinterpret_cast<volatile int *>(sm + LY::BAR + 76);
    volatile int *delta_form = reinterpret_cast<volatile int *>(sm + LY::BAR + 80);
    volatile int *vote = reinterpret_cast<volatile int *>(sm + LY::BAR + 96);  // 2 warp flags
    const Waiter wt{abort_flag, a.stats, a.wait_limit > 0 ? a.wait_limit : (1ll << 32)};

    unsigned char *sX = sm + OFF_X, *sS = sm + OFF_S, *sQ = sm + OFF_Q, *sG = sm + OFF_G;
    float *Kf = reinterpret_cast<float *>(sm + LY::KF);
    float *DLf = reinterpret_cast<float *>(sm + LY::DL);
    float *Gf = reinterpret_cast<float *>(sm + OFF_GF);
    float *Sea = reinterpret_cast<float *>(sm + LY::SEA);
    float4 *SC = reinterpret_cast<float4 *>(sm + LY::SC);
    float *GT = reinterpret_cast<float *>(sm + OFF_GT);
    // intra-chunk readout (ablation): y_t = M^m_b u_t with u_t = G_{t-1} q_t, the gain before
    // the token's own update.  The gain pair forms u_t and leaves it in the token's row of
    // the delta tile; the token pair then reads it out instead of q_t.
    const bool intra = kAbl && (a.control_flags & VH_CTRL_INTRA_READ) != 0;
    float *Qf = reinterpret_cast<float *>(sm + OFF_QF);
    float *CQ = reinterpret_cast<float *>(sm + OFF_CQ);

    // ---- set-up: barriers, TMEM, roles, first TMA, initial state
    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(mb_x, 1);
        mbar_init(mb_gen, 1);
        mbar_init(mb_ro, 1);
        mbar_init(mb_upd, 1);
        mbar_init(mb_g, 2);
        mbar_init(mb_q, 1);
        mbar_init(mb_gram, 1);
        mbar_init(mb_asm, 1);
        mbar_init(mb_drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // Co-resident CTAs hold consecutive groups of four hardware warp slots, and warp w
        // of a CTA runs on SM sub-partition w.  Alternating the gain pair between warps 0-1
        // and 2-3 by slot group spreads the serial recurrences over the sub-partitions.
        unsigned slot;
        asm volatile("mov.u32 %0, %%warpid;" : "=r"(slot));
        *role_slot = (int)((slot >> 2) & 1u);
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
    // copies issued and completions observed per TMA barrier (issuing thread); at most one
    // copy per barrier is in flight, so after an abort the drain waits for completion
    // number n_iss - 1 where n_obs < n_iss
    uint32_t nx_iss = 0, nx_obs = 0, nq_iss = 0, nq_obs = 0;
    auto wait_copy = [&](uint32_t bar, uint32_t ph, uint32_t &n_obs) {
        const bool got = wt.wait(bar, ph);
        n_obs += got;
        return got;
    };
    auto issue_x = [&](int c, int s) {
        ++nx_iss;
        mbar_expect_tx(mb_x, TT * D * 2);
#pragma unroll
        for (int q = 0; q < D / 8; ++q)
            tma_load_4d(smem_u32(sX + q * LBO_X), tm, h * D + 8 * q, box_start(s), line_of(c), b,
                        mb_x);
    };
    __syncthreads();  // barriers initialised, TMEM address and roles written
    // roles: warps 2gp, 2gp+1 run the gain recurrence.  The other pair (first warp rw) holds
    // the tokens: every generated quantity and the readout land in its TMEM lanes
    // 32 rw..32 rw+63, so it runs the per-token step (phase 1), the queries and the readout;
    // lane 0 of warp rw issues the MMAs and TMA copies, warp rw + 1 advances the eta / alpha
    // rows.
    const int gp = *role_slot;
    const int rw = 2 - 2 * gp;
    const bool gainw = (warp >> 1) == gp;
    const int ew = rw + 1;
    const bool issuer = warp == rw && lane == 0;
    const CUtensorMap *tq = rowr ? &tq_row : &tq_col;
    auto issue_q = [&](int c, int s) {
        ++nq_iss;
        mbar_expect_tx(mb_q, 3 * TT * D * 2);
#pragma unroll
        for (int q = 0; q < D / 8; ++q)
            tma_load_5d(smem_u32(sQ + q * QX_LBO), tq, h * D + 8 * q, box_start(s), line_of(c), b, 0,
                        mb_q);
    };
    // (test hook: with the first copies withheld the first wait can only give up, and the
    // kernel then issues no asynchronous work at all)
    if (issuer && !a.withhold_first_copy) {
        issue_x(0, 0);
        if (exact) issue_q(0, 0);
    }
    // checked indices (VH_DEBUG_BOUNDS builds; `true` otherwise): this scan's slices of
    // memories0, memories_out and the backward records, checked once for their whole extent
    const size_t mem_base = ((size_t)r * a.nh + h) * SZ;
    const bool mo_ok = !a.mem_out ||
                       VH_IN(a.stats, (((size_t)b * 4 + r) * a.nh + h) * SZ, SZ, (size_t)a.B * 4 * a.nh * SZ);
    const bool ck_ok = !(kAbl && a.ckpt) ||
                       VH_IN(a.stats, (size_t)blockIdx.x * a.ckpt_stride, (size_t)nlines * SZ,
                             (size_t)gridDim.x * a.ckpt_stride);
    const bool rec_ok = !(kAbl && a.rec) ||
                        VH_IN(a.stats, (size_t)blockIdx.x * a.rec_stride,
                              (size_t)H * W * token_rec_floats(D), (size_t)gridDim.x * a.rec_stride);
    {
        const float *m0 = a.mem0 + (VH_IN(a.stats, mem_base, SZ, (size_t)4 * a.nh * SZ) ? mem_base : 0);
        // memory rows 0..127 (k, v, q, m) -> operand rows 16..143: thread = row
        float v[32];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(m0 + (size_t)tid * D) + e);
            v[4 * e] = f.x; v[4 * e + 1] = f.y; v[4 * e + 2] = f.z; v[4 * e + 3] = f.w;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) store_split8(sS + op_off(ROW_MEM + tid, g), S_PIECE, v + 8 * g);
        if (kAbl && a.ckpt && ck_ok) {  // boundary state of chunk 0 (backward support)
            float4 *d4 = reinterpret_cast<float4 *>(a.ckpt + (size_t)blockIdx.x * a.ckpt_stride +
                                                    (size_t)tid * D);
#pragma unroll
            for (int e = 0; e < 8; ++e) d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            if (tid < 2 * D) a.ckpt[(size_t)blockIdx.x * a.ckpt_stride + 4 * D * D + tid] = m0[4 * D * D + tid];
        }
        // eta / alpha rows: fp32 copy and operand rows 0, 1; rows 2..15 are zero
        if (tid < 2 * D) Sea[tid] = m0[4 * D * D + tid];
        if (tid < ROW_MEM) {
            float z[8];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
#pragma unroll
                for (int e = 0; e < 8; ++e) z[e] = tid < 2 ? m0[4 * D * D + tid * D + 8 * g + e] : 0.0f;
                store_split8(sS + op_off(tid, g), S_PIECE, z);
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
    // no out (backward support: only the boundary states are wanted): no readout adds
    float *ob = (kAbl && !a.out) ? nullptr : a.out + (size_t)b * H * W * Cc + (size_t)h * D;
    unsigned n_spec = 0, n_inj = 0, n_nf = 0;
    uint32_t ph_x = 0, ph_gen = 0, ph_ro = 0, ph_upd = 0, ph_g = 0, ph_q = 0, ph_gram = 0, ph_asm = 0;

    // gain state of the gain pair: its thread t owns row t/2 of G = gam * ghat, columns
    // 16(t%2)..+15
    float gh[16];
    float gam = 1.0f, inv_gam = 1.0f;
    // without the DGD correction (ablation) the G k terms of the recurrence drop:
    // G_j = alpha G_{j-1} - eta delta k^T
    const bool no_dgd = kAbl && (a.control_flags & VH_CTRL_NO_DGD) != 0;
    // this thread's token (box row) when in the token pair: lane l of warp w holds box row
    // 32(w - rw) + l, TMEM lane 32 rw + that row
    const int jq = 32 * (warp - rw) + lane;

    // ---- the phases of one sub-tile, shared by the sequential and the pipelined loop.
    // The per-token tiles (keys, deltas, scalars, Gram entries) are passed in, so the
    // pipelined loop can alternate between two sets of them.
    auto generate = [&](int c, int s) {
        // ---- MMA 1: generation from the boundary state, Eq. (15):
        //   [s_eta s_alpha 0.. | k_raw | v | q_raw] = x (s1 + s2 + s3)^T
        // one M = 128, N = 112 MMA per piece and K step (x is exact in bf16).  The x
        // tile is A rows 32 rw..32 rw+63; the other 64 A rows read the kilobyte next to
        // the tile into TMEM lanes nobody reads.
        if (issuer) {
            tc_after();
            if (wait_copy(mb_x, ph_x, nx_obs) && !*abort_flag) {
                const uint64_t dq = sdesc(smem_u32(sX) - (rw >> 1) * LBO_X, LBO_X, SBO_X);
                const uint64_t ds = sdesc(smem_u32(sS), LBO_K32, SBO_K32);
#pragma unroll
                for (int pc = 0; pc < 3; ++pc)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma(tbase + COL_GEN, dadd(dq, ks * 2 * LBO_X),
                            dadd(ds, pc * S_PIECE + ks * 2 * LBO_K32), idesc_bf16(128, 112),
                            (pc | ks) != 0);
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
    };
    // per-token step, Eqs. (15), (19), (20), (53), on the token pair (lane = token):
    // normalise k, form delta = k - v and their squared norms, publish the token's scalars
    auto token_step = [&](float *KfT, float *DLT, float4 *SCT, bool valid, int jr, int c, int t0) {
        float kr[32], vv[32];
        float se, sa;
        tmem_ld_kvs(tbase + lrow + COL_GEN, kr, vv, se, sa);
        const float kkr = sumsq32(kr);
        const float rk = __frsqrt_rn(kkr + a.knorm_eps);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            kr[e] *= rk;            // k
            vv[e] = kr[e] - vv[e];  // delta = k - v
        }
        const float kn2 = sumsq32(kr), dd2 = sumsq32(vv);
        if (valid) {
            float4 *kd = reinterpret_cast<float4 *>(KfT + jr * KS);
            float4 *dd4 = reinterpret_cast<float4 *>(DLT + jr * KS);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                kd[e] = make_float4(kr[4 * e], kr[4 * e + 1], kr[4 * e + 2], kr[4 * e + 3]);
                dd4[e] = make_float4(vv[4 * e], vv[4 * e + 1], vv[4 * e + 2], vv[4 * e + 3]);
            }
            SCT[jr] = make_float4(se, sa, kn2, dd2);
            if (kAbl && a.rec && rec_ok) {  // token record scalars (backward support); the
                                  // vectors follow while the gain runs
                float4 *rd = reinterpret_cast<float4 *>(rec_at(a, c * Lline + t0 + jr));
                rd[3 * D / 4] = make_float4(kkr, se, sa, kn2);
                rd[3 * D / 4 + 1].x = dd2;
            }
        }
        if (intra) {
            // the normalised query for the gain pair, route order (fp32)
            float qv[32];
            if (!exact) {
                tmem_ld32(tbase + lrow + COL_GEN + COL_QR, qv);
                const float rq = __frsqrt_rn(sumsq32(qv) + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 32; ++e) qv[e] *= rq;
            } else {
                // the outer query's three pieces from its TMA tile
                wait_copy(mb_q, ph_q, nq_obs);  // (the drain reads the issuer's count)
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const unsigned char *src = sQ + g * QX_LBO + jq * 16;
                    const uint4 u1 = *reinterpret_cast<const uint4 *>(src);
                    const uint4 u2 = *reinterpret_cast<const uint4 *>(src + QX_PIECE);
                    const uint4 u3 = *reinterpret_cast<const uint4 *>(src + 2 * QX_PIECE);
                    const uint32_t *w1 = &u1.x, *w2 = &u2.x, *w3 = &u3.x;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        qv[8 * g + 2 * i] = bf16_lo(w1[i]) + (bf16_lo(w2[i]) + bf16_lo(w3[i]));
                        qv[8 * g + 2 * i + 1] = bf16_hi(w1[i]) + (bf16_hi(w2[i]) + bf16_hi(w3[i]));
                    }
                }
            }
            if (valid) {
                float4 *qd = reinterpret_cast<float4 *>(Qf + jr * KS);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    qd[e] = make_float4(qv[4 * e], qv[4 * e + 1], qv[4 * e + 2], qv[4 * e + 3]);
            }
        }
    };
    // gain pair (lane = route-ordered token): the gates and the step control
    auto gate_step = [&](float4 *SCT, int Lt) {
        // gates and step control of route-ordered token jg; the coefficients of the
        // gain recurrence replace the scalars: (alpha, eta/alpha, 1/alpha, eta) for the
        // scaled form, (alpha, 0, 0, eta) where alpha is too small to divide by
        const int jg = tid & 63;
        const bool tv = jg < Lt;
        float alpha = 1.0f;
        if (tv) {
            const float4 sc = SCT[jg];
            float eta, oma;
            gates(a, sc.x, sc.y, eta, alpha, oma);
            float eta_t;
            if (a.gate_mode == VH_GATE_FORCED_EXEC) {
                eta_t = a.forced_eta;
            } else {
                const StepOut so = step_control<kAbl>(a, eta, alpha, oma, sc.z, sc.w);
                eta_t = so.eta_tilde;
                n_spec += so.spec_active;
                n_inj += so.inj_ratio_gt1;
            }
            const bool keep = alpha >= 1e-6f;
            SCT[jg] = make_float4(alpha, keep ? __fdividef(eta_t, alpha) : 0.0f,
                                 keep ? __frcp_rn(alpha) : 0.0f, eta_t);
        }
        // tokens whose retention could underflow the scaled gain within a few steps
        const unsigned small = __ballot_sync(0xffffffffu, tv && !(alpha >= 0.01f));
        if (lane == 0) vote[warp - 2 * gp] = small != 0u;
    };
    // token pair: the Gram entries of the gain recurrence's blocks
    auto gram_step = [&](const float *KfT, float *GTT) {
        // Gram entries k_a . k_b of each block of NB route-ordered tokens.  This
        // warp's tokens are the 32 consecutive route rows from R0 (route order runs
        // with the box rows forwards, against them backwards), eight whole blocks:
        // pair i of block q goes to lane 6q + i (mod 32).
        const int R0 = rev ? TT - 32 - 32 * (warp - rw) : 32 * (warp - rw);
#pragma unroll
        for (int pr = lane; pr < 48; pr += 32) {
            const int q = pr / 6, pi = pr - 6 * q;
            const int ia = pi < 3 ? 0 : (pi < 5 ? 1 : 2);
            const int ib = pi < 3 ? pi + 1 : (pi < 5 ? pi - 1 : 3);
            const float4 *ka = reinterpret_cast<const float4 *>(KfT + (R0 + NB * q + ia) * KS);
            const float4 *kb = reinterpret_cast<const float4 *>(KfT + (R0 + NB * q + ib) * KS);
            float g4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 fa = ka[e], fb = kb[e];
                g4[0] = fmaf(fa.x, fb.x, g4[0]);
                g4[1] = fmaf(fa.y, fb.y, g4[1]);
                g4[2] = fmaf(fa.z, fb.z, g4[2]);
                g4[3] = fmaf(fa.w, fb.w, g4[3]);
            }
            GTT[(R0 / NB + q) * 8 + pi] = (g4[0] + g4[1]) + (g4[2] + g4[3]);
            if (intra) {  // and k_a . q_b for the intra-chunk readout
                const float4 *qb = reinterpret_cast<const float4 *>(Qf + (R0 + NB * q + ib) * KS);
#pragma unroll
                for (int e = 0; e < 4; ++e) g4[e] = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 fa = ka[e], fb = qb[e];
                    g4[0] = fmaf(fa.x, fb.x, g4[0]);
                    g4[1] = fmaf(fa.y, fb.y, g4[1]);
                    g4[2] = fmaf(fa.z, fb.z, g4[2]);
                    g4[3] = fmaf(fa.w, fb.w, g4[3]);
                }
                CQ[(R0 / NB + q) * 8 + pi] = (g4[0] + g4[1]) + (g4[2] + g4[3]);
            }
        }
    };
    // gain pair: the shared gain over one sub-tile (first: the chunk's first; last: write G)
    auto gain_step = [&](const float *KfT, float *DLT, const float4 *SCT, const float *GTT, int Lt,
                         bool first, bool last) {
        // ---- shared gain over this sub-tile's tokens, in route order, on the gain
        // pair: its thread t owns row t/2 of G and columns 16(t%2)..16(t%2)+15 (one
        // shuffle per token).  G = gam * ghat with
        //   ghat <- ghat - (eta/alpha) (ghat k + delta / gam) k^T,  gam <- alpha gam,
        // a pure scaling of G_j = alpha G_{j-1} - eta (G_{j-1} k + delta) k^T.  When
        // every alpha of the sub-tile is >= 0.01 the scale is folded back every eight
        // tokens (it cannot underflow sooner); otherwise every token is checked, and a
        // token with alpha < 1e-6 is applied to G directly with the scale folded in.
        const int grow = (tid & 63) >> 1, gq = tid & 1;
        if (first) {
#pragma unroll
            for (int e = 0; e < 16; ++e) gh[e] = (16 * gq + e == grow) ? 1.0f : 0.0f;
            gam = 1.0f;
            inv_gam = 1.0f;
        }
        const bool careful = (vote[0] | vote[1]) != 0;
        // operands of token j (key half, coefficients, delta entry); the next token's
        // are loaded before the current one is applied, off the serial chain
        struct Tok {
            float k[16];
            float4 c;
            float d;
        };
        auto load = [&](int j, Tok &t) {
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(KfT + j * KS + 16 * gq + e);
                t.k[e] = f.x; t.k[e + 1] = f.y; t.k[e + 2] = f.z; t.k[e + 3] = f.w;
            }
            t.c = SCT[j];
            t.d = DLT[j * KS + grow];
        };
        auto fold = [&]() {
#pragma unroll
            for (int e = 0; e < 16; ++e) gh[e] *= gam;
            gam = 1.0f;
            inv_gam = 1.0f;
        };
        // intra-chunk readout: u_j = gam (ghat . q_j) before token j's update, left
        // in the token's delta slot (read by this row's two lanes only, both done)
        auto read_u = [&](int j) {
            const float4 *qp = reinterpret_cast<const float4 *>(Qf + j * KS + 16 * gq);
            float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 f = qp[e];
                p0 = fmaf(gh[4 * e], f.x, p0);
                p1 = fmaf(gh[4 * e + 1], f.y, p1);
                p0 = fmaf(gh[4 * e + 2], f.z, p0);
                p1 = fmaf(gh[4 * e + 3], f.w, p1);
            }
            float u = p0 + p1;
            u += __shfl_xor_sync(0xffffffffu, u, 1);
            __syncwarp();
            if (gq == 0) DLT[j * KS + grow] = gam * u;
        };
        auto apply = [&](const Tok &t, bool chk, int j) {
            if (intra) read_u(j);
            float p4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) p4[e] = gh[e] * t.k[e];
#pragma unroll
            for (int e = 4; e < 16; ++e) p4[e & 3] = fmaf(gh[e], t.k[e], p4[e & 3]);
            float dot = (p4[0] + p4[1]) + (p4[2] + p4[3]);
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            if (no_dgd) dot = 0.0f;
            if (!chk || t.c.z != 0.0f) {
                const float sc = -t.c.y * fmaf(t.d, inv_gam, dot);
#pragma unroll
                for (int e = 0; e < 16; ++e) gh[e] = fmaf(sc, t.k[e], gh[e]);
                gam *= t.c.x;
                inv_gam *= t.c.z;
                if (chk && gam < 1e-20f) fold();
            } else {  // G_j = alpha G_{j-1} - eta (G_{j-1} k + delta) k^T, unscaled
                const float sc = -t.c.w * fmaf(gam, dot, t.d);
                const float ag = t.c.x * gam;
#pragma unroll
                for (int e = 0; e < 16; ++e) gh[e] = fmaf(sc, t.k[e], ag * gh[e]);
                gam = 1.0f;
                inv_gam = 1.0f;
            }
        };
        // rows Lt..TT-1 of the tiles hold stale values: a prefetch past the last token
        // reads one and never applies it
        if (careful) {
            Tok ta, tb;
            load(0, ta);
            for (int j = 0; j < Lt; j += 2) {
                load(min(j + 1, TT - 1), tb);
                apply(ta, true, j);
                if (j + 1 >= Lt) break;
                load(min(j + 2, TT - 1), ta);
                apply(tb, true, j + 1);
            }
        } else {
            // blocks of NB tokens: with a = ghat_0 . k_j for the block's starting ghat,
            //   ghat_{j-1} . k_j = a_j + sum_{i<j in block} sc_i (k_i . k_j),
            // so the NB dot products are independent, the serial part is an NB-step
            // scalar solve, and ghat takes one rank-NB update.
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
                            *reinterpret_cast<const float4 *>(KfT + (j + t) * KS + 16 * gq + e);
                        kb[t][e] = f.x; kb[t][e + 1] = f.y; kb[t][e + 2] = f.z; kb[t][e + 3] = f.w;
                    }
                    cb[t] = SCT[j + t];
                    db[t] = DLT[(j + t) * KS + grow];
                }
                float4 g0 = *reinterpret_cast<const float4 *>(GTT + (j / NB) * 8);
                float2 g1 = *reinterpret_cast<const float2 *>(GTT + (j / NB) * 8 + 4);
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
                // intra-chunk readout: ghat_0 . q_t for the block's tokens
                float aq[NB];
                if (intra) {
#pragma unroll
                    for (int t = 0; t < NB; ++t) {
                        const float4 *qp = reinterpret_cast<const float4 *>(Qf + (j + t) * KS + 16 * gq);
                        float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float4 f = qp[e];
                            p0 = fmaf(gh[4 * e], f.x, p0);
                            p1 = fmaf(gh[4 * e + 1], f.y, p1);
                            p0 = fmaf(gh[4 * e + 2], f.z, p0);
                            p1 = fmaf(gh[4 * e + 3], f.w, p1);
                        }
                        aq[t] = p0 + p1;
                    }
#pragma unroll
                    for (int t = 0; t < NB; ++t) aq[t] += __shfl_xor_sync(0xffffffffu, aq[t], 1);
                }
                if (no_dgd) {
#pragma unroll
                    for (int t = 0; t < NB; ++t) av[t] = 0.0f;
                    g0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    g1 = make_float2(0.0f, 0.0f);
                }
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
                if (intra) {
                    // ghat_{t-1} . q_t = ghat_0 . q_t + sum_{i<t} s_i (k_i . q_t), and
                    // gam_{t-1} = gam_0 alpha_0 .. alpha_{t-1}
                    const float4 c0 = *reinterpret_cast<const float4 *>(CQ + (j / NB) * 8);
                    const float2 c1 = *reinterpret_cast<const float2 *>(CQ + (j / NB) * 8 + 4);
                    float g = gam;
                    const float u0 = g * aq[0];
                    g *= cb[0].x;
                    const float u1 = g * fmaf(s0, c0.x, aq[1]);
                    g *= cb[1].x;
                    const float u2 = g * fmaf(s1, c0.w, fmaf(s0, c0.y, aq[2]));
                    g *= cb[2].x;
                    const float u3 = g * fmaf(s2, c1.y, fmaf(s1, c1.x, fmaf(s0, c0.z, aq[3])));
                    __syncwarp();
                    if (gq == 0) {
                        DLT[j * KS + grow] = u0;
                        DLT[(j + 1) * KS + grow] = u1;
                        DLT[(j + 2) * KS + grow] = u2;
                        DLT[(j + 3) * KS + grow] = u3;
                    }
                }
                gam *= (cb[0].x * cb[1].x) * (cb[2].x * cb[3].x);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    gh[e] = fmaf(s3, kb[3][e],
                                 fmaf(s2, kb[2][e], fmaf(s1, kb[1][e], fmaf(s0, kb[0][e], gh[e]))));
                if (gam < 1e-20f) fold();
            }
            for (; j < Lt; ++j) {
                Tok t;
                load(j, t);
                apply(t, false, j);
            }
            if (gam < 1e-20f) fold();
        }
        if (intra) {
            __threadfence_block();
            named_arrive(2, NT);  // u of every token of the sub-tile written
        }
        if (last) {
            // G = gam * ghat: fp32 rows for the eta / alpha rows, and the update's B
            // operand in three bf16 pieces (MN-major: this lane's 16 columns of its
            // row are two 16-byte runs per piece).  When the chunk retains at least
            // half of the state the operand is G - I: the MMA forms only the
            // increment M_b (G - I), which the epilogue adds to M_b in fp32, so the
            // tensor core's accumulation error is relative to the change.  Otherwise
            // the state is mostly replaced and the MMA forms M_b G directly (no
            // cancellation).
            const bool use_delta = gam >= 0.5f;
            float gv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) gv[e] = gam * gh[e];
            float4 *gd = reinterpret_cast<float4 *>(Gf + grow * GFS + 16 * gq);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                gd[e] = make_float4(gv[4 * e], gv[4 * e + 1], gv[4 * e + 2], gv[4 * e + 3]);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v8[i] = gv[8 * hh + i] - ((use_delta && 16 * gq + 8 * hh + i == grow) ? 1.0f : 0.0f);
                store_split8(sG + (2 * gq + hh) * G_NSTR + (grow >> 3) * G_KSTR + (grow & 7) * 16,
                             4 * G_NSTR, v8);
            }
            if ((tid & 63) == 0) *delta_form = use_delta ? 1 : 0;
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(mb_g);  // this warp's rows of G are written
        }
    };
    // token pair, after the readout MMA: lambda_r y added at the token's pixel (Eq. (26))
    auto add_readout = [&](int p, int Lidx, bool valid) {
        float y[32];
        tmem_ld32(tbase + lrow + COL_RO, y);
        const int pix = rowr ? Lidx * W + p : p * W + Lidx;
        if (valid && (!kAbl || ob) &&
            VH_IN(a.stats, ((size_t)b * H * W + pix) * Cc + (size_t)h * D, D, map_elems(a))) {
            float *dst = ob + (size_t)pix * Cc;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float4 v4 = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
                if (lam) {
                    v4.x *= lam[4 * e]; v4.y *= lam[4 * e + 1];
                    v4.z *= lam[4 * e + 2]; v4.w *= lam[4 * e + 3];
                }
                n_nf += !isfinite(v4.x) + !isfinite(v4.y) + !isfinite(v4.z) + !isfinite(v4.w);
                red_add_v4(dst + 4 * e, v4);
            }
        }
    };
    // MMA 3 (chunk end, issuing thread): every d x d memory <- M_b G (Eq. (46)), issued as
    // soon as the gain pair has written G's pieces.  The six cross terms go in as three MMAs
    // per K step, one per piece of M_b against the pieces of G stacked along N:
    //   cols [0,32): a1 b1 + a2 b1,  [32,64): a1 b2 + a2 b2,  [64,96): a1 b3 + a3 b1,
    // summed by the epilogue.
    auto issue_update = [&]() {
        if (wt.wait(mb_g, ph_g) && !*abort_flag) {
            tc_after();
            const uint64_t da = sdesc(smem_u32(sS) + ROW_MEM / 8 * SBO_K32, LBO_K32, SBO_K32);
            const uint64_t db = sdesc(smem_u32(sG), G_KSTR, G_NSTR);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint32_t ka = ks * 2 * LBO_K32, kb = ks * 2 * G_KSTR;
                mma(tbase + COL_UPD, dadd(da, ka), dadd(db, kb), idesc_bf16(128, 96, true),
                    ks != 0);
                mma(tbase + COL_UPD, dadd(da, S_PIECE + ka), dadd(db, kb),
                    idesc_bf16(128, 64, true), 1);
                mma(tbase + COL_UPD + 2 * D, dadd(da, 2 * S_PIECE + ka), dadd(db, kb),
                    idesc_bf16(128, 32, true), 1);
            }
            mma_commit(mb_upd);
        }
    };
    // chunk end, after the barrier that follows G: the eta / alpha rows and the new state
    auto chunk_end = [&](int c) {
        // the 1 x d eta and alpha rows on CUDA cores, in fp32 (lane = column); their
        // operand rows are read by no pending MMA
        if (warp == ew && !(kAbl && (a.control_flags & VH_CTRL_FREEZE_DYN))) {
            float ne = 0.0f, na = 0.0f;
#pragma unroll 8
            for (int l = 0; l < D; ++l) {
                const float gv = Gf[l * GFS + lane];
                ne = fmaf(Sea[l], gv, ne);
                na = fmaf(Sea[D + l], gv, na);
            }
            __syncwarp();
            Sea[lane] = ne;
            Sea[D + lane] = na;
            if (kAbl && a.ckpt && ck_ok && c + 1 < nlines) {  // backward support
                float *ck = a.ckpt + (size_t)blockIdx.x * a.ckpt_stride + (size_t)(c + 1) * SZ;
                ck[4 * D * D + lane] = ne;
                ck[4 * D * D + D + lane] = na;
            }
            __nv_bfloat16 p1, p2, p3;
            const int g = lane >> 3, e = lane & 7;
            split3(ne, p1, p2, p3);
            unsigned char *d0 = sS + op_off(ROW_ETA, g) + 2 * e;
            *reinterpret_cast<__nv_bfloat16 *>(d0) = p1;
            *reinterpret_cast<__nv_bfloat16 *>(d0 + S_PIECE) = p2;
            *reinterpret_cast<__nv_bfloat16 *>(d0 + 2 * S_PIECE) = p3;
            split3(na, p1, p2, p3);
            unsigned char *d1 = sS + op_off(ROW_ETA + 1, g) + 2 * e;
            *reinterpret_cast<__nv_bfloat16 *>(d1) = p1;
            *reinterpret_cast<__nv_bfloat16 *>(d1 + S_PIECE) = p2;
            *reinterpret_cast<__nv_bfloat16 *>(d1 + 2 * S_PIECE) = p3;
        }
        wt.wait(mb_upd, ph_upd);
        ph_upd ^= 1;
        tc_after();
        // new state rows: thread = memory row (TMEM lane), the three column blocks
        // summed, re-split into the operand pieces.  In the increment form M_b is
        // recovered exactly from its three pieces (their sum rounds back to the fp32
        // value they were cut from) and added in fp32.
        float v[32], w[32];
        tmem_ld32(tbase + lrow + COL_UPD, v);
        tmem_ld32(tbase + lrow + COL_UPD + D, w);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += w[e];
        tmem_ld32(tbase + lrow + COL_UPD + 2 * D, w);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] += w[e];
        // a memory held fixed by an ablation switch keeps M_b (recovered from its
        // pieces for memories_out) and its operand rows are not rewritten
        const bool frz = frozen_row<kAbl>(a, tid, D);
        if (frz) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.0f;
        }
        const bool add_mb = frz || *delta_form != 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            unsigned char *src = sS + op_off(ROW_MEM + tid, g);
            if (add_mb) {
                const uint4 u1 = *reinterpret_cast<const uint4 *>(src);
                const uint4 u2 = *reinterpret_cast<const uint4 *>(src + S_PIECE);
                const uint4 u3 = *reinterpret_cast<const uint4 *>(src + 2 * S_PIECE);
                const uint32_t *w1 = &u1.x, *w2 = &u2.x, *w3 = &u3.x;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[8 * g + 2 * i] += (bf16_lo(w1[i]) + bf16_lo(w2[i])) + bf16_lo(w3[i]);
                    v[8 * g + 2 * i + 1] += (bf16_hi(w1[i]) + bf16_hi(w2[i])) + bf16_hi(w3[i]);
                }
            }
            if (!frz) store_split8(src, S_PIECE, v + 8 * g);
        }
        if (kAbl && a.ckpt && ck_ok && c + 1 < nlines) {  // boundary state of the next chunk
            float4 *d4 = reinterpret_cast<float4 *>(a.ckpt + (size_t)blockIdx.x * a.ckpt_stride +
                                                    (size_t)(c + 1) * SZ + (size_t)tid * D);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
        if (c == nlines - 1 && a.mem_out && mo_ok) {
            float *mo = a.mem_out + (((size_t)b * 4 + r) * a.nh + h) * SZ;
            float4 *d4 = reinterpret_cast<float4 *>(mo + (size_t)tid * D);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        }
    };

    if constexpr (kPipe) {
    // ================= pipelined sub-tiles (lines longer than one sub-tile).  Step k of a
    // chunk: the token pair reads out sub-tile k - 1 (its queries are still in TMEM), then
    // generates sub-tile k and runs its per-token step and Gram entries into tile set k % 2;
    // meanwhile the gain pair runs the gates and the shared gain of sub-tile k - 1 from set
    // (k - 1) % 2.  One barrier per step; the chunk end follows step nsub.
    static_assert(!kAbl && !kWY, "pipelined form: the method as defined, recurrence gain");
    float *const Kf2 = reinterpret_cast<float *>(sm + OFF_KF2);
    float *const DL2 = reinterpret_cast<float *>(sm + OFF_DL2);
    float4 *const SC2 = reinterpret_cast<float4 *>(sm + OFF_SC2);
    float *const GT2 = reinterpret_cast<float *>(sm + OFF_GT2);
    for (int c = 0; c < nlines; ++c) {
        const int Lidx = line_of(c);
        for (int k = 0; k <= nsub; ++k) {
            if (!gainw) {
                if (k >= 1) {
                    const int sr = k - 1;
                    const int p = box_start(sr) + jq;
                    const bool valid =
                        p >= 0 && p < Lline && VH_IN(a.stats, (rev ? Lline - 1 - p : p) - sr * TT, 1, TT);
                    // queries: q = normalize(M^q_b x), split into the readout's A operand
                    float qr[32];
                    tmem_ld32(tbase + lrow + COL_GEN + COL_QR, qr);
                    const float rq = __frsqrt_rn(sumsq32(qr) + a.knorm_eps);
#pragma unroll
                    for (int e = 0; e < 32; ++e) qr[e] *= rq;
#pragma unroll
                    for (int g = 0; g < 4; ++g) store_split8(sQ + op_off(jq, g), Q_PIECE, qr + 8 * g);
                    fence_async_smem();
                    tc_before();
                    named_sync(1, 64);
                    tc_after();
                    // MMA 2: readout y = q M^m_b^T, Eq. (16)
                    if (issuer && !*abort_flag) {
                        mma_split6<Q_PIECE, S_PIECE>(tbase + COL_RO, smem_u32(sQ) - (rw >> 1) * 8 * SBO_K32,
                                                     smem_u32(sS) + (ROW_MEM + 3 * D) / 8 * SBO_K32,
                                                     idesc_bf16(128, 32));
                        mma_commit(mb_ro);
                    }
                    wt.wait(mb_ro, ph_ro);
                    ph_ro ^= 1;
                    tc_after();
                    add_readout(p, Lidx, valid);
                    // the gain pair finishes the chunk's last sub-tile in this step
                    if (k == nsub && issuer) issue_update();
                }
                if (k < nsub) {
                    tc_before();
                    named_sync(1, 64);  // both warps' TMEM reads above done
                    tc_after();
                    const int p = box_start(k) + jq;
                    const int jr = (rev ? Lline - 1 - p : p) - k * TT;
                    const bool valid = p >= 0 && p < Lline && VH_IN(a.stats, jr, 1, TT);
                    const bool t2 = (k & 1) != 0;
                    generate(c, k);
                    token_step(t2 ? Kf2 : Kf, t2 ? DL2 : DLf, t2 ? SC2 : SC, valid, jr, c, k * TT);
                    named_sync(1, 64);  // every token's key row written
                    gram_step(t2 ? Kf2 : Kf, t2 ? GT2 : GT);
                }
            } else if (k >= 1) {
                const int sg = k - 1;
                const bool t2 = (sg & 1) != 0;
                const int Lt = min(TT, Lline - sg * TT);
                gate_step(t2 ? SC2 : SC, Lt);
                named_sync(3, 64);  // both warps' coefficients and votes written
                gain_step(t2 ? Kf2 : Kf, t2 ? DL2 : DLf, t2 ? SC2 : SC, t2 ? GT2 : GT, Lt, sg == 0, k == nsub);
            }
            tc_before();
            __syncthreads();  // end of step k: tile set (k - 1) % 2 free again
            tc_after();
        }
        ph_g ^= 1;
        chunk_end(c);
        fence_async_smem();
        tc_before();
        __syncthreads();  // end of chunk: operands rewritten, TMEM consumed
    }
    } else {
    for (int c = 0; c < nlines; ++c) {
        const int Lidx = line_of(c);
        for (int s = 0; s < nsub; ++s) {
            const int t0 = s * TT;
            const int Lt = min(TT, Lline - t0);
            const bool last = s == nsub - 1;
            const int p = box_start(s) + jq;   // position along the line (token pair)
            const int jr = (rev ? Lline - 1 - p : p) - t0;  // route-ordered index in the sub-tile
            const bool valid = !gainw && p >= 0 && p < Lline && VH_IN(a.stats, jr, 1, TT);
            generate(c, s);
            if constexpr (kWY) {
            // ================= WY form of the shared gain (one sub-tile per chunk) =========
            float *cpk = reinterpret_cast<float *>(sm + Lay<true>::CP);
            unsigned char *sKP = sm + Lay<true>::KP, *sWP = sm + Lay<true>::WP;
            float *ALP = reinterpret_cast<float *>(SC), *ETA = ALP + TT, *GPRE = ETA + TT, *SIG = GPRE + TT;
            float *gam_slot = reinterpret_cast<float *>(sm + LY::BAR + 84);
            float *scan_tot = reinterpret_cast<float *>(sm + LY::BAR + 88);
            // size of the triangular system: the chunk length where a solve is built for it,
            // else the next of 32 and 64 (tokens past the chunk contribute zero)
            const int Lp = Lt == 56 ? 56 : Lt == 28 ? 28 : Lt <= 32 ? 32 : 64;
            // ---- A. per token (token pair, lane = token): stabilised norms (App. C.1,
            // App. B.5), delta = k - v, the raw scalars, the fp32 key and delta rows and the
            // keys' operand pieces (rows past the chunk's last token are zero)
            if (!gainw) {
                float kr[32], vv[32];
                float se, sa;
                tmem_ld_kvs(tbase + lrow + COL_GEN, kr, vv, se, sa);
                const float kkr = sumsq32(kr);
                const float rk = __frsqrt_rn(kkr + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    kr[e] *= rk;
                    vv[e] = kr[e] - vv[e];
                }
                const float kn2 = sumsq32(kr), dd2 = sumsq32(vv);
                if (valid) {
                    float4 *kd = reinterpret_cast<float4 *>(Kf + jr * KS);
                    float4 *dd4 = reinterpret_cast<float4 *>(DLf + jr * KS);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        kd[e] = make_float4(kr[4 * e], kr[4 * e + 1], kr[4 * e + 2], kr[4 * e + 3]);
                        dd4[e] = make_float4(vv[4 * e], vv[4 * e + 1], vv[4 * e + 2], vv[4 * e + 3]);
                    }
                    SC[jr] = make_float4(se, sa, kn2, dd2);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) kr[e] = 0.0f;
                }
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    store_split8(sKP + (jr >> 3) * KP_GSTR + g * 128 + (jr & 7) * 16, 512, kr + 8 * g);
            }
            fence_async_smem();
            tc_before();
            __syncthreads();
            tc_after();
            // ---- B. the Gram matrix k_i . k_j on the tensor core (six split cross terms,
            // rows i in the token pair's lanes, columns j); the gates and step control of each
            // token with the retention products (gain pair); the queries and the readout MMA
            // (token pair)
            if (issuer && !*abort_flag) {
                constexpr int pa[6] = {0, 0, 1, 0, 2, 1};
                constexpr int pb[6] = {0, 1, 0, 2, 0, 1};
                const uint64_t da = sdesc(smem_u32(sKP) - (rw >> 1) * 8 * KP_GSTR, 128, KP_GSTR);
                const uint64_t db = sdesc(smem_u32(sKP), 128, KP_GSTR);
#pragma unroll
                for (int t = 0; t < 6; ++t)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma(tbase + COL_GRAM, dadd(da, pa[t] * 512 + ks * 256), dadd(db, pb[t] * 512 + ks * 256),
                            idesc_bf16(128, 64), (t | ks) != 0);
                mma_commit(mb_gram);
            }
            if (gainw) {
                const int jg = tid & 63;  // route-ordered token
                const bool tv = jg < Lt;
                float alpha = 1.0f, eta_t = 0.0f;
                if (tv) {
                    const float4 sc = SC[jg];
                    float eta, oma;
                    gates(a, sc.x, sc.y, eta, alpha, oma);
                    if (a.gate_mode == VH_GATE_FORCED_EXEC) {
                        eta_t = a.forced_eta;
                    } else {
                        const StepOut so = step_control<kAbl>(a, eta, alpha, oma, sc.z, sc.w);
                        eta_t = so.eta_tilde;
                        n_spec += so.spec_active;
                        n_inj += so.inj_ratio_gt1;
                    }
                }
                // inclusive prefix and suffix products of the retentions over the sub-tile
                // (tokens past the chunk retain 1), each warp holding 32 tokens
                const int gl = jg & 31;
                const bool hi = jg >= 32;
                float pre = alpha, suf = alpha;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float t1 = __shfl_up_sync(0xffffffffu, pre, o);
                    const float t2 = __shfl_down_sync(0xffffffffu, suf, o);
                    if (gl >= o) pre *= t1;
                    if (gl + o < 32) suf *= t2;
                }
                if (!hi && gl == 31) scan_tot[0] = pre;  // tokens 0..31
                if (hi && gl == 0) scan_tot[1] = suf;    // tokens 32..63
                named_sync(3, 64);                       // both halves written; SC read
                if (hi) pre *= scan_tot[0]; else suf *= scan_tot[1];
                float gpre = __shfl_up_sync(0xffffffffu, pre, 1);    // gamma_{j-1}
                float sig = __shfl_down_sync(0xffffffffu, suf, 1);   // sigma_j
                if (gl == 0) gpre = hi ? scan_tot[0] : 1.0f;
                if (gl == 31) sig = hi ? 1.0f : scan_tot[1];
                ALP[jg] = alpha;
                ETA[jg] = eta_t;
                GPRE[jg] = gpre;
                SIG[jg] = sig;
                if (jg == Lt - 1) *gam_slot = pre;  // gamma_L
                // r_j = gamma_{j-1} k_j + delta_j in place of delta_j (zero past the chunk)
                float4 *dr = reinterpret_cast<float4 *>(DLf + jg * KS);
                const float4 *kk = reinterpret_cast<const float4 *>(Kf + jg * KS);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 dv = dr[e], kv = kk[e];
                    dr[e] = tv ? make_float4(fmaf(gpre, kv.x, dv.x), fmaf(gpre, kv.y, dv.y),
                                             fmaf(gpre, kv.z, dv.z), fmaf(gpre, kv.w, dv.w))
                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                }
            } else {
                // queries: q = normalize(M^q_b x), split into the readout's A operand
                float qr[32];
                tmem_ld32(tbase + lrow + COL_GEN + COL_QR, qr);
                const float rq = __frsqrt_rn(sumsq32(qr) + a.knorm_eps);
#pragma unroll
                for (int e = 0; e < 32; ++e) qr[e] *= rq;
#pragma unroll
                for (int g = 0; g < 4; ++g) store_split8(sQ + op_off(jq, g), Q_PIECE, qr + 8 * g);
                fence_async_smem();
                tc_before();
                named_sync(1, 64);
                tc_after();
                // MMA 2: readout y = q M^m_b^T, Eq. (16), beside the Gram columns
                if (issuer && !*abort_flag) {
                    mma_split6<Q_PIECE, S_PIECE>(tbase + COL_RO_WY, smem_u32(sQ) - (rw >> 1) * 8 * SBO_K32,
                                                 smem_u32(sS) + (ROW_MEM + 3 * D) / 8 * SBO_K32,
                                                 idesc_bf16(128, 32));
                    mma_commit(mb_ro);
                }
            }
            tc_before();
            __syncthreads();
            tc_after();
            // ---- C. the solve's coefficients: row i = jq of the packed matrix from Gram row i
            // (this thread's TMEM lane), c(i, j) = (prod_{i<s<j} alpha_s) k_i . k_j for j > i
            if (!gainw) {
                wt.wait(mb_gram, ph_gram);
                tc_after();
                float gr[64];
                {
                    float g0[32], g1[32];
                    tmem_ld32(tbase + lrow + COL_GRAM, g0);
                    tmem_ld32(tbase + lrow + COL_GRAM + 32, g1);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        gr[e] = g0[e];
                        gr[32 + e] = g1[e];
                    }
                }
                const int i = jq;
                if (i < Lp - 1) {
                    const int j0 = wy_j0(i);
                    float *row = cpk + wy_off(Lp, i) - j0;  // row[j] = c(i, j), j >= j0
                    const bool live = i < Lt;
                    float rat = 1.0f;
#pragma unroll
                    for (int j4 = 0; j4 < TT; j4 += 4) {
                        if (j4 < Lp) {
                            const float4 al = *reinterpret_cast<const float4 *>(ALP + j4);
                            const float av[4] = {al.x, al.y, al.z, al.w};
                            float cv[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int j = j4 + u;
                                cv[u] = (live && j > i && j < Lt) ? rat * gr[j] : 0.0f;
                                if (j > i) rat *= av[u];
                            }
                            if (j4 >= j0)
                                *reinterpret_cast<float4 *>(row + j4) = make_float4(cv[0], cv[1], cv[2], cv[3]);
                        }
                    }
                }
            }
            ph_gram ^= 1;
            tc_before();
            __syncthreads();
            tc_after();
            // ---- D. the solve on one warp of the gain pair (lane = gain row) while the token
            // pair adds the readout to out
            const int gw0 = 2 * gp;
            if (warp == gw0) {
                if (Lp == 56)
                    wy_solve<56>(DLf, cpk, ETA, SIG, sWP, lane);
                else if (Lp == 28)
                    wy_solve<28>(DLf, cpk, ETA, SIG, sWP, lane);
                else if (Lp == 32)
                    wy_solve<32>(DLf, cpk, ETA, SIG, sWP, lane);
                else
                    wy_solve<64>(DLf, cpk, ETA, SIG, sWP, lane);
                fence_async_smem();
            } else if (!gainw) {
                wt.wait(mb_ro, ph_ro);
                tc_after();
                float y[32];
                tmem_ld32(tbase + lrow + COL_RO_WY, y);
                const int pix = rowr ? Lidx * W + p : p * W + Lidx;
                if (valid && VH_IN(a.stats, ((size_t)b * H * W + pix) * Cc + (size_t)h * D, D, map_elems(a))) {
                    float *dst = ob + (size_t)pix * Cc;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float4 v4 = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
                        if (lam) {
                            v4.x *= lam[4 * e]; v4.y *= lam[4 * e + 1];
                            v4.z *= lam[4 * e + 2]; v4.w *= lam[4 * e + 3];
                        }
                        n_nf += !isfinite(v4.x) + !isfinite(v4.y) + !isfinite(v4.z) + !isfinite(v4.w);
                        red_add_v4(dst + 4 * e, v4);
                    }
                }
            }
            tc_before();
            __syncthreads();
            tc_after();
            // ---- E. G = gamma_L I + W' K^T on the tensor core, formed transposed:
            // G^T = gamma_L I + K W'^T with the key pieces as the MN-major A operand (rows =
            // columns b of G, landing in the solving warp's lanes) and W' as B with its three
            // pieces stacked along N.  Per K step (16 tokens) one MMA per key piece against
            // N = 96, 64, 32: the six cross terms in three column blocks.
            if (issuer && !*abort_flag) {
                const uint64_t dk = sdesc(smem_u32(sKP) - 1024 * gp, KP_GSTR, 128);
                const uint64_t dw = sdesc(smem_u32(sWP), 128, WP_SBO);
#pragma unroll
                for (int ks = 0; ks < TT / 16; ++ks)
#pragma unroll
                    for (int pc = 0; pc < 3; ++pc)
                        mma(tbase + COL_ASM, dadd(dk, pc * 512 + ks * 2 * KP_GSTR), dadd(dw, ks * 256),
                            idesc_bf16(128, 96 - 32 * pc, false, true), (ks | pc) != 0);
                mma_commit(mb_asm);
            }
            if (warp == gw0) {
                // column b = lane of G: the three blocks summed, gamma_L on the diagonal; fp32
                // rows for the eta / alpha rows and the update's B operand (K-major: row n = b,
                // K = the rows of G; pieces stacked along N) in three bf16 pieces, as G - I when
                // the chunk retains at least half of the state (as in the recurrence form)
                wt.wait(mb_asm, ph_asm);
                tc_after();
                float v[32], w2[32];
                tmem_ld32(tbase + lrow + COL_ASM, v);
                tmem_ld32(tbase + lrow + COL_ASM + D, w2);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] += w2[e];
                tmem_ld32(tbase + lrow + COL_ASM + 2 * D, w2);
                const float gL = *gam_slot;
                const bool use_delta = gL >= 0.5f;
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = (v[e] + w2[e]) + (e == lane ? gL : 0.0f);
#pragma unroll
                for (int e = 0; e < 32; ++e) Gf[e * GFS + lane] = v[e];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float v8[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        v8[u] = v[8 * g + u] - ((use_delta && 8 * g + u == lane) ? 1.0f : 0.0f);
                    store_split8(sG + (lane >> 3) * SBO_K32 + g * LBO_K32 + (lane & 7) * 16, G_PIECE, v8);
                }
                if (lane == 0) *delta_form = use_delta ? 1 : 0;
                fence_async_smem();
                tc_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(mb_g);
            } else if (warp == gw0 + 1) {
                if (lane == 0) mbar_arrive(mb_g);
            }
            ph_asm ^= 1;
            // ---- MMA 3 (chunk end): every d x d memory <- M_b G, as in the recurrence form
            // but with G's pieces K-major
            if (issuer) {
                if (wt.wait(mb_g, ph_g) && !*abort_flag) {
                    tc_after();
                    const uint64_t da = sdesc(smem_u32(sS) + ROW_MEM / 8 * SBO_K32, LBO_K32, SBO_K32);
                    const uint64_t db = sdesc(smem_u32(sG), LBO_K32, SBO_K32);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint32_t ka = ks * 2 * LBO_K32;
                        mma(tbase + COL_UPD, dadd(da, ka), dadd(db, ka), idesc_bf16(128, 96), ks != 0);
                        mma(tbase + COL_UPD, dadd(da, S_PIECE + ka), dadd(db, ka), idesc_bf16(128, 64), 1);
                        mma(tbase + COL_UPD + 2 * D, dadd(da, 2 * S_PIECE + ka), dadd(db, ka),
                            idesc_bf16(128, 32), 1);
                    }
                    mma_commit(mb_upd);
                }
            }
            } else {
            // ---- per-token step, Eqs. (15), (19), (20), (53).  The token pair (lane = token)
            // normalises k, forms delta = k - v and their squared norms, and publishes the
            // token's scalars; then the gain pair (lane = route-ordered token) evaluates the
            // gates and the step control while the token pair forms the Gram entries.
            if (!gainw) token_step(Kf, DLf, SC, valid, jr, c, t0);
            __syncthreads();
            if (gainw)
                gate_step(SC, Lt);
            else
                gram_step(Kf, GT);
            tc_before();
            __syncthreads();
            tc_after();
            if (gainw) {
                gain_step(Kf, DLf, SC, GT, Lt, s == 0, last);
            } else {
                // ---- the token pair, while the gain runs: queries and the readout of this
                // sub-tile.  For the intra-chunk readout it waits for the gain pair's u_t
                // and reads those out instead.
                if (intra) {
                    named_sync(2, NT);
                    float uv[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) uv[e] = valid ? DLf[jr * KS + e] : 0.0f;
#pragma unroll
                    for (int g = 0; g < 4; ++g) store_split8(sQ + op_off(jq, g), Q_PIECE, uv + 8 * g);
                    fence_async_smem();
                    tc_before();
                    named_sync(1, 64);
                    tc_after();
                } else if (!exact) {
                    float qr[32];
                    tmem_ld32(tbase + lrow + COL_GEN + COL_QR, qr);
                    const float qqr = sumsq32(qr);
                    const float rq = __frsqrt_rn(qqr + a.knorm_eps);
#pragma unroll
                    for (int e = 0; e < 32; ++e) qr[e] *= rq;
                    if (kAbl && a.rec && rec_ok && valid) {  // the token record's vectors: k and delta
                                                   // from their tiles (read-only here), q
                        float *rq4 = rec_at(a, c * Lline + t0 + jr);
                        float4 *rd = reinterpret_cast<float4 *>(rq4);
                        const float4 *ks = reinterpret_cast<const float4 *>(Kf + jr * KS);
                        const float4 *ds = reinterpret_cast<const float4 *>(DLf + jr * KS);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            rd[e] = ks[e];
                            rd[D / 4 + e] = make_float4(qr[4 * e], qr[4 * e + 1], qr[4 * e + 2], qr[4 * e + 3]);
                            rd[2 * D / 4 + e] = ds[e];
                        }
                        rq4[3 * D + TR_QQ] = qqr;
                    }
#pragma unroll
                    for (int g = 0; g < 4; ++g) store_split8(sQ + op_off(jq, g), Q_PIECE, qr + 8 * g);
                    fence_async_smem();
                    tc_before();
                    named_sync(1, 64);
                    tc_after();
                }
                // MMA 2: readout y = q M^m_b^T, Eq. (16) (six split cross terms), M = 128 with
                // the queries as rows 32 rw..32 rw+63 (the other 64 A rows read the region
                // next to each piece).  The outer queries of the VisionHOPE-exact readout
                // arrive by TMA in their own layout.
                if (issuer) {
                    if (!exact || intra) {
                        if (!*abort_flag) {
                            mma_split6<Q_PIECE, S_PIECE>(
                                tbase + COL_RO, smem_u32(sQ) - (rw >> 1) * 8 * SBO_K32,
                                smem_u32(sS) + (ROW_MEM + 3 * D) / 8 * SBO_K32, idesc_bf16(128, 32));
                            mma_commit(mb_ro);
                        }
                    } else if (wait_copy(mb_q, ph_q, nq_obs) && !*abort_flag) {
                        constexpr int pa[6] = {0, 0, 1, 0, 2, 1};
                        constexpr int pb[6] = {0, 1, 0, 2, 0, 1};
                        const uint64_t da = sdesc(smem_u32(sQ) - (rw >> 1) * 8 * SBO_X, QX_LBO, SBO_X);
                        const uint64_t db =
                            sdesc(smem_u32(sS) + (ROW_MEM + 3 * D) / 8 * SBO_K32, LBO_K32, SBO_K32);
#pragma unroll
                        for (int t = 0; t < 6; ++t)
#pragma unroll
                            for (int ks = 0; ks < 2; ++ks)
                                mma(tbase + COL_RO, dadd(da, pa[t] * QX_PIECE + ks * 2 * QX_LBO),
                                    dadd(db, pb[t] * S_PIECE + ks * 2 * LBO_K32), idesc_bf16(128, 32),
                                    (t | ks) != 0);
                        mma_commit(mb_ro);
                    }
                }
                if (exact) ph_q ^= 1;
                wt.wait(mb_ro, ph_ro);
                tc_after();
                // the query tile is free again: fetch the next sub-tile's outer queries
                if (exact && issuer && !*abort_flag) {
                    const int ns = (s + 1 < nsub) ? s + 1 : 0;
                    const int nc = (s + 1 < nsub) ? c : c + 1;
                    if (nc < nlines) issue_q(nc, ns);
                }
                add_readout(p, Lidx, valid);
                if (last && issuer) issue_update();
            }
            }  // recurrence form
            ph_ro ^= 1;
            if (last) {
                ph_g ^= 1;
                tc_before();
                __syncthreads();  // G and its fp32 rows written, readout complete
                tc_after();
                chunk_end(c);
            }
            fence_async_smem();
            tc_before();
            __syncthreads();  // end of sub-tile: operands rewritten, TMEM consumed
        }
    }

    }  // pipelined or sequential sub-tiles

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
    // and the copy in flight on each TMA barrier.
    if (issuer && *abort_flag) {
        mma_commit(mb_drain);
        drain_wait(mb_drain, 0);
        if (nx_obs < nx_iss) drain_wait(mb_x, (nx_iss - 1) & 1);
        if (nq_obs < nq_iss) drain_wait(mb_q, (nq_iss - 1) & 1);
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                     "r"(TMEM_COLS)
                     : "memory");
}

// ------------------------------------------------------------- host side


// 5-D view of the outer-query pieces [3][B][H][W][Cc] bf16: (channel, position along the
// line, line, image, piece); a box is 8 channels x 64 positions x all 3 pieces.
bool make_qmap(CUtensorMap *m, const void *q, int B, int H, int W, int Cc, bool rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t e = 2;
    cuuint64_t dims[5], strides[4];
    dims[0] = (cuuint64_t)Cc;
    dims[1] = (cuuint64_t)(rows ? W : H);
    dims[2] = (cuuint64_t)(rows ? H : W);
    dims[3] = (cuuint64_t)B;
    dims[4] = 3;
    strides[0] = rows ? (cuuint64_t)Cc * e : (cuuint64_t)W * Cc * e;
    strides[1] = rows ? (cuuint64_t)W * Cc * e : (cuuint64_t)Cc * e;
    strides[2] = (cuuint64_t)H * W * Cc * e;
    strides[3] = (cuuint64_t)B * H * W * Cc * e;
    const cuuint32_t box[5] = {8, (cuuint32_t)TT, 1, 1, 3};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(q), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view of x [B][H][W][Cc] bf16 with dims (channel, position along the line,
// line, image); row routes walk W inside a row, column routes walk H inside a column.
bool make_map(CUtensorMap *m, const void *x, int B, int H, int W, int Cc, bool rows)
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

}  // namespace tc

// Tensor-core path: head_dim 32, bf16 x, row/column-aligned chunks.  Sets
// *handled = false (and returns success) for any other shape.  gain: VH_IMPL_TC_WY selects
// the WY form of the shared gain (the method as defined, no outer queries, every chunk
// within one 64-token sub-tile; a request the shape does not admit returns
// cudaErrorNotSupported); anything else takes the blocked recurrence, the faster form.
cudaError_t launch_scan_tc(const ScanArgs &a, int d, bool bf16, cudaStream_t st, bool *handled,
                           int gain)
{
    *handled = false;
    const bool aligned = a.chunk == 0 || (a.chunk == a.W && a.chunk == a.H);
    auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (d != tc::D || !bf16 || !aligned || (a.Cc % 8) != 0 || !a16(a.mem0) ||
        (a.mem_out && !a16(a.mem_out)))
        return cudaSuccess;
    const bool abl = a.control_flags || a.ckpt;
    const bool wy_ok = !abl && !a.qhat && a.H <= tc::TT && a.W <= tc::TT;
    if (gain == VH_IMPL_TC_WY && !wy_ok) return cudaErrorNotSupported;
    const bool wy = wy_ok && gain == VH_IMPL_TC_WY;
    // the pipelined sub-tiles where a line spans several of them, as long as the grid fits
    // the two CTAs per SM its shared memory allows (else the sequential form's three)
    const bool pipe_ok = !abl && !a.qhat;
    if (gain == VH_IMPL_TC_PIPE && !pipe_ok) return cudaErrorNotSupported;
    CUtensorMap mr, mc, qr, qc;
    if (!tc::make_map(&mr, a.x, a.B, a.H, a.W, a.Cc, true) ||
        !tc::make_map(&mc, a.x, a.B, a.H, a.W, a.Cc, false))
        return cudaErrorInvalidValue;
    if (a.qhat) {
        if (!tc::make_qmap(&qr, a.qhat, a.B, a.H, a.W, a.Cc, true) ||
            !tc::make_qmap(&qc, a.qhat, a.B, a.H, a.W, a.Cc, false))
            return cudaErrorInvalidValue;
    } else {
        qr = mr;  // not read
        qc = mc;
    }
    static int attr_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(tc::scan_tc_kernel<false, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::scan_tc_kernel<true, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_INTRA);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::scan_tc_kernel<false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Lay<true>::BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc::scan_tc_kernel<false, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_PIPE);
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const unsigned grid = (unsigned)(a.B * a.ndirs * a.nh);
    bool pipe = gain == VH_IMPL_TC_PIPE;
    if (pipe_ok && (gain == VH_IMPL_AUTO || gain == VH_IMPL_TC) && (a.H > tc::TT || a.W > tc::TT)) {
        int nsm = 0;
        e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        pipe = grid <= 2u * (unsigned)nsm;
    }
    if (abl) {
        const int smem = (a.control_flags & VH_CTRL_INTRA_READ) ? tc::SMEM_INTRA : tc::SMEM_BYTES;
        tc::scan_tc_kernel<true, false><<<grid, tc::NT, smem, st>>>(a, mr, mc, qr, qc);
    } else if (wy) {
        tc::scan_tc_kernel<false, true><<<grid, tc::NT, tc::Lay<true>::BYTES, st>>>(a, mr, mc, qr, qc);
    } else if (pipe) {
        tc::scan_tc_kernel<false, false, true><<<grid, tc::NT, tc::SMEM_PIPE, st>>>(a, mr, mc, qr, qc);
    } else {
        tc::scan_tc_kernel<false, false><<<grid, tc::NT, tc::SMEM_BYTES, st>>>(a, mr, mc, qr, qc);
    }
    *handled = true;
    return cudaGetLastError();
}

}  // namespace vh
