// vh_gemm_tc.cu -- the pointwise layers of the VisionHOPE block ("VisionHOPE: Visual
// Backbones as Self-Modifying Learning Systems", Sec. 2.3 Eq. (27), App. B.5: Proj_in,
// Proj_out and the two FFN layers) as tcgen05 GEMMs with fused epilogues:
//   out[m][n] = act[m][:] . w[n][:]  (+ bias[n])  (+ res[m][n])        fp32 out, or
//   out[m][n] = bf16(GELU(bf16(act[m][:] . w[n][:]) + bias[n]))        bf16 out (FFN1 + GELU)
// act [M][K] and w [N][K] are row-major bf16 (both K-major operands), fp32 accumulation in
// TMEM.  GELU is the exact erf form; the bf16 rounding of the product before its bias is
// the block's rounding point.
//
// Persistent CTAs (one per SM, 448 threads): warp 0 issues the TMA copies of a three-stage
// ring (per stage 64 K-elements of a 128-row activation tile and of the BN-row weight tile,
// each one box of whole 128-byte rows in the 128-byte swizzled K-major layout), warp 1 (one
// lane) issues the MMAs (M = 128, N = BN <= 256, K = 16) into one of two TMEM accumulators,
// and warps 2..13 (thread = tile row, three warps per row quarter taking every third
// 32-column chunk) run the epilogue of one tile while the next one accumulates.  The
// epilogue turns each 32 x 32 chunk around in a padded shared tile, so its global loads
// and stores run along rows.  Tiles are ordered with the N tiles of one M tile adjacent, so an
// activation tile is read from HBM once and from L2 for its other N tiles.  Every mbarrier
// wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "vh_tc_ptx.cuh"

namespace vh {
namespace gemm {

using namespace vh::tc;

constexpr int BM = 128, BK = 64, STAGES = 3;
constexpr int EPI_WARPS = 12;  // warps 2..13: three per TMEM lane quarter, every third 32-column chunk
constexpr int NT = 32 * (2 + EPI_WARPS);
constexpr int MAX_BN = 256;
constexpr int A_STAGE = BM * BK * 2;                 // 16 KB
constexpr int B_STAGE = MAX_BN * BK * 2;             // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
constexpr int STG_WORDS = 32 * 33;                  // per epilogue warp: a 32 x 32 chunk, padded
constexpr int OFF_STG = OFF_B + STAGES * B_STAGE;
constexpr int OFF_BAR = OFF_STG + EPI_WARPS * STG_WORDS * 4;
constexpr int SMEM_BYTES = OFF_BAR + 256;
static_assert(SMEM_BYTES <= 227 * 1024, "one CTA per SM");
static_assert(A_STAGE % 1024 == 0 && B_STAGE % 1024 == 0 && OFF_B % 1024 == 0, "swizzled tiles 1 KB aligned");

enum { EPI_F32 = 0, EPI_GELU_BF16 = 1, EPI_GELU_SPLIT3 = 2 };

struct GemmArgs {
    const float *bias;  // [N] or nullptr
    const float *res;   // [M][N] fp32 or nullptr (may equal out)
    void *out;          // [M][N] fp32 (EPI_F32) or bf16 (EPI_GELU_BF16)
    int M, N, K;
    int BN, ntn, nkb;   // N tile, N tiles, K blocks of BK
    int epi;
    unsigned long long *stats;  // timeout counter (or nullptr)
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int c0, int c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzled layout:
// rows of 64 bf16 (128 bytes) with their 16-byte chunks permuted by row % 8 (the layout
// the TMA writes with 128-byte swizzle), 8-row groups 1 KB apart, the tile 1 KB aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr)
{
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Exact GELU, a Phi(a) with Phi the standard normal CDF.  With z = |a| / sqrt(2),
//   Phi(a) = e(z) for a < 0 and 1 - e(z) for a >= 0,   e(z) = erfc(z) / 2 = exp(-z^2) t S(t),
//   t = 1 / (1 + z / 2),
// the substitution of the Chebyshev erfc fit in Numerical Recipes (2nd ed., Sec. 6.2).  S
// is our own degree-8 polynomial in t, fitted (fp32 coefficients) by least squares weighted
// for relative error at Chebyshev nodes of t in [1/6, 1], i.e. z in [0, 10]: the relative
// error of e is below 7e-8 in exact arithmetic.  e is accurate in relative terms on both
// tails, so a Phi(a) keeps its precision for negative a, where 1 + erf(a / sqrt 2) would
// cancel.  exp(-z^2) = 2^(a^2 K) with K = -log2(e) / 2; the roundings of a^2 and of a^2 K
// are carried into a first-order correction, so they do not reach the result.  Beyond
// |a| = 13 the tail underflows: Phi is 0 or 1 there (GELU(a) = -0 or a).
__device__ __forceinline__ float gelu_exact(float a)
{
    const float ax = fminf(fabsf(a), 13.5f);
    const float t = rcp_approx(fmaf(ax, 0.353553391f, 1.0f));  // 1 / (1 + |a| / (2 sqrt 2))
    float S = -0.0300543532f;
    S = fmaf(S, t, 0.144723058f);
    S = fmaf(S, t, -0.248414785f);
    S = fmaf(S, t, 0.144257575f);
    S = fmaf(S, t, -0.0166995097f);
    S = fmaf(S, t, 0.102680214f);
    S = fmaf(S, t, 0.121239692f);
    S = fmaf(S, t, 0.141226918f);
    S = fmaf(S, t, 0.141041175f);
    constexpr float K = -0.721347520f;           // -log2(e) / 2, rounded
    constexpr float K_LO = -9.62981495e-09f;      // -log2(e) / 2 - K
    const float a2 = ax * ax;
    const float a2_lo = fmaf(ax, ax, -a2);        // a^2 = a2 + a2_lo exactly
    const float yh = a2 * K;
    const float yl = fmaf(a2, K, -yh) + fmaf(a2_lo, K, a2 * K_LO);
    const float p = ex2_approx(yh);
    const float ex = fmaf(p, yl * 0.693147181f, p);  // 2^(yh + yl), to first order in yl
    const float e = t * S * ex;
    return a * (a < 0.0f ? e : 1.0f - e);
}

// Packed fp32 pairs (element 0 in the low word): each lane of an .f32x2 instruction is the
// same correctly rounded fp32 operation as its scalar form.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpk2(f32x2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 neg2(f32x2 a) { return a ^ 0x8000000080000000ull; }
__device__ __forceinline__ f32x2 splat2(float v) { return pk2(v, v); }

// gelu_exact on two values at once, the same operations in the same order on packed
// pairs (bit for bit the scalar results): about half the instruction issues.
__device__ __forceinline__ void gelu_exact2(float a0, float a1, float &g0, float &g1)
{
    const f32x2 ax = pk2(fminf(fabsf(a0), 13.5f), fminf(fabsf(a1), 13.5f));
    float d0, d1;
    unpk2(fma2(ax, splat2(0.353553391f), splat2(1.0f)), d0, d1);
    const f32x2 t = pk2(rcp_approx(d0), rcp_approx(d1));
    f32x2 S = splat2(-0.0300543532f);
    S = fma2(S, t, splat2(0.144723058f));
    S = fma2(S, t, splat2(-0.248414785f));
    S = fma2(S, t, splat2(0.144257575f));
    S = fma2(S, t, splat2(-0.0166995097f));
    S = fma2(S, t, splat2(0.102680214f));
    S = fma2(S, t, splat2(0.121239692f));
    S = fma2(S, t, splat2(0.141226918f));
    S = fma2(S, t, splat2(0.141041175f));
    const f32x2 K = splat2(-0.721347520f), K_LO = splat2(-9.62981495e-09f);
    const f32x2 a2 = mul2(ax, ax);
    const f32x2 a2_lo = fma2(ax, ax, neg2(a2));
    const f32x2 yh = mul2(a2, K);
    const f32x2 yl = add2(fma2(a2, K, neg2(yh)), fma2(a2_lo, K, mul2(a2, K_LO)));
    float y0, y1;
    unpk2(yh, y0, y1);
    const f32x2 p = pk2(ex2_approx(y0), ex2_approx(y1));
    const f32x2 ex = fma2(p, mul2(yl, splat2(0.693147181f)), p);
    const f32x2 e = mul2(mul2(t, S), ex);
    const f32x2 ome = add2(splat2(1.0f), neg2(e));
    float e0, e1, o0, o1;
    unpk2(e, e0, e1);
    unpk2(ome, o0, o1);
    unpk2(mul2(pk2(a0, a1), pk2(a0 < 0.0f ? e0 : o0, a1 < 0.0f ? e1 : o1)), g0, g1);
}

// kSplit3: the fp32-intermediate test mode's epilogue alone (EPI_GELU_SPLIT3), in an
// instantiation of its own so that its code does not shape the production epilogues'
// register allocation; otherwise g.epi picks EPI_F32 or EPI_GELU_BF16 at run time.
template <bool kSplit3>
__global__ void __launch_bounds__(NT, 1)
    gemm_tc_kernel(const GemmArgs g, const __grid_constant__ CUtensorMap tm_a,
                   const __grid_constant__ CUtensorMap tm_b)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
    // bars[0..3] full, [4..7] empty, [8..9] tmem full, [10..11] tmem empty
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 128);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_BAR + 136);
    const Waiter wt{abort_flag, g.stats};
    const int BN = g.BN;
    const uint32_t tcols = BN <= 64 ? 128 : (BN <= 128 ? 256 : 512);  // two accumulators

    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[4 + s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars[8 + b]), 1);
            mbar_init(smem_u32(&bars[10 + b]), EPI_WARPS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)), "r"(tcols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tbase = *tmem_slot;
    const int ntiles = ((g.M + BM - 1) / BM) * g.ntn;
    const uint32_t a_bytes = BM * BK * 2, b_bytes = (uint32_t)BN * BK * 2;

    if (warp == 0) {
        // ---- TMA producer (one lane)
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
                const int tm = t / g.ntn, tn = t % g.ntn;
                for (int kb = 0; kb < g.nkb; ++kb) {
                    if (!wt.wait_inline(smem_u32(&bars[4 + s]), ph ^ 1)) break;  // stage free
                    const uint32_t full = smem_u32(&bars[s]);
                    mbar_expect_tx(full, a_bytes + b_bytes);
                    const uint32_t sa = smem_u32(sm + OFF_A + s * A_STAGE);
                    const uint32_t sb = smem_u32(sm + OFF_B + s * B_STAGE);
                    tma_load_2d(sa, &tm_a, kb * BK, tm * BM, full);
                    tma_load_2d(sb, &tm_b, kb * BK, tn * BN, full);
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (*abort_flag) break;
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer (one lane)
        if (lane == 0) {
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;  // bit b: phase of accumulator b (no indexed arrays: registers)
            const uint32_t idesc = idesc_bf16(BM, BN);
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
                if (!wt.wait_inline(smem_u32(&bars[10 + acc]), ((aph >> acc) & 1u) ^ 1u)) break;  // accumulator free
                aph ^= 1u << acc;
                tc_after();
                const uint32_t dt = tbase + (uint32_t)(acc * BN);
                for (int kb = 0; kb < g.nkb; ++kb) {
                    if (!wt.wait_inline(smem_u32(&bars[s]), ph)) break;  // stage landed
                    tc_after();
                    const uint64_t da = sdesc_sw128(smem_u32(sm + OFF_A + s * A_STAGE));
                    const uint64_t db = sdesc_sw128(smem_u32(sm + OFF_B + s * B_STAGE));
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)  // K step of 16 elements: 32 bytes into each row
                        mma(dt, dadd(da, 32 * k), dadd(db, 32 * k), idesc, (kb | k) != 0);
                    mma_commit(smem_u32(&bars[4 + s]));  // the stage is free once these complete
                    if (++s == STAGES) { s = 0; ph ^= 1; }
                }
                if (*abort_flag) break;
                mma_commit(smem_u32(&bars[8 + acc]));  // the tile's accumulator is complete
                acc ^= 1;
            }
        }
    } else {
        // ---- epilogue: thread = tile row (TMEM lane), 32 columns per TMEM load; the three
        // warps of a lane quarter take every third chunk
        const int q = warp & 3;  // TMEM lane quarter of this warp
        const int part = (warp - 2) >> 2;  // which third of the chunks
        const uint32_t lrow = ((uint32_t)q * 32u) << 16;
        float *stg = reinterpret_cast<float *>(sm + OFF_STG) + (warp - 2) * STG_WORDS;
        int acc = 0;
        uint32_t fph = 0;  // bit b: phase of accumulator b
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
            const int tm = t / g.ntn, tn = t % g.ntn;
            const bool ok = wt.wait_inline(smem_u32(&bars[8 + acc]), (fph >> acc) & 1u);
            fph ^= 1u << acc;
            tc_after();
            const int mbase = tm * BM + 32 * q;  // first of this warp's 32 rows
            for (int cb = 32 * part; ok && cb < BN; cb += 32 * (EPI_WARPS / 4)) {
                float v[32];
                tmem_ld32(tbase + lrow + (uint32_t)(acc * BN + cb), v);
                const int n0 = tn * BN + cb;
                if (n0 >= g.N) continue;
                // the chunk (row per lane) goes through the warp's staging tile so that the
                // global accesses run along rows: lane = column (fp32) or 32-bit word (bf16)
                // (bf16 out) a whole chunk in range leaves straight from the lanes; fp32 rows
                // are twice as long, and there the staged, row-coalesced form measured faster
                const bool whole = n0 + 32 <= g.N && (g.N & 7) == 0 &&
                                   (reinterpret_cast<uintptr_t>(g.out) & 15u) == 0 &&
                                   (reinterpret_cast<uintptr_t>(g.bias) & 15u) == 0;
                if (!kSplit3 && g.epi == EPI_F32) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) stg[lane * 33 + e] = v[e];
                    __syncwarp();
                    const int n = n0 + lane;
                    const float bn = (g.bias && n < g.N) ? __ldg(g.bias + n) : 0.0f;
                    float *out = reinterpret_cast<float *>(g.out);
                    // the residual rows first, all in flight together (they may be out itself)
                    float rv[32];
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) {
                        const int m = mbase + rr;
                        rv[rr] = (g.res && m < g.M && n < g.N) ? g.res[(size_t)m * g.N + n] : 0.0f;
                    }
#pragma unroll
                    for (int rr = 0; rr < 32; ++rr) {
                        const int m = mbase + rr;
                        if (m < g.M && n < g.N)
                            out[(size_t)m * g.N + n] = (stg[rr * 33 + lane] + bn) + rv[rr];
                    }
                    __syncwarp();
                } else if (kSplit3) {
                    // fp32-intermediate test mode: GELU(acc + bias) unrounded, written as its
                    // three bf16 pieces, out[m][n], out[m][N + n], out[m][2N + n]
                    const int m = mbase + lane;
                    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(g.out) + (size_t)m * 3 * g.N;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int n = n0 + e;
                        if (m < g.M && n < g.N) {
                            const float y = gelu_exact(v[e] + __ldg(g.bias + n));
                            const __nv_bfloat16 p1 = __float2bfloat16_rn(y);
                            const float r1 = y - __bfloat162float(p1);
                            const __nv_bfloat16 p2 = __float2bfloat16_rn(r1);
                            out[n] = p1;
                            out[g.N + n] = p2;
                            out[2 * g.N + n] = __float2bfloat16_rn(r1 - __bfloat162float(p2));
                        }
                    }
                } else if (whole) {
                    // whole chunk in range: the row's 32 values straight out of this lane
                    // (four 16-byte stores; a bias vector read as float4)
                    const int m = mbase + lane;
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 b4 = __ldg(reinterpret_cast<const float4 *>(g.bias + n0 + e));
                        const float p0 = __bfloat162float(__float2bfloat16_rn(v[e])) + b4.x;
                        const float p1 = __bfloat162float(__float2bfloat16_rn(v[e + 1])) + b4.y;
                        const float p2 = __bfloat162float(__float2bfloat16_rn(v[e + 2])) + b4.z;
                        const float p3 = __bfloat162float(__float2bfloat16_rn(v[e + 3])) + b4.w;
                        float g0, g1, g2, g3;
                        gelu_exact2(p0, p1, g0, g1);
                        gelu_exact2(p2, p3, g2, g3);
                        w[e / 2] = pack_bf16x2_rn(g0, g1);
                        w[e / 2 + 1] = pack_bf16x2_rn(g2, g3);
                    }
                    if (m < g.M) {
                        uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(g.out) +
                                                               (size_t)m * g.N + n0);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                    }
                } else {
                    uint32_t *stw = reinterpret_cast<uint32_t *>(stg);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float b0 = (n0 + e < g.N) ? __ldg(g.bias + n0 + e) : 0.0f;
                        const float b1 = (n0 + e + 1 < g.N) ? __ldg(g.bias + n0 + e + 1) : 0.0f;
                        // the product rounded to bf16, then the bias and GELU, rounded again
                        const float p0 = __bfloat162float(__float2bfloat16_rn(v[e])) + b0;
                        const float p1 = __bfloat162float(__float2bfloat16_rn(v[e + 1])) + b1;
                        float g0, g1;
                        gelu_exact2(p0, p1, g0, g1);
                        stw[lane * 17 + e / 2] = pack_bf16x2_rn(g0, g1);
                    }
                    __syncwarp();
                    // two rows of 16 words per pass
                    const int wd = lane & 15, n = n0 + 2 * wd;
                    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(g.out);
#pragma unroll 4
                    for (int rr = lane >> 4; rr < 32; rr += 2) {
                        const int m = mbase + rr;
                        if (m < g.M && n < g.N) {
                            const uint32_t val = stw[rr * 17 + wd];
                            const size_t idx = (size_t)m * g.N + n;
                            if (n + 1 < g.N)
                                *reinterpret_cast<uint32_t *>(out + idx) = val;
                            else
                                *reinterpret_cast<uint16_t *>(out + idx) = (uint16_t)(val & 0xffffu);
                        }
                    }
                    __syncwarp();
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars[10 + acc]));  // accumulator free again
            acc ^= 1;
            if (!ok) break;
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(tcols)
                     : "memory");
}

// 2-D view of a row-major bf16 matrix [rows][K]: dims (K, rows), a box of 64 elements (128
// bytes) x box_rows rows written with 128-byte swizzle.  Out-of-range elements read as zero.
bool make_gemm_map(CUtensorMap *m, const void *p, int rows, int K, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The epilogue's GELU alone: out[i] = bf16(GELU(a[i])).
__global__ void gelu_debug_kernel(const float *__restrict__ a, __nv_bfloat16 *__restrict__ out, long long n)
{
    // pairs through the packed form the FFN1 epilogue uses, a last odd element alone
    for (long long i = 2 * (blockIdx.x * (long long)blockDim.x + threadIdx.x); i < n;
         i += 2 * (long long)gridDim.x * blockDim.x) {
        if (i + 1 < n) {
            float g0, g1;
            gelu_exact2(a[i], a[i + 1], g0, g1);
            out[i] = __float2bfloat16_rn(g0);
            out[i + 1] = __float2bfloat16_rn(g1);
        } else {
            out[i] = __float2bfloat16_rn(gelu_exact(a[i]));
        }
    }
}

}  // namespace gemm

cudaError_t launch_gelu_debug(const float *a, __nv_bfloat16 *out, long long n, cudaStream_t st)
{
    if (n <= 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    gemm::gelu_debug_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>(a, out, n);
    return cudaGetLastError();
}

// out = act . w^T with the epilogue `epi` (0: + bias + res, fp32 out; 1: bf16 GELU of the
// bf16-rounded product plus bias; 2: GELU of the unrounded product plus bias as three bf16
// pieces, out [M][3N]).  act [M][K], w [N][K] bf16 row-major; K a multiple of 8
// (16-byte rows), 16-byte aligned pointers.  Returns a CUDA error code.
cudaError_t launch_gemm_tc(int M, int N, int K, const __nv_bfloat16 *w, const __nv_bfloat16 *act,
                           const float *bias, const float *res, void *out, int epi,
                           cudaStream_t st)
{
    if (M < 1 || N < 1 || K < 8 || (K & 7) || epi < gemm::EPI_F32 || epi > gemm::EPI_GELU_SPLIT3 ||
        (epi != gemm::EPI_F32 && !bias))
        return cudaErrorInvalidValue;
    gemm::GemmArgs g{};
    g.bias = bias;
    g.res = res;
    g.out = out;
    g.M = M;
    g.N = N;
    g.K = K;
    // whole 32-column TMEM loads; for wide outputs an N tile whose chunks split evenly over
    // the three epilogue warps of a lane quarter
    g.BN = N <= gemm::MAX_BN ? (N + 31) / 32 * 32 : (N % 192 == 0 ? 192 : gemm::MAX_BN);
    g.ntn = (N + g.BN - 1) / g.BN;
    g.nkb = (K + gemm::BK - 1) / gemm::BK;
    g.epi = epi;
    g.stats = nullptr;
    CUtensorMap ma, mb;
    if (!gemm::make_gemm_map(&ma, act, M, K, gemm::BM) || !gemm::make_gemm_map(&mb, w, N, K, g.BN))
        return cudaErrorInvalidValue;
    static int attr_set[64] = {0};
    static int nsm[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        for (auto fn : {gemm::gemm_tc_kernel<false>, gemm::gemm_tc_kernel<true>}) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, gemm::SMEM_BYTES);
            if (e != cudaSuccess) return e;
        }
        e = cudaDeviceGetAttribute(&nsm[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const int ntiles = ((M + gemm::BM - 1) / gemm::BM) * g.ntn;
    const unsigned grid = (unsigned)(ntiles < nsm[dev] ? ntiles : nsm[dev]);
    if (epi == gemm::EPI_GELU_SPLIT3)
        gemm::gemm_tc_kernel<true><<<grid, gemm::NT, gemm::SMEM_BYTES, st>>>(g, ma, mb);
    else
        gemm::gemm_tc_kernel<false><<<grid, gemm::NT, gemm::SMEM_BYTES, st>>>(g, ma, mb);
    return cudaGetLastError();
}

}  // namespace vh

