// vh_qproj_tc.cu -- tensor-core form of the VisionHOPE-exact readout's query projection
// ("VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.1.2 Eq. (14),
// App. B.5) for heads of d = 32 over bf16 maps with Cc <= 128 channels.
//
// Q = Z W_q^T is a dense GEMM: one persistent CTA walks 128-pixel tiles.  W_q is split
// once per CTA into three bf16 pieces (24 bits; the B operand, K-major, resident in shared
// memory); each tile of z (exact in bf16) arrives by TMA and takes 3 x Cc/16 MMAs into
// TMEM (M = 128 pixels, N = Cc).  The epilogue (thread = pixel = TMEM lane) normalises
// each 32-column head, writes it as three bf16 pieces, and seeds out with the channel-wise
// skip sum_r lambda_r D_r z.  Every mbarrier wait is bounded.
#include "vh_tc_ptx.cuh"

namespace vh {
namespace tc {
namespace {

constexpr int QM = 128;              // pixels per tile (M)
constexpr int QMAXC = 128;           // largest Cc handled here
constexpr int QA_LBO = QM * 16;      // A: K-group stride (one 8-channel TMA box, 2 KB)
constexpr int QA_SBO = 128;          // A: 8-row stride
constexpr int QB_LBO = 128;          // B: K-group stride
constexpr int QST_ROW = 80;          // staging row: one head's 32 bf16 values (64 B) + 16 B pad
constexpr int QST_PIECE = QM * QST_ROW;
// Shared memory, sized by Cc at launch: z tile (Cc/8 boxes) | 3 W_q pieces | Cc skip
// coefficients | the epilogue's staging of one head's three pieces | mbarriers, TMEM slot,
// flags.
__host__ __device__ constexpr int qoff_b(int Cc) { return Cc * QA_LBO / 8; }
__host__ __device__ constexpr int qoff_coef(int Cc) { return qoff_b(Cc) + 3 * Cc * Cc * 2; }
__host__ __device__ constexpr int qoff_st(int Cc) { return (qoff_coef(Cc) + Cc * 4 + 15) / 16 * 16; }
__host__ __device__ constexpr int qoff_bar(int Cc) { return qoff_st(Cc) + 3 * QST_PIECE; }
__host__ __device__ constexpr int qsmem(int Cc) { return qoff_bar(Cc) + 64; }

__global__ void __launch_bounds__(128, 2)
    qproj_tc_kernel(const __grid_constant__ CUtensorMap tz, const __nv_bfloat16 *__restrict__ x,
                    const float *__restrict__ wq, const float *__restrict__ skip,
                    const float *__restrict__ dir_scale, unsigned dirs,
                    __nv_bfloat16 *__restrict__ qhat, float *__restrict__ out, int accumulate,
                    long npix, int Cc, float knorm_eps)
{
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5;
    unsigned char *sA = sm, *sB = sm + qoff_b(Cc);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + qoff_bar(Cc));
    const uint32_t mb_a = smem_u32(&bars[0]), mb_d = smem_u32(&bars[1]);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + qoff_bar(Cc) + 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + qoff_bar(Cc) + 40);
    const Waiter wt{abort_flag, nullptr};
    const int bsbo = (Cc / 8) * 128;           // B: 8-row (output) group stride
    const int bpiece = Cc * Cc * 2;
    const long ntiles = (npix + QM - 1) / QM;

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(mb_a, 1);
        mbar_init(mb_d, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)), "r"(128) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // W_q as the B operand: element (n = output, k = input) at
    // (n/8) * bsbo + (k/8) * 128 + (n%8) * 16 + (k%8) * 2 of each piece
#pragma unroll 4
    for (int it = tid; it < Cc * (Cc / 8); it += 128) {
        const int n = it / (Cc / 8), kg = it % (Cc / 8);
        const float4 *w4 = reinterpret_cast<const float4 *>(wq + (size_t)n * Cc + 8 * kg);
        const float4 u0 = __ldg(w4), u1 = __ldg(w4 + 1);
        const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        store_split8(sB + (n >> 3) * bsbo + kg * QB_LBO + (n & 7) * 16, bpiece, v);
    }
    // sum over the enabled routes of lambda_r D_r, per channel
    float *coef = reinterpret_cast<float *>(sm + qoff_coef(Cc));
    if (skip && tid < Cc) {
        float sc = 0.0f;
        for (int r = 0; r < 4; ++r)
            if (dirs & (1u << r))
                sc = fmaf(dir_scale ? dir_scale[(size_t)r * Cc + tid] : 1.0f, skip[(size_t)r * Cc + tid], sc);
        coef[tid] = sc;
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tbase = *tmem_slot;
    const bool issuer = tid == 0;
    auto issue_a = [&](long t) {
        mbar_expect_tx(mb_a, (uint32_t)(Cc * QA_LBO / 8));
        for (int g = 0; g < Cc / 8; ++g)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(sA + g * QA_LBO)),
                "l"(reinterpret_cast<uint64_t>(&tz)), "r"(8 * g), "r"((int)(t * QM)), "r"(mb_a)
                : "memory");
    };
    long t = blockIdx.x;
    if (issuer && t < ntiles) issue_a(t);
    uint32_t ph = 0;
    for (; t < ntiles; t += gridDim.x) {
        if (issuer) {
            if (wt.wait(mb_a, ph) && !*abort_flag) {
                tc_after();
                const uint64_t da = sdesc(smem_u32(sA), QA_LBO, QA_SBO);
                const uint64_t db = sdesc(smem_u32(sB), QB_LBO, bsbo);
                const uint32_t id = idesc_bf16(QM, Cc);
                for (int pc = 0; pc < 3; ++pc)
                    for (int ks = 0; ks < Cc / 16; ++ks)
                        mma(tbase, dadd(da, ks * 2 * QA_LBO), dadd(db, pc * bpiece + ks * 2 * QB_LBO),
                            id, (pc | ks) != 0);
                mma_commit(mb_d);
            }
        }
        wt.wait(mb_d, ph);
        ph ^= 1;
        tc_after();
        // the z tile has been consumed: fetch the next one while the epilogue runs
        if (issuer && !*abort_flag && t + gridDim.x < ntiles) issue_a(t + gridDim.x);
        const long pix = t * QM + tid;
        const long tile0 = t * QM;                       // first pixel of the tile
        const int tpix = (int)(npix - tile0 < QM ? npix - tile0 : QM);
        const uint32_t lrow = ((uint32_t)warp * 32u) << 16;
        const size_t plane = (size_t)npix * Cc;
        unsigned char *stg = sm + qoff_st(Cc);
        for (int h0 = 0; h0 < Cc; h0 += 32) {
            float q[32];
            tmem_ld32(tbase + lrow + (uint32_t)h0, q);
            if (pix < npix) {
                const float rq = 1.0f / sqrtf(sumsq32(q) + knorm_eps);
#pragma unroll
                for (int e = 0; e < 32; ++e) q[e] *= rq;
                // three pieces of the head's 32 values, staged by pixel row
                unsigned char *row = stg + tid * QST_ROW;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint4 w1, w2, w3;
                    uint32_t *a = &w1.x, *b = &w2.x, *c = &w3.x;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float x0 = q[8 * g + 2 * i], x1 = q[8 * g + 2 * i + 1];
                        a[i] = pack_bf16x2_rn(x0, x1);
                        const float r0 = x0 - bf16_lo(a[i]), r1 = x1 - bf16_hi(a[i]);
                        b[i] = pack_bf16x2_rn(r0, r1);
                        c[i] = pack_bf16x2_rn(r0 - bf16_lo(b[i]), r1 - bf16_hi(b[i]));
                    }
                    *reinterpret_cast<uint4 *>(row + 16 * g) = w1;
                    *reinterpret_cast<uint4 *>(row + QST_PIECE + 16 * g) = w2;
                    *reinterpret_cast<uint4 *>(row + 2 * QST_PIECE + 16 * g) = w3;
                }
            }
            __syncthreads();
            // the tile's rows of this head, piece by piece: four 16-byte chunks a row, so a
            // warp writes eight whole 64-byte row segments per store
#pragma unroll 4
            for (int e = tid; e < 3 * 4 * tpix; e += 128) {
                const int pcs = e / (4 * tpix), rem = e - pcs * 4 * tpix, r = rem >> 2, ch = rem & 3;
                const uint4 v = *reinterpret_cast<const uint4 *>(stg + pcs * QST_PIECE + r * QST_ROW + 16 * ch);
                *reinterpret_cast<uint4 *>(qhat + pcs * plane + (size_t)(tile0 + r) * Cc + h0 + 8 * ch) = v;
            }
            __syncthreads();
        }
        if (skip) {
            // out over the tile's contiguous block of pixels x channels, four channels a
            // thread per pass, coalesced
            const size_t base = (size_t)tile0 * Cc;
            const int n4 = tpix * Cc / 4;
#pragma unroll 8
            for (int e = tid; e < n4; e += 128) {
                const int c0 = (4 * e) % Cc;
                const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(x + base + 4 * (size_t)e));
                const float4 c4 = *reinterpret_cast<const float4 *>(coef + c0);
                float4 v = make_float4(c4.x * bf16_lo(raw.x), c4.y * bf16_hi(raw.x), c4.z * bf16_lo(raw.y),
                                       c4.w * bf16_hi(raw.y));
                float4 *dst = reinterpret_cast<float4 *>(out + base) + e;
                if (accumulate) {
                    const float4 a4 = *dst;
                    v.x += a4.x; v.y += a4.y; v.z += a4.z; v.w += a4.w;
                }
                *dst = v;
            }
        }
        tc_before();
        __syncthreads();  // TMEM read before the next tile's MMAs overwrite it
        tc_after();
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(128)
                     : "memory");
}

}  // namespace

// Tensor-core query projection; *handled = false (success) for shapes it does not take.
cudaError_t launch_qproj_tc(const void *x, bool bf16, int d, const float *wq, const float *skip,
                            const float *dir_scale, unsigned dirs, __nv_bfloat16 *qhat, float *out,
                            int accumulate, long npix, int Cc, float knorm_eps, cudaStream_t st,
                            bool *handled)
{
    *handled = false;
    if (!wq || !bf16 || d != 32 || Cc % 32 != 0 || Cc > QMAXC || npix < 1 ||
        (reinterpret_cast<uintptr_t>(wq) & 15u))
        return cudaSuccess;
    auto fn = encode_fn();
    if (!fn) return cudaSuccess;
    CUtensorMap tz;
    const cuuint64_t dims[2] = {(cuuint64_t)Cc, (cuuint64_t)npix};
    const cuuint64_t strides[1] = {(cuuint64_t)Cc * 2};
    const cuuint32_t box[2] = {8, (cuuint32_t)QM};
    const cuuint32_t es[2] = {1, 1};
    if (fn(&tz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    static int attr_set[64] = {0};
    if (dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(qproj_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 qsmem(QMAXC));
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const long ntiles = (npix + QM - 1) / QM;
    const int per_sm = qsmem(Cc) <= 112 * 1024 ? 2 : 1;  // two CTAs per SM when they fit
    const long slots = (long)per_sm * nsm;
    const unsigned grid = (unsigned)(ntiles < slots ? ntiles : slots);
    qproj_tc_kernel<<<grid, 128, qsmem(Cc), st>>>(tz, static_cast<const __nv_bfloat16 *>(x), wq, skip,
                                              dir_scale, dirs, qhat, out, accumulate, npix, Cc,
                                              knorm_eps);
    *handled = true;
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace vh
