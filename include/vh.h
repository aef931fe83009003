/*
 * vh.h -- C ABI of the GB300 VisionHOPE four-direction memory scan (libvh).
 *
 * The operation is the VisionHOPE operator F_VH of "VisionHOPE: Visual
 * Backbones as Self-Modifying Learning Systems", Sec. 2.3 Eqs. (24)-(26):
 * serialise a feature map along four routes, run one self-referential
 * memory scan (SRNL, Sec. 2.1.2-2.1.3 Eqs. (9)-(16), stabilised by Def. 1
 * Eqs. (19)-(21)) per route and head, restore the positions and sum the
 * routes channel-wise.  The memory set is the six-memory form of "Nested
 * Learning: The Illusion of Deep Learning Architectures", part 12,
 * Eqs. (94)-(96): key, value, query and content memories (d x d) and the
 * learning-rate and retention memories (1 x d).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library allocates no device memory inside a call, keeps no state
 *    between calls (apart from the thread-local error string and a cached
 *    per-device attribute query) and never frees caller memory.
 *  - Every call is asynchronous on params->stream (a cudaStream_t; NULL is
 *    the legacy default stream).  Host-side argument errors are reported
 *    before anything is enqueued.
 *  - No C++ exception, abort or device trap crosses the ABI: every call
 *    returns a vh_status; vh_last_error() gives a one-line reason.
 *  - Layouts are row-major, NHWC for feature maps: x[B][H][W][Cc] with
 *    Cc = n_heads * head_dim; head h owns channels [h*d, (h+1)*d).
 *  - Route r: 0 = row-major forward (right), 1 = its full reversal (left),
 *    2 = column-major forward (down: transpose, then flatten), 3 = its full
 *    reversal (up).  The route visits pixel P_r(t) at step t:
 *      P_0(t) = t, P_1(t) = N-1-t, P_2(t) = (t mod H)*W + t div H,
 *      P_3(t) = P_2(N-1-t),  N = H*W.
 */
#ifndef VH_H_
#define VH_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VH_OK = 0,
    VH_ERR_INVALID_ARG = -1,   /* bad pointer, shape, alignment, mask or parameter */
    VH_ERR_UNSUPPORTED = -2,   /* valid but not built: head_dim not in {16,32,64}, dtype */
    VH_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
    VH_ERR_WORKSPACE = -4,     /* workspace missing, too small or misaligned */
    VH_ERR_NONFINITE = -5,     /* vh_check: a readout value was not finite */
    VH_ERR_TIMEOUT = -6,       /* vh_check: a bounded wait on an asynchronous copy or MMA
                                  expired; that call's results are invalid */
    VH_ERR_BOUNDS = -7         /* vh_check: an index check of a VH_DEBUG_BOUNDS build failed
                                  (the access was skipped; results are invalid) */
} vh_status;

typedef enum { VH_DTYPE_F32 = 0, VH_DTYPE_BF16 = 1 } vh_dtype;

enum { VH_DIR_RIGHT = 1, VH_DIR_LEFT = 2, VH_DIR_DOWN = 4, VH_DIR_UP = 8, VH_DIR_ALL = 15 };

/* Ablation switches ("VisionHOPE" Sec. 3.5 and App. C.5):
 *   VH_CTRL_NO_INJ_CAP     no injection control (eta_bar = eta)
 *   VH_CTRL_NO_SPEC_CLAMP  no spectral control (eta_tilde = eta_bar)
 *   VH_CTRL_HARD_INJ       injection clamp min(eta, eta_inj) instead of the soft cap
 *   VH_CTRL_SOFT_SPEC      soft spectral cap eta_spec (1 - exp(-eta_bar / eta_spec))
 *                          instead of the clamp min(eta_bar, eta_spec)
 *   VH_CTRL_NO_DGD         no key-dependent DGD correction -eta_tilde M k k^T
 *   VH_CTRL_FREEZE_KV      M^k, M^v fixed within the image (no adaptive K/V)
 *   VH_CTRL_FREEZE_DYN     m^eta, m^alpha fixed within the image (no adaptive dynamics)
 *   VH_CTRL_INTRA_READ     intra-chunk readout: token t reads the working content memory
 *                          M^m_b G_{t-1} (Prop. 2's shared gain before its own update)
 *                          instead of the chunk's boundary state M^m_b (Eq. (16)); the two
 *                          agree at chunk length 1.  The tensor-core kernel runs this switch
 *                          with 9.5 KB more shared memory per CTA (two CTAs per SM).
 * NO_INJ_CAP takes precedence over HARD_INJ and NO_SPEC_CLAMP over SOFT_SPEC; other
 * bits are rejected. */
enum {
    VH_CTRL_NO_INJ_CAP = 1, VH_CTRL_NO_SPEC_CLAMP = 2, VH_CTRL_HARD_INJ = 4,
    VH_CTRL_SOFT_SPEC = 8, VH_CTRL_NO_DGD = 16, VH_CTRL_FREEZE_KV = 32, VH_CTRL_FREEZE_DYN = 64,
    VH_CTRL_INTRA_READ = 128, VH_CTRL_ALL = 255
};

/* Gate test hooks. */
enum {
    VH_GATE_GENERATED = 0,     /* eta, alpha from their memories, Eq. (15) and Eq. (53) */
    VH_GATE_FORCED_RAW = 1,    /* raw eta = forced_eta, alpha = forced_alpha, then Def. 1 */
    VH_GATE_FORCED_EXEC = 2    /* executed step = forced_eta, alpha = forced_alpha, no control */
};

/* Kernel selection. */
enum {
    VH_IMPL_AUTO = 0,          /* the fastest built kernel for the shape */
    VH_IMPL_SIMT = 1,          /* fp32 CUDA-core kernel */
    VH_IMPL_TC = 2,            /* tensor-core (tcgen05) kernel, its faster gain form: the
                                  recurrence at head_dim 32, WY at head_dim 64 where every
                                  chunk fits one 32-token sub-tile */
    VH_IMPL_TC_WY = 3,         /* tensor-core kernel, shared gain in WY form ("VisionHOPE",
                                  App. B.4 Prop. 2, Eqs. (46), (49) unrolled: the chunk's
                                  triangular system on CUDA cores, the gain assembly
                                  G = gamma_L I + W' K^T on the tensor core); the method as
                                  defined only, with H, W <= 64 at head_dim 32 and H, W <= 32
                                  at head_dim 64, else VH_ERR_UNSUPPORTED */
    VH_IMPL_TC_RECUR = 4,      /* tensor-core kernel, shared gain as the blocked per-token
                                  recurrence of Eq. (46), one sub-tile after the other */
    VH_IMPL_TC_PIPE = 5        /* head_dim 32 tensor-core kernel, the blocked recurrence with
                                  the 64-token sub-tiles of a line pipelined: one warp pair
                                  prepares and reads out sub-tile s + 1 while the other runs
                                  the gain over sub-tile s (the same arithmetic as
                                  VH_IMPL_TC_RECUR).  The method as defined only (no
                                  control_flags, no w_query), else VH_ERR_UNSUPPORTED.
                                  VH_IMPL_AUTO and VH_IMPL_TC take it where a line spans
                                  several sub-tiles and the grid fits two CTAs per SM */
};

/* Indices of the optional device counters (params->stats, 8 x uint64). */
enum {
    VH_STAT_TOKENS = 0,        /* token updates executed (sum over routes and heads) */
    VH_STAT_SPEC_ACTIVE = 1,   /* spectral clamp strictly below the capped candidate */
    VH_STAT_INJ_RATIO_GT1 = 2, /* raw step above the injection limit (eta/eta_inj > 1) */
    VH_STAT_NONFINITE = 3,     /* non-finite readout values */
    VH_STAT_TIMEOUT = 4,       /* CTAs whose bounded wait on an asynchronous copy or MMA
                                  expired (the kernel then stops issuing work; results
                                  of that call are invalid) */
    VH_STAT_BOUNDS = 5,        /* index checks that failed; counted only by a library built
                                  with VH_DEBUG_BOUNDS (libvh_dbg.so), where every global
                                  access of the scan kernels computed from an index (and the
                                  shared-memory rows addressed by token position) is checked
                                  against its array before it is made, and skipped if out
                                  of range */
    VH_STAT_COUNT = 8
};

typedef struct vh_params {
    int batch;                 /* B >= 1 */
    int channels;              /* Cc = n_heads * head_dim */
    int head_dim;              /* d in {16, 32, 64} */
    vh_dtype x_dtype;          /* element type of x: bf16 or f32 */
    /* method constants ("VisionHOPE", App. C.1 and App. B.3) */
    float gamma_eta;           /* raw-step scale, 0.025 */
    float alpha_init;          /* initial retention in (0,1), 0.9 */
    float eta_bias;            /* added to s^eta before softplus; 0 on the pages */
    float eps;                 /* epsilon of Def. 1, 1e-6 */
    float knorm_eps;           /* stabiliser of the key/query L2 norm, 1e-6 */
    float inj_inward;          /* inward factor on eta_inj: limit * (1 - 1e-3) */
    float spec_inward;         /* inward factor on eta_spec: limit * (1 - 1e-6) */
    float kk_floor;            /* floor on ||k||^2 in eta_spec, 1e-20 */
    const float *dir_scale;    /* device [4][Cc] channel-wise lambda_r of Eq. (26); NULL = 1 */
    float *memories_out;       /* device [B][4][n_heads][4d^2+2d]: state after the last
                                  token of each enabled route; NULL = not written; slots of
                                  disabled routes are left untouched */
    int gate_mode;             /* VH_GATE_* */
    float forced_eta, forced_alpha;
    unsigned control_flags;    /* VH_CTRL_* */
    unsigned long long *stats; /* device [VH_STAT_COUNT] counters, accumulated (not cleared);
                                  NULL = off */
    int impl;                  /* VH_IMPL_* */
    int accumulate;            /* 0: out is overwritten (the call zeroes it first);
                                  1: the fused sum of Eq. (26) is added to out's contents */
    void *stream;              /* cudaStream_t */
    /* VisionHOPE-exact readout ("VisionHOPE", Sec. 2.1.2 Eq. (14) and App. B.5): the query
     * is an outer Cc x Cc projection applied once to x and reused by the four routes,
     * L2-normalised within each head (stabiliser knorm_eps), instead of M^q_b x.  The
     * query feeds only the readout, so the memories (memories_out) are the same as in
     * the six-memory form; the M^q slot is carried but not read. */
    const float *w_query;      /* device [Cc][Cc] row-major, q = W_q z; NULL = q from M^q */
    const float *skip;         /* device [4][Cc] channel-wise skip D_r of each route:
                                  Y_r = reads + D_r * Z_r before the fusion; NULL = none */
    void *workspace;           /* device, >= vh_workspace_size() bytes, 16-byte aligned;
                                  holds the normalised queries while the call runs */
    size_t workspace_bytes;
    /* Bounded waits.  Every wait of the tensor-core kernels on an asynchronous copy or MMA
     * gives up after a limit: the CTA then records VH_STAT_TIMEOUT (when stats are given),
     * issues no further copy or MMA and runs to its end; vh_check reports VH_ERR_TIMEOUT
     * and the call's results are invalid.  The context stays usable. */
    long long wait_limit;      /* clock cycles before a wait gives up; 0 = 2^32 (about 2 s) */
    int withhold_first_copy;   /* test hook, head_dim 32 tensor-core kernel only (else
                                  VH_ERR_INVALID_ARG): the kernel never issues its first
                                  input copy, so its first wait can only end by giving up,
                                  with nothing asynchronous issued before or after */
} vh_params;

/* Fill *p with the pages' constants (gamma_eta 0.025, alpha_init 0.9, eps
 * and knorm_eps 1e-6, inward factors 1e-3 / 1e-6, kk_floor 1e-20), bf16 x,
 * no optional outputs, default stream.  batch/channels/head_dim are zeroed
 * and must be set by the caller. */
void vh_params_init(vh_params *p);

/*
 * vh_scan_forward -- the VisionHOPE operator F_VH (Sec. 2.3, Eqs. (24)-(26)).
 *
 *   x          device, [B][H][W][Cc] of p->x_dtype, 16-byte aligned.
 *   memories0  device fp32 [4][n_heads][4d^2+2d]: the learned initial state
 *              of every (route, head), shared by all images (Sec. 2.3: "initialized
 *              from learned values at the beginning of each image").  Block
 *              order: M^k, M^v, M^q, M^m (d x d row-major, acting on column
 *              vectors), m^eta, m^alpha (1 x d).
 *   H, W       map size, H*W*Cc*B elements must fit in 2^31 per image row math.
 *   dirs       nonzero mask of VH_DIR_* routes to run and sum.
 *   chunk      0 = row/column aligned chunks (C_right = C_left = W,
 *              C_down = C_up = H, Eq. (25)); > 0 = that fixed length on every
 *              route, counted from each route's first token, last chunk partial.
 *   out        device fp32 [B][H][W][Cc]: out = sum over enabled r of
 *              lambda_r * P_r^{-1}(Y_r) (p->accumulate = 0), or out += that sum
 *              (p->accumulate = 1).  Must not alias x.  The sum over routes
 *              is taken with device atomics, so its fp32 rounding order is not
 *              fixed from run to run.
 *
 * Per route and head, every chunk generates k, v, q, eta, alpha and the
 * readout y_t = M^m_b q_t from its boundary state (Eqs. (15)-(16)), applies the
 * step control of Def. 1 per token, and advances all six memories with
 * M_t = M_{t-1} A_t + M_b B_t (App. B.4 Eq. (45)), computed through the shared
 * gain M_end = M_b G (Prop. 2 Eq. (46)).
 *
 * With p->w_query set the readout query is the outer projection instead (see
 * vh_params); with p->skip set, lambda_r * D_r * x is added per enabled route.
 *
 * Errors: VH_ERR_INVALID_ARG (null/misaligned pointers, sizes < 1, dirs == 0,
 * chunk < 0, Cc != n_heads*d, alias), VH_ERR_WORKSPACE (w_query without a large
 * enough, 16-byte aligned workspace), VH_ERR_UNSUPPORTED (head_dim or dtype),
 * VH_ERR_CUDA (launch failure; the stream may then hold partial results).
 */
vh_status vh_scan_forward(const void *x, const float *memories0, const vh_params *p,
                          int H, int W, unsigned dirs, int chunk, float *out);

/*
 * vh_debug_permute -- Z_r = P_r(Z) of Eq. (24) for one route, computed with
 * the same device index code the scan uses.  x as in vh_scan_forward; seq
 * device [B][N][Cc] of the same dtype, seq[b][t][:] = x[b][P_r(t)][:].
 * Exists so the index maps can be checked bit for bit.
 */
vh_status vh_debug_permute(const void *x, const vh_params *p, int H, int W, int route,
                           void *seq);

/*
 * vh_debug_gelu -- out[i] = bf16(GELU(a[i])) with the exact GELU a Phi(a) ("VisionHOPE",
 * Sec. 2.3 Eq. (27): the block's FFN; the form the block's FFN1 epilogue applies to its
 * bias-added product), computed by the same device function.  a: device fp32 [n];
 * out: device bf16 [n]; stream: cudaStream_t (NULL = legacy default).  n = 0 is a no-op.
 * Errors: VH_ERR_INVALID_ARG (n < 0, NULL pointers with n > 0), VH_ERR_CUDA.
 * Exists so the activation can be checked element by element.
 */
vh_status vh_debug_gelu(const float *a, void *out, long long n, void *stream);

/*
 * vh_check -- wait for `stream` (a cudaStream_t; NULL = legacy default) and read the
 * device counters a scan wrote into `stats` (device [VH_STAT_COUNT], as passed in
 * vh_params.stats).  Returns VH_ERR_TIMEOUT if any CTA's bounded wait expired (the
 * results of that call are invalid), else VH_ERR_BOUNDS if an index check of a
 * VH_DEBUG_BOUNDS build failed, else VH_ERR_NONFINITE if a non-finite readout value was
 * produced, else VH_OK.  VH_ERR_INVALID_ARG for a NULL stats pointer,
 * VH_ERR_CUDA if the synchronisation or the 64-byte copy fails.  The pages define no
 * such step: it surfaces the kernel's own status flags.
 */
vh_status vh_check(const unsigned long long *stats, void *stream);

/* 1 in a library built with VH_DEBUG_BOUNDS (libvh_dbg.so: checked indices, counted in
 * stats[VH_STAT_BOUNDS]), else 0. */
int vh_debug_bounds_build(void);

/* Bytes of device workspace a vh_scan_forward call with these parameters needs: 0 in
 * the six-memory form, 6 * B * H * W * Cc (the normalised queries as three bf16
 * pieces) when p->w_query is set.  NULL p gives 0. */
size_t vh_workspace_size(const vh_params *p, int H, int W, unsigned dirs, int chunk);

/*
 * vh_scan_backward -- outer gradients of vh_scan_forward ("VisionHOPE" Sec. 2.1.2: the
 * recurrence is explicit and differentiable, so gradients pass through the memory
 * trajectory; Sec. 3.4 Eq. (60) for the activation storage of training).  With
 * L = <dout, out> + <dmem_final, memories_out> for the forward call with the same x,
 * memories0, p, H, W, dirs and chunk, it writes
 *   dx     device fp32 [B][H][W][Cc], 16-byte aligned: dL/dx (overwritten);
 *   dmem0  device fp32 [4][n_heads][4d^2+2d]: dL/dmemories0 summed over the batch
 *          (overwritten; the blocks of disabled routes are zero).
 * dout is device fp32 [B][H][W][Cc]; dmem_final is device fp32 [B][4][n_heads][4d^2+2d]
 * or NULL (no loss on the final memories).  None of the outputs may alias an input.
 *
 * The call recomputes the forward: it keeps every chunk's boundary state and, per scan,
 * the current chunk's gain slices and token records in p->workspace, which must hold
 * vh_backward_workspace_size() bytes, 16-byte aligned.  Where the tensor-core forward
 * applies (head_dim 32, bf16 x, chunks aligned with rows and columns, impl not SIMT) it
 * runs first and writes the boundary states and every token's record; one CUDA-core
 * kernel, fp32, then forms the gradients, summed over routes and images with device
 * atomics (their rounding order is not fixed).  The branch of the step control follows
 * the forward's choice.  p->stats, when set, receives the tensor-core pre-pass's counters
 * (as a forward call's), expired waits and, in a VH_DEBUG_BOUNDS build, failed index
 * checks of both kernels; read them with vh_check.
 *
 * Errors: as vh_scan_forward; VH_ERR_UNSUPPORTED for control_flags != 0, w_query or
 * skip (the ablation switches and the VisionHOPE-exact readout have no backward);
 * VH_ERR_WORKSPACE for a missing, small or misaligned workspace.
 */
vh_status vh_scan_backward(const void *x, const float *memories0, const vh_params *p, int H,
                           int W, unsigned dirs, int chunk, const float *dout,
                           const float *dmem_final, float *dx, float *dmem0);

/* Bytes of device workspace vh_scan_backward needs for these parameters: per scan
 * (image, enabled route, head) the boundary states of its chunks and, for its longest
 * chunk, a d^2 gain slice per four tokens and 4d + 24 floats per token; where the
 * tensor-core forward applies, also 3d + 8 floats per token of the whole scan.  0 for
 * invalid arguments. */
size_t vh_backward_workspace_size(const vh_params *p, int H, int W, unsigned dirs, int chunk);

/*
 * The VisionHOPE block around the operator ("VisionHOPE" Sec. 2.3 Eq. (27), App. B.5),
 * inference, NHWC:
 *   X0 = X + CPE(X);  U = Proj_in(LN1(X0));  Z = U + SiLU(DW(U));
 *   Y = F_VH(Z) + DW_pos(Z);  X1 = X0 + Proj_out(Y);  out = X1 + FFN(LN2(X1)),
 * FFN(a) = W_ff2 GELU(W_ff1 a + b_ff1) + b_ff2 (exact erf GELU).  CPE, DW and DW_pos are
 * 3 x 3 depthwise convolutions with zero padding and a bias per channel; LN normalises
 * the D channels of each pixel (biased variance, ln_eps) with a scale and shift per
 * channel.  The pages fix the structure only; these forms are this library's readings.
 * All pointers are device pointers owned by the caller.
 */
typedef struct {
    int dim;                   /* D, block width (channels of x and out), multiple of 8, <= 1024 */
    int hidden;                /* FFN width (4 D in the pages' models), multiple of 8 */
    float ln_eps;              /* LayerNorm epsilon (1e-5 if 0) */
    const float *cpe_w, *cpe_b;      /* [D][3][3], [D] */
    const float *ln1_g, *ln1_b;      /* [D] */
    const void *w_in;                /* bf16 [D_m][D], D_m = vh_params.channels */
    const float *b_in;               /* [D_m] */
    const float *dw_w, *dw_b;        /* [D_m][3][3], [D_m]: gated depthwise branch */
    const float *pos_w, *pos_b;      /* [D_m][3][3], [D_m]: positional branch */
    const void *w_out;               /* bf16 [D][D_m] */
    const float *b_out;              /* [D] */
    const float *ln2_g, *ln2_b;      /* [D] */
    const void *w_ff1;               /* bf16 [hidden][D] */
    const float *b_ff1;              /* [hidden] */
    const void *w_ff2;               /* bf16 [D][hidden] */
    const float *b_ff2;              /* [D] */
    int f32_intermediates;           /* test mode (0 = off): 1 keeps every intermediate in
                                        fp32 -- the LN outputs, Z, Y and the FFN's hidden
                                        layer are never rounded to bf16.  The GEMMs then take
                                        each fp32 activation as its three bf16 pieces
                                        (24 significant bits) against the bf16 weights
                                        repeated three times along K, and the operator runs
                                        on fp32 Z (CUDA-core scan).  Slower, and a larger
                                        workspace; it exists so the block can be compared
                                        element by element with an oracle that rounds
                                        nothing. */
} vh_block_weights;

/*
 * vh_block_forward -- one block.  x, out: device fp32 [B][H][W][D], 16-byte aligned, not
 * aliased.  p describes the operator on the internal width: p->batch = B,
 * p->channels = D_m, p->head_dim, p->x_dtype must be VH_DTYPE_BF16 (Z is bf16), and the
 * operator's optional inputs as in vh_scan_forward (w_query, skip, dir_scale, stats,
 * impl, gate and step-control constants); the operator runs all four routes with
 * row/column-aligned chunks.  p->workspace must hold vh_block_workspace_size() bytes,
 * 16-byte aligned: the block's intermediates and the operator's query planes.
 * Activations between layers are bf16 (LN outputs, Z, Y, the FFN's hidden layer before
 * and after GELU; fp32 throughout with w->f32_intermediates); the residual stream is
 * fp32.  p->accumulate and p->memories_out must be 0 / NULL.
 *
 * The four pointwise layers run as the library's own tcgen05 GEMMs (bf16 operands, fp32
 * accumulation in TMEM) with the bias, the residual and (FFN1) the GELU in their
 * epilogues.  Errors: as vh_scan_forward, plus VH_ERR_CUDA for a GEMM launch failure.
 */
vh_status vh_block_forward(const float *x, const float *memories0, const vh_params *p,
                           const vh_block_weights *w, int H, int W, float *out);

/* Bytes of workspace vh_block_forward needs; 0 for invalid arguments. */
size_t vh_block_workspace_size(const vh_params *p, const vh_block_weights *w, int H, int W);

/*
 * vh_scan_forward_static -- vh_scan_forward with the outer-query readout (p->w_query set)
 * for callers that cannot allocate device memory.  The paper has no counterpart: this is
 * a packaging of the same computation.  Some callers can't call cudaMalloc or keep a
 * workspace of their own -- a plug-in inside a host application that owns every device
 * allocation, for instance -- yet the outer-query readout needs scratch for its query
 * planes.  Here that scratch is a 16 MiB array compiled into the library (every GPU that
 * loads the library holds it until the process exits), so B*H*W*channels may be at most
 * 2,796,202 (6 bytes per element); larger calls return VH_ERR_WORKSPACE.  p->workspace
 * and p->workspace_bytes are ignored; everything else is as in vh_scan_forward, whose
 * kernels run.  Every call looks up the array's device address in the current context (so
 * a device reset that moves the array is harmless); the first call on a device also loads
 * the library's device code there, so make it before any stream capture.  Every call
 * uses the same array and
 * rewrites it completely before reading it, so nothing needs clearing, but two calls
 * that overlap on the GPU (different streams, or another thread) race on it and corrupt
 * each other's queries: serialise them.  Without w_query it returns VH_ERR_INVALID_ARG
 * (vh_scan_forward needs no scratch then).
 */
vh_status vh_scan_forward_static(const void *x, const float *memories0, const vh_params *p,
                                 int H, int W, unsigned dirs, int chunk, float *out);

/* Static string for a status code. */
const char *vh_status_string(vh_status s);

/* Thread-local description of the last failure on this thread ("" if none). */
const char *vh_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int vh_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VH_H_ */
