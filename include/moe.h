/*
 * moe.h -- C ABI of the GB300 MoE layer hot path (route, dispatch, grouped
 * SwiGLU expert FFN, combine, and the layer's forward and backward).
 *
 * Method: "Enabling trillion-parameter models on AWS EFA" (Licker, Hu,
 * Zaytsev, Chen; 2025).  Section "Introduction": an MoE layer routes each token
 * to a few experts with a small linear router; dispatch groups tokens by
 * expert and combine, its dual, brings the expert outputs back and takes their
 * weighted average.  Section "Send and receive buffers": T tokens, each routed
 * to R of E experts.  Section "Dispatch and combine": per-expert counts and a
 * cumulative sum give the offsets that pack each expert's tokens contiguously
 * for the grouped GEMM.  Here everything runs on one GPU; the page's
 * network send/receive halves have no counterpart.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates device memory and never synchronises, unless MOE_CHECK is
 *    passed (then the call waits for its own work and reads the device error
 *    word back).  Work is enqueued on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream).
 *  - bf16 tensors cross the ABI as raw uint16_t bit patterns.  All tensors are
 *    dense row-major; every pointer must be 16-byte aligned and d, f must be
 *    multiples of 8 (rows move as 16-byte vectors), else MOE_ERR_UNSUPPORTED.
 *  - Shapes: T tokens, hidden size d, E experts, top-R routing, expert FFN
 *    width f, N = T*R routed rows.  A "slot" is s = t*R + r (token t, choice r).
 *    Limits: 1 <= R <= 32, R <= E <= 1024, T*R < 2^31.
 *  - Weight layout (nn.Linear [out, in]): W1, W3 bf16 [E, f, d]; W2 bf16
 *    [E, d, f]; the router weight W_g is fp32 [d, E], its bias fp32 [E].
 *  - Workspace: calls that need scratch memory take (ws, ws_bytes).  With
 *    ws == NULL the call only writes the required size to *ws_bytes and
 *    returns MOE_OK.  Otherwise *ws_bytes must be at least that size and ws
 *    256-byte aligned; the workspace must not be shared by calls that may run
 *    concurrently.
 *  - Errors: host-side argument checks return MOE_ERR_INVALID_ARG /
 *    MOE_ERR_UNSUPPORTED / MOE_ERR_WORKSPACE before anything is enqueued; a
 *    failed launch returns MOE_ERR_CUDA.  Kernels that detect bad routing
 *    (expert index outside [0,E) or repeated within a token) or a stalled
 *    pipeline wait set bits in a device error word inside the workspace and
 *    never trap; with MOE_CHECK the call returns MOE_ERR_BAD_ROUTING or
 *    MOE_ERR_TIMEOUT from it.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size */
  MOE_ERR_UNSUPPORTED = 2,   /* misaligned pointer, d or f not a multiple of 8, limits */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned */
  MOE_ERR_BAD_ROUTING = 4,   /* device saw an expert index outside [0,E) or a repeat */
  MOE_ERR_TIMEOUT = 5,       /* a bounded pipeline wait gave up (kernel returned early) */
  MOE_ERR_CUDA = 6           /* a CUDA runtime call or launch failed */
} moe_status_t;

typedef void* moe_stream_t;  /* cudaStream_t */

/* flags */
#define MOE_LOGITS_IN 0x1u   /* moe_route: `logits` is an input; skip the gate projection */
#define MOE_CHECK 0x2u       /* wait for the call's work and report device-side errors */
#define MOE_WEIGHTS_PREPACKED 0x4u  /* moe_grouped_ffn / moe_layer_fwd: W1, W3, W2 are the
                                       tiles written by moe_prepack_weights */
#define MOE_SINGLE_CTA_TILES 0x8u   /* moe_grouped_ffn / moe_layer_fwd / moe_layer_bwd: run
                                       the expert GEMMs on single-CTA 128-row tiles instead
                                       of 256-row tiles on CTA pairs (same results, bit for
                                       bit; for comparison) */
#define MOE_SHARED_SERIAL 0x10u     /* moe_layer_fwd / moe_layer_bwd: run the shared expert on the
                                       caller's stream after the routed path instead of on the
                                       library's side stream beside it (same results, bit for
                                       bit; for comparison) */
#define MOE_FP8_DISPATCH 0x20u      /* moe_layer_fwd: dispatch the tokens in block-scaled fp8
                                       (as moe_dispatch_fp8) and give the grouped FFN their
                                       dequantised rows (as moe_dequant_fp8), which saved->x_perm
                                       keeps (a backward treats the quantisation as the
                                       identity); needs d % 128 == 0 and a workspace queried
                                       with this flag */
#define MOE_FP8_MX 0x40u            /* moe_layer_fwd: run the expert FFN on the fp8 tensor cores
                                       in the microscaled fp8 format (moe_dispatch_mx, then
                                       moe_grouped_ffn_mx on layer->mx's weights); saved->o gets
                                       the expert outputs, saved->x_perm, h, a and b are not
                                       written (may be NULL) and moe_layer_bwd does not apply;
                                       needs d, f multiples of 128 and a workspace queried with
                                       this flag */

/* Stages of moe_layer_fwd / moe_layer_bwd, for moe_trace_events. */
typedef enum {
  MOE_STAGE_GATE = 0,      /* router projection (logits) */
  MOE_STAGE_TOPK,          /* softmax top-R */
  MOE_STAGE_DISPATCH,      /* histogram, scan, stable rank, row copies */
  MOE_STAGE_GATEUP,        /* tile list + grouped x W1^T | x W3^T with the SwiGLU epilogue */
  MOE_STAGE_DOWN,          /* grouped h W2^T */
  MOE_STAGE_COMBINE,       /* weighted gather-sum */
  MOE_STAGE_BWD_ROUTE,     /* dw, do, router logit gradient */
  MOE_STAGE_BWD_DH,        /* tile list + grouped do W2 with the SwiGLU backward epilogue */
  MOE_STAGE_BWD_DX,        /* grouped [da|db] [W1;W3] */
  MOE_STAGE_BWD_WG2,       /* dW2 = do^T h per expert */
  MOE_STAGE_BWD_WG13,      /* [dW1;dW3] = [da|db]^T x_perm per expert */
  MOE_STAGE_BWD_DWG,       /* router weight gradient */
  MOE_STAGE_BWD_DXC,       /* W_g transpose + dx gather-sum */
  MOE_STAGE_SHARED_FWD,    /* shared expert forward (side stream unless MOE_SHARED_SERIAL) */
  MOE_STAGE_SHARED_BWD,    /* shared expert backward (same stream rule) */
  MOE_STAGE_COUNT
} moe_stage_t;

/*
 * moe_trace_events -- per-stage timing (utility; the page has no counterpart).
 * events: NULL to disable, else 2*MOE_STAGE_COUNT cudaEvent_t handles created
 * by the caller on the current device; while set, moe_layer_fwd and
 * moe_layer_bwd record events[2*i] on their stream just before stage i and
 * events[2*i+1] just after it (the shared-expert stages on the stream that
 * runs them).  The pointer is kept (not copied) until the
 * next call; one setting is shared by all threads of the process.
 */
moe_status_t moe_trace_events(void* const* events);

/* Number of CUDA kernels this library has launched in this process (utility). */
unsigned long long moe_kernel_launches(void);

/*
 * moe_selftest_wait_timeout -- failure-detection self-test (utility; the page
 * has no counterpart).  Launches one small block whose pipeline wait is on an
 * mbarrier that nothing ever arrives on, through the same bounded-wait routine
 * the GEMM pipelines use, with a limit of limit_us microseconds (1..10^6).  The
 * wait gives up, the kernel records the timeout in ws (at least 256 bytes,
 * 256-byte aligned, device memory) and returns; the call waits for it and
 * returns MOE_ERR_TIMEOUT when the timeout was detected and reported, MOE_OK if
 * the wait was (wrongly) satisfied.  The GPU context stays usable.
 */
moe_status_t moe_selftest_wait_timeout(unsigned limit_us, void* ws, moe_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

/* The cudaError_t behind the calling thread's most recent MOE_ERR_CUDA (0 if
 * none yet); for diagnostics. */
int moe_last_cuda_error(void);

/*
 * moe_route -- the router: a small linear layer scores the experts and the R
 * best are chosen for each token (section "Introduction").
 *   logits[t,e] = sum_k x[t,k] * W_g[k,e] + bias[e]        (fp32 accumulation)
 *   idx[t,0..R-1] = the R experts of largest logit, ordered by (logit desc,
 *                   expert index asc): ties go to the lower index
 *   w[t,r] = exp(l_{idx[t,r]} - l_{idx[t,0]}) / sum_s exp(l_{idx[t,s]} - l_{idx[t,0]})
 *            (softmax over the chosen experts: the weights sum to 1)
 * x: bf16 [T,d]; w_gate: fp32 [d,E]; bias: fp32 [E] or NULL.
 * logits: fp32 [T,E], written (or read, with MOE_LOGITS_IN: then x, w_gate
 * and bias are ignored and may be NULL).  topk_idx: int32 [T,R]; topk_w: fp32
 * [T,R].  Logits must be finite.
 * Workspace (two-call convention; ignored with MOE_LOGITS_IN): when d is a
 * multiple of 64 the projection runs on the tensor cores with W_g split into
 * three bf16 terms (hi + mid + lo carry its fp32 significand; products with
 * the bf16 x are exact), which needs 6*E*d bytes of workspace; otherwise an
 * fp32 FMA kernel runs and the workspace holds only the error word.
 */
moe_status_t moe_route(const uint16_t* x, const float* w_gate, const float* bias,
                       int T, int d, int E, int R, float* logits,
                       int32_t* topk_idx, float* topk_w, void* ws, size_t* ws_bytes,
                       unsigned flags, moe_stream_t stream);

/*
 * moe_dispatch -- group the routed tokens by expert (section "Dispatch and
 * combine": per-expert counts, their cumulative sum as offsets, tokens packed
 * contiguously per expert into the grouped-GEMM input).
 *   counts[e]  = #{slots s : topk_idx[s] == e}
 *   offsets    = exclusive prefix sum of counts, offsets[E] = T*R
 *   rows offsets[e] .. offsets[e+1]-1 belong to expert e, in ascending token order
 *   row_slot[row] = s,  slot_row[s] = row  (inverse maps)
 *   x_perm[row]   = x[row_slot[row] / R]   (bit copy)
 * x: bf16 [T,d] (may be NULL together with x_perm: plan only); topk_idx:
 * int32 [T,R]; counts int32 [E]; offsets int32 [E+1]; row_slot, slot_row
 * int32 [T*R]; x_perm bf16 [T*R, d].  Needs a workspace (per-block expert
 * histograms and the error word).  Deterministic: the result does not depend
 * on scheduling.
 */
moe_status_t moe_dispatch(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int R,
                          int32_t* counts, int32_t* offsets, int32_t* row_slot, int32_t* slot_row,
                          uint16_t* x_perm, void* ws, size_t* ws_bytes, unsigned flags,
                          moe_stream_t stream);

/*
 * moe_dispatch_fp8 -- dispatch in block-scaled fp8 (section "Evaluation": the
 * page dispatches tokens in block-scaled fp8 and combines in bf16).  Same plan
 * as moe_dispatch (counts, offsets, row_slot, slot_row); instead of bf16 rows
 * it writes, per row and per 128-channel block b of the row's token x_t:
 *   xscale_perm[row, b] = amax_b / 448          (fp32; amax_b = max |x_t| over the block)
 *   xq_perm[row, c]     = E4M3(x_t[c] / xscale) (OCP E4M3 codes, round to nearest
 *                                                even, saturating at +-448)
 * An all-zero block has scale 0 and zero codes; code * scale approximates x
 * within half an E4M3 step (2^-4 relative).  d must be a multiple of 128.
 * xq_perm: uint8 [T*R, d]; xscale_perm: fp32 [T*R, d/128].  Workspace as for
 * moe_dispatch.
 */
moe_status_t moe_dispatch_fp8(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E,
                              int R, int32_t* counts, int32_t* offsets, int32_t* row_slot,
                              int32_t* slot_row, uint8_t* xq_perm, float* xscale_perm, void* ws,
                              size_t* ws_bytes, unsigned flags, moe_stream_t stream);

/*
 * moe_dequant_fp8 -- out[i, c] = bf16(E4M3 value of xq[i, c] * xscale[i, c/128])
 * for N rows of width d (d a multiple of 128): the identity expert on
 * fp8-dispatched rows.  xq: uint8 [N, d]; xscale: fp32 [N, d/128]; out: bf16
 * [N, d].  No workspace.
 */
moe_status_t moe_dequant_fp8(const uint8_t* xq, const float* xscale, int N, int d, uint16_t* out,
                             moe_stream_t stream);

/*
 * moe_grouped_ffn -- the grouped GEMMs that apply each expert's weights to its
 * rows (section "MoE all-to-all over EFA"), as a SwiGLU FFN.  For every expert
 * e and row i in [offsets[e], offsets[e+1]):
 *   a = x_perm[i] W1[e]^T,  b = x_perm[i] W3[e]^T      (fp32 accumulation)
 *   h[i]   = bf16(silu(a) * b),   silu(a) = a / (1 + exp(-a))
 *   out[i] = bf16(s_i * (h[i] W2[e]^T)),   s_i = row_scale[i], or 1 when row_scale is NULL
 * x_perm: bf16 [N,d]; offsets: int32 [E+1] on the device with offsets[E] == N;
 * W1, W3: bf16 [E,f,d]; W2: bf16 [E,d,f]; row_scale: fp32 [N] or NULL -- e.g.
 * each row's gate weight, so that an unweighted moe_combine (topk_w NULL) of
 * the outputs sums already-weighted rows (the weighting moved to the expert
 * side, before the output's bf16 rounding); h: bf16 [N,f] (written, kept for
 * the backward); a_save, b_save: bf16 [N,f] or NULL (bf16(a), bf16(b) for the
 * backward); out: bf16 [N,d].  Needs a workspace (tile list, error word).
 */
moe_status_t moe_grouped_ffn(const uint16_t* x_perm, const int32_t* offsets, int N, int d, int f,
                             int E, const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                             const float* row_scale, uint16_t* a_save, uint16_t* b_save,
                             uint16_t* h, uint16_t* out, void* ws, size_t* ws_bytes,
                             unsigned flags, moe_stream_t stream);

/*
 * moe_grouped_ffn_fp8 -- moe_grouped_ffn on the block-scaled fp8 rows that
 * moe_dispatch_fp8 writes (section "Evaluation": tokens travel in
 * block-scaled fp8).  The rows are dequantised once, as moe_dequant_fp8 does
 * (bf16(code value * scale)), into the workspace, and the bf16 grouped FFN
 * runs on them: every output equals that of moe_dequant_fp8 followed by
 * moe_grouped_ffn, bit for bit, in one call.
 * xq_perm: uint8 [N, d], 16-byte aligned; xscale_perm: fp32 [N, d/128];
 * d must be a multiple of 128 (else MOE_ERR_UNSUPPORTED).  The workspace is
 * that of moe_grouped_ffn plus N * d * 2 bytes (rounded up to 256).  Every
 * other argument and the flags as for moe_grouped_ffn.
 */
moe_status_t moe_grouped_ffn_fp8(const uint8_t* xq_perm, const float* xscale_perm,
                                 const int32_t* offsets, int N, int d, int f, int E,
                                 const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                                 const float* row_scale, uint16_t* a_save, uint16_t* b_save,
                                 uint16_t* h, uint16_t* out, void* ws, size_t* ws_bytes,
                                 unsigned flags, moe_stream_t stream);

/*
 * Microscaled fp8 ("MX") operands for expert GEMMs that take fp8 directly
 * (section "Evaluation": the tokens travel as block-scaled fp8; here the
 * tensor cores multiply the fp8 codes themselves).  A matrix [rows, K] becomes
 * E4M3 codes uint8 [rows, K] and one UE8M0 scale byte per 32 consecutive
 * elements of a row along K, stored in rows of sk = 16 * ceil(K / 512) bytes
 * (K/32 bytes, padded to a multiple of 16), uint8 [rows, sk].  A block's scale
 * is 2^k with k the smallest integer such that 448 * 2^k >= the block's
 * largest magnitude (clamped to [-127, 127]; an all-zero block gets k = -127),
 * stored as k + 127; codes are the E4M3 values nearest x / 2^k, ties to even
 * (no code saturates).  value = E4M3(code) * 2^(scale - 127).
 */

/*
 * moe_quantize_mx -- codes and scales of a bf16 matrix W [rows, K] along K (K a
 * multiple of 32): codes uint8 [rows, K], scales uint8 [rows, sk].  Used once for
 * the expert weights (W1, W3 as [E*f, d]; W2 as [E*d, f]) before
 * moe_grouped_ffn_mx.  All pointers 16-byte aligned.  No workspace.
 */
moe_status_t moe_quantize_mx(const uint16_t* W, long long rows, int K, uint8_t* codes,
                             uint8_t* scales, moe_stream_t stream);

/*
 * moe_dispatch_mx -- moe_dispatch whose rows are written in the microscaled
 * fp8 format above (codes xq_perm uint8 [T*R, d], scales xscale_perm uint8
 * [T*R, sk(d)]) instead of bf16: the same plan (counts, offsets, row_slot,
 * slot_row), each token's row quantised once and copied to its R rows.
 * d must be a multiple of 128.  Workspace as for moe_dispatch.
 */
moe_status_t moe_dispatch_mx(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E, int R,
                             int32_t* counts, int32_t* offsets, int32_t* row_slot,
                             int32_t* slot_row, uint8_t* xq_perm, uint8_t* xscale_perm, void* ws,
                             size_t* ws_bytes, unsigned flags, moe_stream_t stream);

/*
 * moe_grouped_ffn_mx -- the grouped SwiGLU FFN with fp8 tensor-core GEMMs on
 * microscaled operands (tcgen05 block-scaled fp8 multiply, fp32 accumulation).
 * For every expert e and row i in [offsets[e], offsets[e+1]), with every
 * operand taken at its dequantised value:
 *   a = x_i W1[e]^T,  b = x_i W3[e]^T,  h_i = silu(a) * b           (fp32)
 *   (hq_i, hs_i) = the microscaled fp8 form of h_i along f
 *   out_i = bf16(s_i * (h~_i W2[e]^T))   h~ = dequantised h, s_i = row_scale[i] or 1
 * xq, xs: the rows (moe_dispatch_mx); W1q/W1s, W3q/W3s: [E*f, d] codes and
 * scales, W2q/W2s: [E*d, f] (moe_quantize_mx); hq uint8 [N, f] and hs uint8
 * [N, sk(f)] receive h (or NULL: kept in the workspace); out bf16 [N, d].
 * d and f must be multiples of 128 (else MOE_ERR_UNSUPPORTED).  Needs a
 * workspace (error word, tile list, and h when hq/hs are NULL).
 */
moe_status_t moe_grouped_ffn_mx(const uint8_t* xq, const uint8_t* xs, const int32_t* offsets,
                                int N, int d, int f, int E, const uint8_t* W1q,
                                const uint8_t* W1s, const uint8_t* W3q, const uint8_t* W3s,
                                const uint8_t* W2q, const uint8_t* W2s, const float* row_scale,
                                uint8_t* hq, uint8_t* hs, uint16_t* out, void* ws,
                                size_t* ws_bytes, unsigned flags, moe_stream_t stream);

/*
 * moe_prepack_weights -- copy the expert weights into the tile layout the
 * forward grouped GEMMs stream (a performance layout for forward-only use, e.g.
 * inference; the page's grouped GEMMs take the weights as they are):
 *   W1p, W3p[e][j][k][r][c] = W1, W3[e][128 j + r][64 k + c]   ([E][f/128][d/64][128][64])
 *   W2p[e][j][k][r][c]      = W2[e][256 j + r][64 k + c]       ([E][d/256][f/64][256][64])
 * so that every 128x64 (W1, W3) or 256x64 (W2) box the GEMM loads is one
 * contiguous 16 or 32 KB region.  Requires d % 256 == 0 and f % 128 == 0.
 * Pass MOE_WEIGHTS_PREPACKED to moe_grouped_ffn / moe_layer_fwd to use them
 * (same results, bit for bit); moe_layer_bwd takes the plain layout only.
 * W1p, W3p, W2p: bf16, the sizes of W1, W3, W2; must not alias them.
 */
moe_status_t moe_prepack_weights(const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, int E,
                                 int d, int f, uint16_t* W1p, uint16_t* W3p, uint16_t* W2p,
                                 moe_stream_t stream);

/*
 * moe_combine -- bring each token's R expert outputs back and take their
 * gate-weighted sum (sections "Introduction" and "Dispatch and combine"):
 *   y[t] = bf16( sum_{r=0..R-1} topk_w[t,r] * expert_out[slot_row[t*R+r]] )
 * accumulated in fp32 in r order (bitwise reproducible).  topk_w NULL means
 * unweighted.  expert_out: bf16 [T*R,d]; slot_row: int32 [T*R]; y: bf16 [T,d].
 * Rows outside [0, T*R) contribute nothing.  No workspace.
 */
moe_status_t moe_combine(const uint16_t* expert_out, const int32_t* slot_row, const float* topk_w,
                         int T, int d, int R, uint16_t* y, moe_stream_t stream);

/*
 * moe_dispatch_noalloc -- moe_dispatch without a workspace argument, for
 * callers that cannot allocate device memory: code running inside a host
 * application or framework whose allocator owns all device memory, and
 * latency-critical loops that cannot afford cudaMalloc's implicit device
 * synchronisation.  (The page has no counterpart; this is a packaging of the
 * dispatch step above.)
 * Same arguments, results and error behaviour as moe_dispatch.  Its scratch
 * (the device error word and 2*E*ceil(T/256) int32 histogram entries) lives in
 * a 4 MiB array that the library reserves statically on every GPU that loads
 * it, until the process exits; calls whose scratch would not fit
 * (256 + 8*E*ceil(T/256) bytes, rounded up to 256, above 4 MiB) return
 * MOE_ERR_WORKSPACE before anything is enqueued.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.  The first call on each device looks
 * up the array's device address (set-up; make that first call before any
 * stream capture).  Every call uses the same array and clears its error word
 * first; calls that may overlap on the GPU (different streams, or different
 * host threads) race on it and must be serialised by the caller.
 */
moe_status_t moe_dispatch_noalloc(const uint16_t* x, const int32_t* topk_idx, int T, int d, int E,
                                  int R, int32_t* counts, int32_t* offsets, int32_t* row_slot,
                                  int32_t* slot_row, uint16_t* x_perm, unsigned flags,
                                  moe_stream_t stream);

/* Layer parameters (device pointers, caller-owned). */
/*
 * Optional shared expert (section "Introduction": while dispatch is in
 * flight the GPU can do other work, such as the shared expert's
 * multiplication).  A SwiGLU FFN that every token passes through, added to
 * the routed experts' weighted sum with weight 1:
 *   s_t = bf16( bf16(silu(x_t Ws1^T) * (x_t Ws3^T)) Ws2^T ),
 *   y_t = bf16( s_t + sum_r w[t,r] o[slot_row[t*R+r]] ).
 * The forward runs it on a side stream the library owns (one per device),
 * forked from the caller's stream after the gate projection and joined before
 * combine, so it overlaps top-R and dispatch; the backward forks it at the
 * start and joins it before the dx gather.  Callers see ordinary stream
 * semantics on their stream.
 */
typedef struct {
  int fs;               /* hidden size; multiple of 8 (of 64 for the backward) */
  const uint16_t* W1;   /* bf16 [fs,d] */
  const uint16_t* W3;   /* bf16 [fs,d] */
  const uint16_t* W2;   /* bf16 [d,fs] */
  float* dW1;           /* moe_layer_bwd outputs, fp32 [fs,d], [fs,d], [d,fs]; */
  float* dW3;           /*   unused by the forward (may be NULL there)        */
  float* dW2;
} moe_shared_t;

/* The expert weights in the microscaled fp8 format (moe_quantize_mx along each
 * matrix's K): W1q, W3q uint8 [E*f, d] with scales uint8 [E*f, sk(d)]; W2q
 * uint8 [E*d, f] with scales uint8 [E*d, sk(f)]. */
typedef struct {
  const uint8_t* W1q;
  const uint8_t* W1s;
  const uint8_t* W3q;
  const uint8_t* W3s;
  const uint8_t* W2q;
  const uint8_t* W2s;
} moe_mx_weights_t;

typedef struct {
  int T, d, E, R, f;
  const float* w_gate;  /* fp32 [d,E] */
  const float* bias;    /* fp32 [E] or NULL */
  const uint16_t* W1;   /* bf16 [E,f,d] */
  const uint16_t* W3;   /* bf16 [E,f,d] */
  const uint16_t* W2;   /* bf16 [E,d,f] */
  const moe_shared_t* shared;   /* NULL: no shared expert */
  const moe_mx_weights_t* mx;   /* microscaled fp8 expert weights for MOE_FP8_MX, or NULL */
} moe_layer_t;

/* Forward intermediates (caller-owned device buffers, written by the forward,
 * read by the backward).  N = T*R. */
typedef struct {
  float* logits;       /* fp32 [T,E] */
  int32_t* topk_idx;   /* int32 [T,R] */
  float* topk_w;       /* fp32 [T,R] */
  int32_t* counts;     /* int32 [E] */
  int32_t* offsets;    /* int32 [E+1] */
  int32_t* row_slot;   /* int32 [N] */
  int32_t* slot_row;   /* int32 [N] */
  uint16_t* x_perm;    /* bf16 [N,d] */
  uint16_t* a;         /* bf16 [N,f] or NULL (inference: nothing saved for the backward) */
  uint16_t* b;         /* bf16 [N,f] or NULL (must be NULL iff a is) */
  uint16_t* h;         /* bf16 [N,f] */
  uint16_t* o;         /* bf16 [N,d] expert outputs */
  /* shared expert (only read when the layer has one): its pre-activations
   * and hidden rows for the backward, bf16 [T,fs]; all three NULL for
   * inference (the forward then keeps its hidden rows in the workspace) */
  uint16_t* sa;
  uint16_t* sb;
  uint16_t* sh;
} moe_saved_t;

/*
 * moe_layer_fwd -- y = combine(FFN(dispatch(x, route(x)))): route, dispatch,
 * grouped SwiGLU FFN and combine, as the entry points above define them.
 * x: bf16 [T,d]; y: bf16 [T,d]; saved: all intermediates (a and b may be NULL).
 * With layer->shared, y also adds the shared expert's output (moe_shared_t);
 * saved->sa, sb, sh then hold its intermediates (all NULL for inference).
 */
moe_status_t moe_layer_fwd(const moe_layer_t* layer, const uint16_t* x, uint16_t* y,
                           const moe_saved_t* saved, void* ws, size_t* ws_bytes, unsigned flags,
                           moe_stream_t stream);

/*
 * moe_layer_bwd -- gradients of a loss L given dy = dL/dy (bf16 [T,d]), from
 * the intermediates of moe_layer_fwd (which must have saved a and b):
 *   dw[t,r]  = <dy_t, o_row>,  do_row = bf16(w[t,r] dy_t)      (row = slot_row[t*R+r])
 *   per expert: dh = do W2[e];  da = bf16(dh * b * silu'(a)),  db = bf16(dh * silu(a))
 *               dx_perm = bf16(da W1[e] + db W3[e])
 *               dW2[e] = do^T h,  dW1[e] = da^T x_perm,  dW3[e] = db^T x_perm
 *   router:  dlogits[t, idx[t,q]] = w_q (dw_q - sum_r w_r dw_r), 0 for unchosen experts
 *            dW_gate = x^T dlogits
 *   dx_t = bf16( sum_r dx_perm[row(t,r)] + dlogits_t W_g^T [+ dxs_t] )
 *   shared expert (layer->shared; saved->sa, sb, sh required), with dy as its
 *   output gradient:  dhs = dy Ws2;  das = bf16(dhs * sb * silu'(sa)),
 *   dbs = bf16(dhs * silu(sa));  dxs = bf16(das Ws1 + dbs Ws3);
 *   shared->dW2 = dy^T sh,  shared->dW1 = das^T x,  shared->dW3 = dbs^T x
 * (a, b as saved in bf16; silu'(a) = s(a)(1 + a(1 - s(a))), s the logistic
 * function.)  x: bf16 [T,d]; dx: bf16 [T,d]; dW_gate: fp32 [d,E]; dW1, dW3:
 * fp32 [E,f,d]; dW2: fp32 [E,d,f] -- all overwritten (experts with no rows get
 * zero gradients).  The router bias is treated as a constant.
 */
moe_status_t moe_layer_bwd(const moe_layer_t* layer, const uint16_t* x, const moe_saved_t* saved,
                           const uint16_t* dy, uint16_t* dx, float* dW_gate, float* dW1,
                           float* dW3, float* dW2, void* ws, size_t* ws_bytes, unsigned flags,
                           moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
