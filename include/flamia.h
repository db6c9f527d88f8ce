/*
 * flamia.h -- C ABI of the GB300 (sm_103a) FLAMIA attention library.
 *
 * Causal flash attention forward + backward for training with microscaled FP8
 * operands, following "FLAMIA: FLAsh MIcroscaling Attention for Fast and
 * Causally Safe Training on Blackwell" (arXiv 2611.03344) as described by the
 * FLAMIA technical review (English, sections 2-7, Algorithms 1 and 2) and the
 * Korean review (jaehun.me, section 3).
 *
 * Conventions for every entry point
 *  - All tensor arguments are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or retains them, and keeps no global state beyond
 *    a cached driver entry point (and, for flamia_bwd_static_scratch, its
 *    static device scratch array and that array's per-device address).  Every call is asynchronous on `stream`
 *    (a cudaStream_t passed as void*; NULL = legacy default stream) and never
 *    synchronises the host (the plan, quantize, forward and backward calls
 *    of a training call are replayed as a CUDA graph by the benchmark).
 *  - Packed variable-length batches: `cu_seqlens` (device, int32, num_seqs+1
 *    entries, cu[0] = 0, non-decreasing, cu[num_seqs] <= total_tokens).
 *    Document n holds tokens [cu[n], cu[n+1]).  Tokens at or after
 *    cu[num_seqs] belong to no document: their codes are 0, scale bytes 127,
 *    outputs and gradients 0 and LSE +inf.  (FLAMIA review section 6,
 *    "Preserve the logical row before optimizing the physical tile".)
 *  - Activations are row-major [total_tokens, heads, head_dim], head_dim
 *    contiguous; bf16 in, bf16 out.  head_dim must be 64 or 128.
 *  - GQA: hq query heads share hkv key/value heads, hq % hkv == 0; query head
 *    h reads kv head h / (hq / hkv).
 *  - Return value: FLAMIA_OK (0) or a negative FLAMIA_ERR_* code; on error
 *    nothing is launched.  Errors found on the device (malformed cu_seqlens,
 *    a bounded wait that timed out) set bits in the plan's status word, read
 *    back with flamia_get_device_status().
 */
#ifndef FLAMIA_H_
#define FLAMIA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------- status codes */
#define FLAMIA_OK 0
#define FLAMIA_ERR_INVALID_ARG (-1)   /* null pointer, negative size, bad count */
#define FLAMIA_ERR_UNSUPPORTED (-2)   /* head_dim not 64/128, hq % hkv != 0, too many tokens, a window with
                                         the strict options or the mixed route */
#define FLAMIA_ERR_MISALIGNED (-3)    /* a tensor pointer is not 16-byte aligned */
#define FLAMIA_ERR_WORKSPACE (-4)     /* workspace / plan buffer too small */
#define FLAMIA_ERR_CUDA (-5)          /* a CUDA launch or driver call failed */

/* device status bits (plan status word) */
#define FLAMIA_DEV_BAD_CU_SEQLENS 1   /* cu[0] != 0, decreasing, or cu[N] > total_tokens */
#define FLAMIA_DEV_TIMEOUT 2          /* a bounded mbarrier wait expired; outputs invalid */
#define FLAMIA_DEV_CAPACITY 4         /* more work items than the plan was sized for */

/* ----------------------------------------------------------- options */
typedef struct flamia_options {
  /* Boost beta = 2^p_boost_log2 applied to forward probabilities before E4M3
     rounding, with the retained row maximum exact (tau = 0), so beta * 2^tau
     = 256 <= 448 (FLAMIA review section 5, "A range budget for probability
     quantization").  Only 8 is supported. */
  int p_boost_log2;
  /* Boost of the backward probability operand of dV = P^T dO (same section;
     the value is stripped on the page, read as 2^8).  Only 8 is supported. */
  int bwd_p_boost_log2;
  /* dQ FP16 partial boost target: c = 2^floor(log2(2^headroom / M)) per
     (document, query head) (FLAMIA review section 4, "Forward locality and
     backward locality differ").  Default 14. */
  int dq_headroom_log2;
  /* Strict options (FLAMIA review section 4, "Strict options"; Korean review
     section 4.5).  Set all three together, or none (a partial set returns
     FLAMIA_ERR_UNSUPPORTED):
       strict_per_token: Q, K, V and dO carry one UE8M0 scale per token (quantize
         them with per_token = 1; flamia_bwd encodes dO per token itself).  Each
         per-token scale of a contraction-axis operand is folded into the
         companion operand (the probabilities for P V and dV, dS for dK and dQ),
         which is E4M3-rounded with one round-up exponent per (row, document-
         local 32-token group);
       strict_row_ds: dQ uses one dS exponent per (query row, 32-key block);
       strict_causal_dq: the dQ boost is per query row, from prefix maxima
         (c_i = 2^floor(log2(2^headroom / M_i)), M_i = 2 ||dO^_i||
         max_{j<=i} ||V^_j|| max_{j<=i,d} |K^_jd|).
     With them, the dQ partials are summed in increasing key-tile order by one
     CTA per query tile (no atomics): results are bitwise reproducible and a
     later token never changes an earlier row's O, LSE or dQ.
     Documents of any length are supported (the forward reads the per-key
     scale bytes of key tiles past its shared-memory table from global memory).
     deterministic: accepted only with the strict set (which implies it).
     mixed_nvfp4: the mixed NVFP4/FP8 route (head_dim 128 only; not with the
     strict options): scores and their backward recomputation from NVFP4 Q and
     K (opt->mixed), diagonal key tiles of the forward with per-key V scales
     folded into P. */
  int strict_per_token;
  int strict_row_ds;
  int strict_causal_dq;
  int mixed_nvfp4;
  int deterministic;
  /* Optional profiling hook (NULL = off): cudaEvent_t handles, two per internal
     launch.  The call records timing_events[2i] just before and
     timing_events[2i+1] just after its i-th launch, on its stream.
     flamia_fwd: launch 0 = attention forward kernel.  flamia_bwd: 0 = dO
     encoding with D (backward prep), 1 = dQ boosts, 2 = attention backward
     kernel, 3 = dQ finalisation (strict: the ordered dQ kernel and the zeroing
     of rows outside every document).  The events are caller-owned. */
  void* const* timing_events;
  /* Mixed route operands (required when mixed_nvfp4 = 1, else ignored). */
  const struct flamia_mixed_operands* mixed;
  /* Diagnostic output of flamia_bwd (NULL = off), for checking the centred
     softmax gradient (FLAMIA review section 2, "The softmax gradient is a
     centered product"; section 5, "An error decomposition for the centering
     term"): device float [2, hq, T, T], caller-zeroed.  Slice 0 receives the
     recomputed P_ij = exp(S_ij - LSE_i) and slice 1 dS_ij = P_ij (dP_ij - D_i),
     both fp32 before any quantization, at [query token][key token] for every
     visible pair (other entries are left untouched).  Default route only
     (not strict, not mixed) and total_tokens <= 1024, else
     FLAMIA_ERR_UNSUPPORTED.  A slower build of the backward kernel runs. */
  float* debug_p_ds;
  /* Visible keys: query i sees key j of its document (document-local
     positions) iff i - window_left <= j <= i + window_right; a negative value
     means no limit on that side (default -1, -1).  With causal = 1 the right
     bound is 0 whatever window_right holds, so the defaults give plain causal
     attention and, with causal = 0, attention over the whole document (the
     packed noncausal calls the FLAMIA review reports beside the causal ones,
     section 8).  Other values give sliding windows.  The strict options and
     the mixed route are causal only (a window there returns
     FLAMIA_ERR_UNSUPPORTED).  Bounds of total_tokens or more count as no
     limit. */
  int window_left;
  int window_right;
  /* Q and K were quantized with flamia_quantize_hadamard (each token row
     multiplied by H / 2^k, H the +-1 Sylvester Hadamard matrix of order
     head_dim, k = ceil(log2(head_dim) / 2); FLAMIA review section 3,
     "Rotation, range, and the alternative").  The exact score is unchanged up
     to the factor head_dim / 4^k, which the call folds into the softmax scale;
     the same rotated codes serve the gradient products, and dQ and dK are
     rotated back (by the same map) before their bf16 rounding.  V and dO are
     not rotated.  Default 0; the strict options and the mixed route do not
     take it (FLAMIA_ERR_UNSUPPORTED). */
  int rotate;
  /* Work acquisition of flamia_fwd (FLAMIA review section 6, Algorithm 2):
     0 (default) = static: the cost-sorted (work item, query head) units are
     dealt to one persistent CTA per SM in boustrophedon order (step 06);
     1 = dynamic: the grid holds a CTA per possible unit, and a running CTA,
     right after issuing the last K/V load of a unit, cancels the launch of a
     CTA that has not started (cluster launch control) and takes the next unit
     of the cost-sorted list in its stead (steps 07 and 09).  Results are
     identical either way.  Used by causal MXFP8 calls (not strict, not mixed,
     no window); other calls take the static order.  0 or 1, else
     FLAMIA_ERR_UNSUPPORTED. */
  int dynamic_schedule;
} flamia_options;

/* Operands of the mixed NVFP4/FP8 route (FLAMIA review section 2, "The mixed
   route quantizes Q and K again in E4M3 for the gradient products"; Korean
   review section 3.1: only the Q and K used by the scores and their
   recomputation are stored as NVFP4).  All device pointers, 16-byte aligned.
   The E4M3 token-block q, k, v views of flamia_fwd / flamia_bwd stay in use
   for every other product. */
typedef struct flamia_mixed_operands {
  const void* q_codes_e2m1;   /* uint8 [T, hq, head_dim/2]: two E2M1 codes per byte,
                                 element 2k in the low nibble (flamia_quantize_nvfp4) */
  const void* q_scales_e4m3;  /* uint8 [T, hq, head_dim/16]: E4M3 scale per 16 elements */
  const void* k_codes_e2m1;   /* uint8 [T, hkv, head_dim/2] */
  const void* k_scales_e4m3;  /* uint8 [T, hkv, head_dim/16] */
  const void* v_tok_codes;    /* uint8 E4M3 [T, hkv, head_dim]: V quantized per token
                                 (flamia_quantize_tokenblock with per_token = 1); the
                                 forward reads it on diagonal key tiles only (reading
                                 C-8: per-key V scales folded into P there) */
  const void* v_tok_scales;   /* uint8 UE8M0 [T, hkv] */
} flamia_mixed_operands;

/* Fill *opt with the defaults above (p_boost_log2 = 8, bwd_p_boost_log2 = 8,
   dq_headroom_log2 = 14, window_left = window_right = -1, everything else
   0 / NULL). */
void flamia_default_options(flamia_options* opt);

/* ----------------------------------------------------------- quantized tensor view */
typedef struct flamia_qtensor {
  const void* codes;    /* uint8 E4M3 codes [T, H, head_dim] */
  const void* scales;   /* uint8 UE8M0 scale bytes [T, H]; value 2^(byte-127),
                           replicated over the tokens of each document-local
                           32-token block (dense per-token metadata) */
  const float* stats;   /* float2 [T, H]: (||x^_t||_2, max_d |x^_td|) of the
                           reconstructed row, or NULL (required for k and v in
                           flamia_bwd: the dQ boost reads them) */
} flamia_qtensor;

/* ----------------------------------------------------------- plan (work list)
 * Algorithm 2 of the FLAMIA review ("Document-local work list and launch"),
 * built on the GPU once per microbatch without a host synchronisation:
 *   - per-document prefix counts of 32-token blocks and 128-token tiles;
 *   - forward items: up to 2 query tiles (256 queries) of one document, cost =
 *     visible 128-key tiles summed over the item's query tiles, sorted by
 *     decreasing cost (ties keep document order, then query order);
 *   - backward items: one per document-local 128-key tile, cost = number of
 *     query tiles that see it, sorted the same way.
 * Layout of the plan buffer (int32 words, all offsets in words):
 *   [0]  status bits (FLAMIA_DEV_*)         [1]  num_seqs
 *   [2]  total_tokens                         [3]  valid tokens = cu[num_seqs]
 *   [4]  number of 32-token blocks            [5]  number of 128-token tiles
 *   [6]  number of forward items              [7]  number of backward items
 *   [8]  capacity (items)                     [16 ...] blk_prefix[num_seqs+1]
 *   then tile_prefix[num_seqs+1] and item_prefix[num_seqs+1], then (16-byte
 *   aligned) forward items as int4 {doc, first query tile, query tile count,
 *   cost} x capacity, then backward items as int4 {doc, key tile, cost, 0} x
 *   capacity, then each backward item's document as int2 {first token, length}
 *   x capacity, the same for each forward item, then the sort scratch.
 * Ownership: caller-allocated device memory of flamia_plan_bytes() bytes,
 * 16-byte aligned; it must stay valid until every call using it completed. */
size_t flamia_plan_bytes(int64_t total_tokens, int num_seqs);
int flamia_plan_build(const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, void* plan,
                      size_t plan_bytes, void* stream);
/* The same plan with costs for the given visible-key window (causal, and
   window_left / window_right as in flamia_options): forward items cost the key
   tiles their query tiles see, backward items the query tiles that see them.
   flamia_plan_build equals causal = 1 with no left bound.  The item sets do not
   depend on the window, so any plan of the same cu_seqlens gives correct
   results; a plan built for the call's own window orders the work best. */
int flamia_plan_build_window(const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int causal,
                             int window_left, int window_right, void* plan, size_t plan_bytes, void* stream);

/* ----------------------------------------------------------- quantizer (a1)
 * Token-block MXFP8 quantizer (FLAMIA review section 3, "Why one shared
 * exponent can serve two reductions"; section 4 for the exponent rule; Korean
 * review sections 3.1-3.2; Algorithm 1 step 03).  For each document, head and
 * document-local block of 32 consecutive tokens (per_token != 0: of 1 token,
 * the strict option of review section 4):
 *   amax = max |x| over the block x head_dim,
 *   e    = smallest integer with amax <= 448 * 2^e (0 for an all-zero block),
 *          clamped to [-127, 127],
 *   code = E4M3(x * 2^-e), round to nearest even, saturating,
 *   scale byte = e + 127, written for every token of the block.
 * x: bf16 [T, heads, head_dim] (device).  codes: uint8 [T, heads, head_dim];
 * scales: uint8 [T, heads]; stats: float2 [T, heads] (||x^_t||_2, max |x^_t|)
 * or NULL.  `plan` must have been built from the same cu_seqlens.  Codes and
 * scale bytes are bit-exact with the oracle.  Non-finite inputs are not
 * supported (their codes are unspecified). */
int flamia_quantize_tokenblock(const void* x_bf16, int64_t total_tokens, int heads, int head_dim,
                               const int32_t* cu_seqlens, int num_seqs, const void* plan, int per_token,
                               void* codes_e4m3, void* scales_ue8m0, float* stats, void* stream);

/* The three flamia_quantize_tokenblock calls of a training call (Q without
 * stats, K and V with stats) in one launch.  q_bf16: [T, hq, head_dim]; k_bf16,
 * v_bf16: [T, hkv, head_dim]; outputs as in flamia_quantize_tokenblock, with the
 * same per_token rule for all three.  Results are those of the three separate
 * calls. */
int flamia_quantize_qkv(const void* q_bf16, const void* k_bf16, const void* v_bf16, int64_t total_tokens, int hq,
                        int hkv, int head_dim, const int32_t* cu_seqlens, int num_seqs, const void* plan,
                        int per_token, void* q_codes, void* q_scales, void* k_codes, void* k_scales, float* k_stats,
                        void* v_codes, void* v_scales, float* v_stats, void* stream);

/* ----------------------------------------------------------- rotated quantizer
 * flamia_quantize_tokenblock of x H / 2^k instead of x (Korean review section
 * 3.4: rotation, block statistics, codes and scales in one pass), for Q and K
 * of calls with opt->rotate = 1.  H is the +-1 Sylvester Hadamard matrix of
 * order head_dim and k = ceil(log2(head_dim) / 2) (H / 2^k is orthonormal at
 * 64 and H H / 256 = I / 2 at 128).  Each row is rotated in fp32 by the fast
 * Walsh-Hadamard butterflies, strides 1, 2, ..., head_dim / 2 in increasing
 * order, (a, b) -> (a + b, a - b); then the power of two.  Codes, scale bytes
 * and stats follow the token-block rule on the rotated values and are
 * bit-exact with the oracle.  Arguments as flamia_quantize_tokenblock without
 * per_token. */
int flamia_quantize_hadamard(const void* x_bf16, int64_t total_tokens, int heads, int head_dim,
                             const int32_t* cu_seqlens, int num_seqs, const void* plan, void* codes_e4m3,
                             void* scales_ue8m0, float* stats, void* stream);

/* ----------------------------------------------------------- NVFP4 quantizer (a2)
 * Score operands of the mixed route (FLAMIA review section 2: E2M1 codes and
 * an E4M3 scale per 16 elements; Korean review section 3.2: the scale groups
 * stay inside one token, so no document or block structure is involved).
 * Per (token, head, 16 consecutive head-dim elements), reading C-7 (no
 * tensor-level scale):
 *   s    = E4M3(amax / 6), IEEE fp32 division, round to nearest even,
 *          saturating; a non-zero group whose s rounds to 0 gets 2^-9;
 *   code = E2M1(x / s), IEEE fp32 division, round to nearest even,
 *          saturating to +-6 (0 for an all-zero group).
 * x: bf16 [T, heads, head_dim] (device).  codes_e2m1: uint8 [T, heads,
 * head_dim/2], element 2k in the low nibble of byte k; scales_e4m3: uint8
 * [T, heads, head_dim/16].  Bit-exact with the oracle.  head_dim 64 or 128;
 * x and codes 16-byte aligned. */
int flamia_quantize_nvfp4(const void* x_bf16, int64_t total_tokens, int heads, int head_dim, void* codes_e2m1,
                          void* scales_e4m3, void* stream);

/* ----------------------------------------------------------- forward (a4-a6)
 * Algorithm 1 steps 04-08 of the FLAMIA review.  For each document, query
 * head and document-local 128-query tile, over the visible document-local
 * 128-key tiles in increasing order:
 *   S   = (scale * s_Q(i) * s_K(j)) * sum_d c_Q[i,d] c_K[j,d]   (E4M3 MMA
 *         without block scales; row/column factors applied afterwards --
 *         review section 3, "Factoring the scales out of the score MMA"),
 *         keys after the query masked,
 *   m   = running row max (exact), p = exp(S - m), l = running sum of p,
 *   P^  = E4M3(2^8 p), O += P^ V^ / 2^8 (MXFP8 block-scaled MMA, V's token-
 *         block scale per 32 keys),
 * then O = bf16(O / l) and LSE = m + ln l (natural log).
 * With causal = 0 (or a window in opt) the key tiles are those the query
 * tile's window sees, and every tile holding a hidden pair or keys past the
 * document end is masked element by element.
 * q, k, v: quantized views (stats unused here).  out: bf16 [T, hq, head_dim];
 * lse: float [hq, T].  causal: 1 (keys up to the query) or 0.  softmax_scale
 * <= 0 selects 1/sqrt(head_dim).  opt may be NULL (defaults). */
int flamia_fwd(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v,
               const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int hq, int hkv, int head_dim,
               int causal, float softmax_scale, const flamia_options* opt, const void* plan, void* out_bf16,
               float* lse, void* stream);

/* ----------------------------------------------------------- backward (a7-a12)
 * Algorithm 1 steps 09-16 of the FLAMIA review:
 *   dO^ = token-block E4M3 encoding of dO (encoded once), D_i = dO^_i . O_i
 *   (saved bf16 O; Korean review section 3.3), dQ boost c per (document,
 *   query head) = 2^floor(log2(2^14 / M)) with M = 2 max||dO^_i|| max||V^_j||
 *   max|K^_jd|; then per document-local key tile and every query tile that
 *   sees it: S recomputed exactly as the forward, P = exp(S - LSE),
 *   dP = dO^ V^T, dS = P o (dP - D), dS^ = E4M3 with one round-up exponent per
 *   document-local 32x32 block, dV += (E4M3(2^8 P)/2^8)^T dO^,
 *   dK += dS^^T Q^, dQ partial = fp16(c * dS^ K^) reduce-added into an fp16
 *   accumulator; finally dQ = bf16(scale * acc / c), dK = bf16(scale * dK),
 *   dV = bf16(dV).
 * k and v need stats (from flamia_quantize_tokenblock).  out/lse: the
 * forward's outputs; dout: bf16 [T, hq, head_dim].  dq: bf16 [T, hq, head_dim];
 * dk, dv: bf16 [T, hkv, head_dim].  workspace: device scratch of at least
 * flamia_bwd_workspace_bytes() bytes, 256-byte aligned, owned by the caller
 * (holds the dO codes, scales and stats, D, the boosts and the fp16 dQ
 * accumulator; contents on return are unspecified). */
size_t flamia_bwd_workspace_bytes(int64_t total_tokens, int num_seqs, int hq, int hkv, int head_dim);
int flamia_bwd(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v, const void* out_bf16,
               const float* lse, const void* dout_bf16, const int32_t* cu_seqlens, int num_seqs,
               int64_t total_tokens, int hq, int hkv, int head_dim, int causal, float softmax_scale,
               const flamia_options* opt, const void* plan, void* dq_bf16, void* dk_bf16, void* dv_bf16,
               void* workspace, size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------- backward without allocation
 * No counterpart in the paper: a library convenience.
 * flamia_bwd for callers that cannot allocate device memory (for example a
 * plugin whose host framework hands it only input and output buffers, or a
 * latency-critical loop that must avoid cudaMalloc's device-wide
 * synchronisation).  Same arguments and results as flamia_bwd minus the
 * workspace: the scratch is a file-scope device array of
 * FLAMIA_STATIC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits.  Problems whose flamia_bwd_workspace_bytes() exceeds it
 * are rejected with FLAMIA_ERR_WORKSPACE before anything is launched.  The
 * first call on each device resolves the array's address (cudaGetSymbolAddress,
 * with that device current) and caches it.  The cached address is only valid for the device's current
 * context: after cudaDeviceReset on that device do not call this function
 * again in the same process.  The call allocates nothing.  All calls share the array:
 * calls whose GPU work overlaps race and give wrong results; the fp16 dQ
 * accumulator is cleared by every call. */
#define FLAMIA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
int flamia_bwd_static_scratch(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v,
                              const void* out_bf16, const float* lse, const void* dout_bf16,
                              const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int hq, int hkv,
                              int head_dim, int causal, float softmax_scale, const flamia_options* opt,
                              const void* plan, void* dq_bf16, void* dk_bf16, void* dv_bf16, void* stream);

/* ----------------------------------------------------------- status */
/* Copy the plan's device status word into *status_out (synchronises `stream`). */
int flamia_get_device_status(const void* plan, int* status_out, void* stream);
/* Static string for a FLAMIA_OK / FLAMIA_ERR_* code. */
const char* flamia_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* FLAMIA_H_ */
