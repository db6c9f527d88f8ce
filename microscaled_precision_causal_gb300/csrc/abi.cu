// extern "C" entry points of libflamia: argument validation, workspace
// layout and kernel launches.  Every function only enqueues work on the given
// stream (flamia_get_device_status is the one call that synchronises).
#include <cmath>
#include <cstdint>
#include <cstring>

#include "common.cuh"

namespace flamia {
cudaError_t launch_plan(const int32_t* cu, int N, int T, Window win, void* plan, cudaStream_t s);
cudaError_t launch_quantize(const void* x, int T, int H, int D, const int32_t* cu, int N, const void* plan,
                            int per_token, void* codes, void* scales, float* stats, const void* o, float* dvec,
                            void* dq_acc, cudaStream_t s, const float* k_stats = nullptr,
                            const float* v_stats = nullptr, int hkv = 1, float* maxima = nullptr);
cudaError_t launch_fwd(int D, const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                       const void* vs, const int32_t* cu, int N, int T, int hq, int hkv, float scale,
                       const void* plan, void* out, float* lse, cudaStream_t stream, void* const* ev, bool strict,
                       Window win, bool dynamic);
cudaError_t launch_quantize_nvfp4(const void* x, int64_t elems, void* codes, void* scales, cudaStream_t s);
cudaError_t launch_quantize_rot(const void* x, int T, int H, int D, const int32_t* cu, int N, const void* plan,
                                void* codes, void* scales, float* stats, cudaStream_t s);
cudaError_t launch_quantize_qkv(const void* q, const void* k, const void* v, int T, int hq, int hkv, int D,
                                const int32_t* cu, int N, const void* plan, int per_token, void* qc, void* qs,
                                void* kc, void* ks, float* kst, void* vc, void* vs, float* vst, cudaStream_t s);
cudaError_t launch_fwd_coop(int D, int mixed, const void* qc, const void* qs, const void* kc, const void* ks,
                            const void* vc, const void* vs, const void* q4c, const void* q4s, const void* k4c,
                            const void* k4s, const void* vtc, const void* vts, const int32_t* cu, int N, int T, int hq,
                            int hkv, float scale, const void* plan, void* out, float* lse, cudaStream_t stream);
cudaError_t launch_fwd_tail(int D, const void* plan, int T, int hq, void* out, float* lse, cudaStream_t stream);
cudaError_t launch_boost(const int32_t* cu, int N, const void* plan, const float* st_do, const float* st_k,
                         const float* st_v, int T, int hq, int hkv, int headroom, float* boost, bool causal,
                         const float* maxima, cudaStream_t s);
cudaError_t launch_bwd(int D, const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                       const void* vs, const void* doc_codes, const void* dos, const float* lse, const float* dvec,
                       const float* boost, const int32_t* cu, int N, int T, int hq, int hkv, float scale,
                       const void* plan, void* dq_acc, void* dq, void* dk, void* dv, cudaStream_t stream,
                       void* const* ev, bool strict, const void* q4c, const void* q4s, const void* k4c,
                       const void* k4s, float* dbg, Window win, bool rot);
}  // namespace flamia

using namespace flamia;

namespace {

constexpr int64_t kMaxTokens = (int64_t)1 << 26;   // row indices stay in int32 with headroom

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

int check_common(int64_t T, int N, const void* cu, const void* plan) {
  if (T < 0 || N < 0 || !cu || !plan) return FLAMIA_ERR_INVALID_ARG;
  if (T > kMaxTokens || N > kMaxTokens) return FLAMIA_ERR_UNSUPPORTED;
  if (!aligned16(plan)) return FLAMIA_ERR_MISALIGNED;
  return FLAMIA_OK;
}

// The strict options come as a set (per-token operand scales, per-query-row dS
// exponents, causal dQ boost; the dQ reduction is then deterministic).
bool is_strict(const flamia_options* o) { return o && o->strict_per_token; }

int check_opts(const flamia_options* o) {
  if (!o) return FLAMIA_OK;
  if (o->p_boost_log2 != 8 || o->bwd_p_boost_log2 != 8) return FLAMIA_ERR_UNSUPPORTED;
  if (o->dq_headroom_log2 < 1 || o->dq_headroom_log2 > 15) return FLAMIA_ERR_UNSUPPORTED;
  const int s = o->strict_per_token + o->strict_row_ds + o->strict_causal_dq;
  if (s != 0 && s != 3) return FLAMIA_ERR_UNSUPPORTED;
  if (o->deterministic && s == 0) return FLAMIA_ERR_UNSUPPORTED;
  if (o->dynamic_schedule != 0 && o->dynamic_schedule != 1) return FLAMIA_ERR_UNSUPPORTED;
  if (o->mixed_nvfp4) {
    if (s != 0) return FLAMIA_ERR_UNSUPPORTED;        // the strict options and the mixed route are separate
    const flamia_mixed_operands* m = o->mixed;
    if (!m || !m->q_codes_e2m1 || !m->q_scales_e4m3 || !m->k_codes_e2m1 || !m->k_scales_e4m3 || !m->v_tok_codes ||
        !m->v_tok_scales)
      return FLAMIA_ERR_INVALID_ARG;
    if (!aligned16(m->q_codes_e2m1) || !aligned16(m->k_codes_e2m1) || !aligned16(m->v_tok_codes) ||
        (reinterpret_cast<uintptr_t>(m->q_scales_e4m3) & 7u) || (reinterpret_cast<uintptr_t>(m->k_scales_e4m3) & 7u))
      return FLAMIA_ERR_MISALIGNED;
  }
  return FLAMIA_OK;
}

bool is_mixed(const flamia_options* o) { return o && o->mixed_nvfp4; }

int check_heads(int hq, int hkv, int d) {
  if (hq <= 0 || hkv <= 0) return FLAMIA_ERR_INVALID_ARG;
  if (hq % hkv != 0 || (d != 64 && d != 128) || hq > 1024) return FLAMIA_ERR_UNSUPPORTED;
  return FLAMIA_OK;
}

int check_qt(const flamia_qtensor* t, bool need_stats) {
  if (!t || !t->codes || !t->scales) return FLAMIA_ERR_INVALID_ARG;
  if (need_stats && !t->stats) return FLAMIA_ERR_INVALID_ARG;
  if (!aligned16(t->codes)) return FLAMIA_ERR_MISALIGNED;
  if (t->stats && (reinterpret_cast<uintptr_t>(t->stats) & 7u)) return FLAMIA_ERR_MISALIGNED;
  return FLAMIA_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA; }

inline void record(void* const* ev, int i, cudaStream_t s) {
  if (ev) record_timing_event(ev[i], s);
}

float resolve_scale(float s, int d) { return s > 0.f ? s : 1.0f / std::sqrt((float)d); }

// The call's visible-key window: causal forces the right bound to 0; negative
// values and bounds of T or more mean no limit (-1).
Window resolve_window(int causal, int left, int right, int64_t T) {
  Window w;
  w.left = (left < 0 || (int64_t)left >= T) ? -1 : left;
  w.right = causal ? 0 : ((right < 0 || (int64_t)right >= T) ? -1 : right);
  return w;
}
Window call_window(const flamia_options* o, int causal, int64_t T) {
  return resolve_window(causal, o ? o->window_left : -1, o ? o->window_right : -1, T);
}
inline bool is_causal_window(Window w) { return w.left < 0 && w.right == 0; }

bool is_rotated(const flamia_options* o) { return o && o->rotate; }
// Rotated operands: S = (d / 4^k) Q~ K~^T, folded into the softmax scale.
float score_scale(float s, int d, bool rot) { return rot ? s * (d == 128 ? 2.0f : 1.0f) : s; }

struct BwdWorkspace {
  size_t do_codes, do_scales, do_stats, dvec, boost, maxima, dq_acc, total;
};
BwdWorkspace bwd_layout(int64_t T, int N, int hq, int d) {
  BwdWorkspace w;
  size_t off = 0;
  w.do_codes = off; off = round256(off + (size_t)T * hq * d);
  w.do_scales = off; off = round256(off + (size_t)T * hq);
  w.do_stats = off; off = round256(off + (size_t)T * hq * 8);
  w.dvec = off; off = round256(off + (size_t)T * hq * 4);
  w.boost = off; off = round256(off + ((size_t)(N > 0 ? N : 1) + (size_t)T) * hq * 4);   // per doc, or per row (strict)
  w.maxima = off; off = round256(off + (size_t)(N > 0 ? N : 1) * hq * 3 * 4);   // dQ boost inputs per (doc, head)
  w.dq_acc = off; off = round256(off + dq_acc_bytes(T, N, hq, d));   // fp16 chunks per (document tile, head, slice)
  w.total = off;
  return w;
}

}  // namespace

extern "C" {

void flamia_default_options(flamia_options* opt) {
  if (!opt) return;
  std::memset(opt, 0, sizeof(*opt));
  opt->p_boost_log2 = 8;
  opt->bwd_p_boost_log2 = 8;
  opt->dq_headroom_log2 = 14;
  opt->window_left = -1;
  opt->window_right = -1;
  opt->rotate = 0;
}

size_t flamia_plan_bytes(int64_t total_tokens, int num_seqs) {
  if (total_tokens < 0 || num_seqs < 0) return 0;
  return plan_bytes(total_tokens, num_seqs);
}

int flamia_plan_build(const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, void* plan, size_t plan_bytes_,
                      void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (rc) return rc;
  if (plan_bytes_ < plan_bytes(total_tokens, num_seqs)) return FLAMIA_ERR_WORKSPACE;
  return cuda_status(launch_plan(cu_seqlens, num_seqs, (int)total_tokens, resolve_window(1, -1, -1, total_tokens), plan,
                                 (cudaStream_t)stream));
}

int flamia_plan_build_window(const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int causal,
                             int window_left, int window_right, void* plan, size_t plan_bytes_, void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return FLAMIA_ERR_INVALID_ARG;
  if (plan_bytes_ < plan_bytes(total_tokens, num_seqs)) return FLAMIA_ERR_WORKSPACE;
  return cuda_status(launch_plan(cu_seqlens, num_seqs, (int)total_tokens,
                                 resolve_window(causal, window_left, window_right, total_tokens), plan,
                                 (cudaStream_t)stream));
}

int flamia_quantize_tokenblock(const void* x_bf16, int64_t total_tokens, int heads, int head_dim,
                               const int32_t* cu_seqlens, int num_seqs, const void* plan, int per_token,
                               void* codes_e4m3, void* scales_ue8m0, float* stats, void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (rc) return rc;
  if (!x_bf16 || !codes_e4m3 || !scales_ue8m0 || heads <= 0) return FLAMIA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FLAMIA_ERR_UNSUPPORTED;
  if (!aligned16(x_bf16) || !aligned16(codes_e4m3) || (stats && (reinterpret_cast<uintptr_t>(stats) & 7u)))
    return FLAMIA_ERR_MISALIGNED;
  if (total_tokens == 0) return FLAMIA_OK;
  return cuda_status(launch_quantize(x_bf16, (int)total_tokens, heads, head_dim, cu_seqlens, num_seqs, plan,
                                     per_token, codes_e4m3, scales_ue8m0, stats, nullptr, nullptr, nullptr,
                                     (cudaStream_t)stream));
}

int flamia_quantize_qkv(const void* q_bf16, const void* k_bf16, const void* v_bf16, int64_t total_tokens, int hq,
                        int hkv, int head_dim, const int32_t* cu_seqlens, int num_seqs, const void* plan,
                        int per_token, void* q_codes, void* q_scales, void* k_codes, void* k_scales, float* k_stats,
                        void* v_codes, void* v_scales, float* v_stats, void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (!rc) rc = check_heads(hq, hkv, head_dim);
  if (rc) return rc;
  if (!q_bf16 || !k_bf16 || !v_bf16 || !q_codes || !q_scales || !k_codes || !k_scales || !v_codes || !v_scales)
    return FLAMIA_ERR_INVALID_ARG;
  auto bad8 = [](const float* p) { return p && (reinterpret_cast<uintptr_t>(p) & 7u); };
  if (!aligned16(q_bf16) || !aligned16(k_bf16) || !aligned16(v_bf16) || !aligned16(q_codes) || !aligned16(k_codes) ||
      !aligned16(v_codes) || bad8(k_stats) || bad8(v_stats))
    return FLAMIA_ERR_MISALIGNED;
  if (total_tokens == 0) return FLAMIA_OK;
  return cuda_status(launch_quantize_qkv(q_bf16, k_bf16, v_bf16, (int)total_tokens, hq, hkv, head_dim, cu_seqlens,
                                         num_seqs, plan, per_token, q_codes, q_scales, k_codes, k_scales, k_stats,
                                         v_codes, v_scales, v_stats, (cudaStream_t)stream));
}

int flamia_quantize_hadamard(const void* x_bf16, int64_t total_tokens, int heads, int head_dim,
                             const int32_t* cu_seqlens, int num_seqs, const void* plan, void* codes_e4m3,
                             void* scales_ue8m0, float* stats, void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (rc) return rc;
  if (!x_bf16 || !codes_e4m3 || !scales_ue8m0 || heads <= 0) return FLAMIA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FLAMIA_ERR_UNSUPPORTED;
  if (!aligned16(x_bf16) || !aligned16(codes_e4m3) || (stats && (reinterpret_cast<uintptr_t>(stats) & 7u)))
    return FLAMIA_ERR_MISALIGNED;
  if (total_tokens == 0) return FLAMIA_OK;
  return cuda_status(launch_quantize_rot(x_bf16, (int)total_tokens, heads, head_dim, cu_seqlens, num_seqs, plan,
                                         codes_e4m3, scales_ue8m0, stats, (cudaStream_t)stream));
}

int flamia_quantize_nvfp4(const void* x_bf16, int64_t total_tokens, int heads, int head_dim, void* codes_e2m1,
                          void* scales_e4m3, void* stream) {
  if (total_tokens < 0 || heads <= 0) return FLAMIA_ERR_INVALID_ARG;
  if (!x_bf16 || !codes_e2m1 || !scales_e4m3) return FLAMIA_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return FLAMIA_ERR_UNSUPPORTED;
  if (!aligned16(x_bf16) || !aligned16(codes_e2m1)) return FLAMIA_ERR_MISALIGNED;
  if (total_tokens == 0) return FLAMIA_OK;
  return cuda_status(launch_quantize_nvfp4(x_bf16, total_tokens * heads * head_dim, codes_e2m1, scales_e4m3,
                                           (cudaStream_t)stream));
}

int flamia_fwd(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v, const int32_t* cu_seqlens,
               int num_seqs, int64_t total_tokens, int hq, int hkv, int head_dim, int causal, float softmax_scale,
               const flamia_options* opt, const void* plan, void* out_bf16, float* lse, void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (!rc) rc = check_heads(hq, hkv, head_dim);
  if (!rc) rc = check_opts(opt);
  if (!rc) rc = check_qt(q, false);
  if (!rc) rc = check_qt(k, false);
  if (!rc) rc = check_qt(v, false);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return FLAMIA_ERR_INVALID_ARG;
  const Window win = call_window(opt, causal, total_tokens);
  if ((is_strict(opt) || is_mixed(opt)) && (!is_causal_window(win) || is_rotated(opt))) return FLAMIA_ERR_UNSUPPORTED;
  if (!out_bf16 || !lse) return FLAMIA_ERR_INVALID_ARG;
  if (!aligned16(out_bf16) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FLAMIA_ERR_MISALIGNED;
  if (is_mixed(opt) && head_dim != 128) return FLAMIA_ERR_UNSUPPORTED;
  if (total_tokens == 0) return FLAMIA_OK;
  const float scale = score_scale(resolve_scale(softmax_scale, head_dim), head_dim, is_rotated(opt));
  if (is_mixed(opt)) {
    const flamia_mixed_operands* m = opt->mixed;
    cudaStream_t s = (cudaStream_t)stream;
    record(opt->timing_events, 0, s);
    cudaError_t e = launch_fwd_coop(head_dim, 1, q->codes, q->scales, k->codes, k->scales, v->codes, v->scales,
                                    m->q_codes_e2m1, m->q_scales_e4m3, m->k_codes_e2m1, m->k_scales_e4m3,
                                    m->v_tok_codes, m->v_tok_scales, cu_seqlens, num_seqs, (int)total_tokens, hq, hkv,
                                    scale, plan, out_bf16, lse, s);
    record(opt->timing_events, 1, s);
    if (e == cudaSuccess) e = launch_fwd_tail(head_dim, plan, (int)total_tokens, hq, out_bf16, lse, s);
    return cuda_status(e);
  }
  return cuda_status(launch_fwd(head_dim, q->codes, q->scales, k->codes, k->scales, v->codes, v->scales, cu_seqlens,
                                num_seqs, (int)total_tokens, hq, hkv, scale, plan, out_bf16, lse, (cudaStream_t)stream,
                                opt ? opt->timing_events : nullptr, is_strict(opt), win,
                                opt && opt->dynamic_schedule));
}

size_t flamia_bwd_workspace_bytes(int64_t total_tokens, int num_seqs, int hq, int hkv, int head_dim) {
  (void)hkv;
  if (total_tokens < 0 || num_seqs < 0 || hq <= 0 || head_dim <= 0) return 0;
  return bwd_layout(total_tokens, num_seqs, hq, head_dim).total;
}

int flamia_bwd(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v, const void* out_bf16,
               const float* lse, const void* dout_bf16, const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
               int hq, int hkv, int head_dim, int causal, float softmax_scale, const flamia_options* opt,
               const void* plan, void* dq_bf16, void* dk_bf16, void* dv_bf16, void* workspace, size_t workspace_bytes,
               void* stream) {
  int rc = check_common(total_tokens, num_seqs, cu_seqlens, plan);
  if (!rc) rc = check_heads(hq, hkv, head_dim);
  if (!rc) rc = check_opts(opt);
  if (!rc) rc = check_qt(q, false);
  if (!rc) rc = check_qt(k, true);
  if (!rc) rc = check_qt(v, true);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return FLAMIA_ERR_INVALID_ARG;
  const Window win = call_window(opt, causal, total_tokens);
  if ((is_strict(opt) || is_mixed(opt)) && (!is_causal_window(win) || is_rotated(opt))) return FLAMIA_ERR_UNSUPPORTED;
  if (!out_bf16 || !lse || !dout_bf16 || !dq_bf16 || !dk_bf16 || !dv_bf16 || !workspace) return FLAMIA_ERR_INVALID_ARG;
  if (!aligned16(out_bf16) || !aligned16(dout_bf16) || !aligned16(dq_bf16) || !aligned16(dk_bf16) ||
      !aligned16(dv_bf16) || (reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FLAMIA_ERR_MISALIGNED;
  if (is_mixed(opt) && head_dim != 128) return FLAMIA_ERR_UNSUPPORTED;
  float* dbg = opt ? opt->debug_p_ds : nullptr;
  if (dbg && (is_mixed(opt) || is_strict(opt) || is_rotated(opt) || !is_causal_window(win) || total_tokens > 1024))
    return FLAMIA_ERR_UNSUPPORTED;
  if (dbg && (reinterpret_cast<uintptr_t>(dbg) & 3u)) return FLAMIA_ERR_MISALIGNED;
  const BwdWorkspace w = bwd_layout(total_tokens, num_seqs, hq, head_dim);
  if (workspace_bytes < w.total) return FLAMIA_ERR_WORKSPACE;
  if (total_tokens == 0) return FLAMIA_OK;
  const int headroom = opt ? opt->dq_headroom_log2 : 14;
  const int T = (int)total_tokens;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* do_codes = ws + w.do_codes;
  void* do_scales = ws + w.do_scales;
  float* do_stats = reinterpret_cast<float*>(ws + w.do_stats);
  float* dvec = reinterpret_cast<float*>(ws + w.dvec);
  float* boost = reinterpret_cast<float*>(ws + w.boost);
  float* maxima = reinterpret_cast<float*>(ws + w.maxima);
  void* dq_acc = ws + w.dq_acc;
  void* const* ev = opt ? opt->timing_events : nullptr;
  record(ev, 0, s);
  const bool strict = is_strict(opt);
  cudaError_t e = cudaSuccess;
  if (!strict) e = cudaMemsetAsync(maxima, 0, (size_t)num_seqs * hq * 3 * 4, s);
  // the fp16 dQ accumulator starts at zero: the dO quantizer clears, for each 32-token
  // block, its query rows (head_dim 64, query-major chunks) or its query columns of every
  // head-dim row (head_dim 128, head-dim-major chunks); the strict route has no accumulator
  if (e == cudaSuccess)
    e = launch_quantize(dout_bf16, T, hq, head_dim, cu_seqlens, num_seqs, plan, strict ? 1 : 0, do_codes, do_scales,
                        do_stats, out_bf16, dvec, strict ? nullptr : dq_acc, s, k->stats, v->stats,
                        hkv, strict ? nullptr : maxima);
  record(ev, 1, s);
  record(ev, 2, s);
  if (e == cudaSuccess)
    e = launch_boost(cu_seqlens, num_seqs, plan, do_stats, k->stats, v->stats, T, hq, hkv, headroom, boost, strict,
                     maxima, s);
  record(ev, 3, s);
  if (e == cudaSuccess)
    e = launch_bwd(head_dim, q->codes, q->scales, k->codes, k->scales, v->codes, v->scales, do_codes, do_scales, lse,
                   dvec, boost, cu_seqlens, num_seqs, T, hq, hkv,
                   score_scale(resolve_scale(softmax_scale, head_dim), head_dim, is_rotated(opt)), plan, dq_acc,
                   dq_bf16, dk_bf16, dv_bf16, s, ev ? ev + 4 : nullptr, strict,
                   is_mixed(opt) ? opt->mixed->q_codes_e2m1 : nullptr,
                   is_mixed(opt) ? opt->mixed->q_scales_e4m3 : nullptr,
                   is_mixed(opt) ? opt->mixed->k_codes_e2m1 : nullptr,
                   is_mixed(opt) ? opt->mixed->k_scales_e4m3 : nullptr, dbg, win, is_rotated(opt));
  return cuda_status(e);
}

int flamia_get_device_status(const void* plan, int* status_out, void* stream) {
  if (!plan || !status_out) return FLAMIA_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(status_out, plan, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(s));
}

const char* flamia_status_string(int status) {
  switch (status) {
    case FLAMIA_OK: return "ok";
    case FLAMIA_ERR_INVALID_ARG: return "invalid argument";
    case FLAMIA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FLAMIA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FLAMIA_ERR_WORKSPACE: return "workspace or plan buffer too small";
    case FLAMIA_ERR_CUDA: return "CUDA launch or driver error";
    default: return "unknown status";
  }
}

}  // extern "C"
