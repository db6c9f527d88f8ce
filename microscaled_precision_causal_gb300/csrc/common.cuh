// Shared definitions of the FLAMIA CUDA library: plan layout accessors and
// small device helpers used by several kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/flamia.h"

namespace flamia {

constexpr int kTile = 128;        // query / key tile (document-local rows)
constexpr int kBlock = 32;        // operand token block
constexpr int kItemTiles = 2;     // forward work item: up to 2 query tiles (256 queries)

// ---------------------------------------------------------------- plan layout
// int32 words; see include/flamia.h for the documented layout.
enum PlanWord : int {
  kPlanStatus = 0,
  kPlanNumSeqs = 1,
  kPlanTotal = 2,
  kPlanValid = 3,
  kPlanBlocks = 4,
  kPlanTiles = 5,
  kPlanFwdItems = 6,
  kPlanBwdItems = 7,
  kPlanCapacity = 8,
  kPlanWindowLeft = 9,      // the window the costs were computed for
  kPlanWindowRight = 10,
  kPlanFwdTicket = 11,      // the forward's dynamic acquisition counter (0 between launches)
  kPlanHeaderWords = 16,
};

struct PlanView {
  int* hdr;
  const int* blk_prefix;    // [N+1] cumulative ceil(L/32)
  const int* tile_prefix;   // [N+1] cumulative ceil(L/128)
  const int* item_prefix;   // [N+1] cumulative ceil(L/256)
  const int4* fwd_items;    // [cap] {doc, tile0, ntiles, cost}
  const int4* bwd_items;    // [cap] {doc, ktile, cost, 0}
  const int2* bwd_span;     // [cap] the backward item's document: {first token, length}
  const int2* fwd_span;     // [cap] the forward item's document: {first token, length}
  unsigned long long* sort_keys;  // [pow2(cap)]
};

__host__ __device__ inline int64_t plan_capacity(int64_t T, int N) { return T / kTile + N + 1; }
// ---------------------------------------------------------------- visible keys
// Query i of a document sees key j of the same document (document-local
// positions) iff i - left <= j <= i + right; a negative bound means no limit on
// that side.  Causal calls use right = 0, noncausal calls (-1, -1) (the packed
// noncausal calls of the FLAMIA review, section 8 and its Appendix H); other
// values give sliding windows.
struct Window {
  int left, right;
};
// Key tiles [win_klo, win_khi] seen by some query of query tile t (nt tiles in
// the document): the rows' visible ranges are consecutive, so the union runs
// from the first row's first key to the last row's last key.
__host__ __device__ inline int win_klo(int t, Window w) {
  return w.left < 0 ? 0 : (t * kTile - w.left > 0 ? t * kTile - w.left : 0) / kTile;
}
__host__ __device__ inline int win_khi(int t, int nt, Window w) {
  if (w.right < 0) return nt - 1;
  const int h = (t * kTile + kTile - 1 + w.right) / kTile;
  return h < nt - 1 ? h : nt - 1;
}
// Query tiles [win_tlo, win_thi] holding some query that sees a key of key tile u.
__host__ __device__ inline int win_tlo(int u, Window w) {
  return w.right < 0 ? 0 : (u * kTile - w.right > 0 ? u * kTile - w.right : 0) / kTile;
}
__host__ __device__ inline int win_thi(int u, int nt, Window w) {
  if (w.left < 0) return nt - 1;
  const int h = (u * kTile + kTile - 1 + w.left) / kTile;
  return h < nt - 1 ? h : nt - 1;
}
// True when some (query, key) pair of query tile t x key tile u is hidden by the
// window, or the key tile runs past the document end: the tile needs a mask.
__host__ __device__ inline bool win_masked(int t, int u, int doc_len, Window w) {
  if ((u + 1) * kTile > doc_len) return true;
  if (w.right >= 0 && u * kTile + kTile - 1 > t * kTile + w.right) return true;
  if (w.left >= 0 && u * kTile < t * kTile + kTile - 1 - w.left) return true;
  return false;
}

// fp16 dQ accumulator of the default backward at head_dim 64 (workspace-internal
// layout): one contiguous 8 KB chunk per (document tile, query head, 32-column
// slice of the head dim), tile = tile_prefix[doc] + document-local tile index.  A chunk holds
// the tile's 128 rows of 32 fp16 (64 bytes each) with the 16-byte units of every
// row permuted by the 64-byte TMA/UMMA swizzle, the layout in which the backward
// stages a slice in shared memory and reduces it with one bulk copy.
__host__ __device__ inline size_t dq_chunk_elems(int64_t tile, int h, int slice, int hq, int D) {
  return (((size_t)tile * hq + h) * (size_t)(D / 32) + slice) * (size_t)(kTile * 32);
}
// Byte offset of byte `col_byte` (0..63) of row `r` inside a chunk.
__host__ __device__ inline uint32_t dq_chunk_byte(int r, int col_byte) {
  const uint32_t lin = (uint32_t)r * 64u + (uint32_t)col_byte;
  return lin ^ (((lin >> 7) & 3u) << 4);
}
// At head_dim 128 (default and mixed routes) the backward produces dQ^T, so the
// accumulator is head-dim-major: one contiguous 32 KB chunk per (document tile,
// query head) of [query half hf][head-dim row d][64 queries] fp16, the eight
// 16-byte units of each 128-byte row permuted by XOR with (d mod 8).
__host__ __device__ inline size_t dqt_chunk_elems(int64_t tile, int h, int hq) {
  return ((size_t)tile * hq + h) * (size_t)(kTile * 128);
}
// Byte offset of 16-byte unit `unit` (queries 64 hf + 8 unit .. + 7) of row d.
__host__ __device__ inline uint32_t dqt_chunk_byte(int hf, int d, int unit) {
  return (uint32_t)hf * 16384u + (uint32_t)d * 128u + ((uint32_t)(unit ^ (d & 7)) << 4);
}
__host__ __device__ inline size_t dq_acc_bytes(int64_t T, int N, int hq, int D) {
  return (size_t)plan_capacity(T, N) * hq * D * kTile * 2;
}
__host__ __device__ inline int64_t pow2_ceil(int64_t x) {
  int64_t p = 1;
  while (p < x) p <<= 1;
  return p;
}
__host__ __device__ inline int64_t plan_prefix_words(int N) { return ((int64_t)kPlanHeaderWords + 3 * (N + 1) + 3) & ~3LL; }
__host__ __device__ inline size_t plan_bytes(int64_t T, int N) {
  const int64_t cap = plan_capacity(T, N);
  return (size_t)plan_prefix_words(N) * 4 + (size_t)cap * 48 + (size_t)pow2_ceil(cap) * 8 + 16;
}
__host__ __device__ inline PlanView plan_view(const void* plan, int64_t T, int N) {
  PlanView v;
  int* w = (int*)plan;
  v.hdr = w;
  v.blk_prefix = w + kPlanHeaderWords;
  v.tile_prefix = v.blk_prefix + (N + 1);
  v.item_prefix = v.tile_prefix + (N + 1);
  const int64_t cap = plan_capacity(T, N);
  int4* items = (int4*)(w + plan_prefix_words(N));
  v.fwd_items = items;
  v.bwd_items = items + cap;
  v.bwd_span = (const int2*)(items + 2 * cap);
  v.fwd_span = v.bwd_span + cap;
  v.sort_keys = (unsigned long long*)(v.fwd_span + cap);
  return v;
}

// Document containing prefix-table index `idx`: largest n with prefix[n] <= idx.
__device__ __forceinline__ int upper_doc(const int* prefix, int N, int idx) {
  int lo = 0, hi = N;  // prefix[lo] <= idx < prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= idx) lo = mid; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- dQ boost
// dQ boost of one (document, query head) from its maxima (review section 4, "Forward
// locality and backward locality differ"; reading C-10): c = 2^floor(log2(2^headroom /
// M)), M = 2 max ||dO^_i|| max ||V^_j|| max |K^_jd|; 1 when M is 0 (or not finite).
// With M = m 2^x, m in [0.5, 1) (frexp), the largest e with M 2^e <= 2^headroom is
// headroom - x, plus one when m is exactly 1/2; e is clamped to [-100, 100].
__device__ inline float dq_boost_from_maxima(float max_do, float max_v, float max_k, int headroom) {
  const double M = 2.0 * (double)max_do * (double)max_v * (double)max_k;
  if (!(M > 0.0 && M < 1e300)) return 1.0f;
  int x;
  const double m = frexp(M, &x);
  int e = headroom - x + (m == 0.5 ? 1 : 0);
  e = e < -100 ? -100 : (e > 100 ? 100 : e);
  return __int_as_float((e + 127) << 23);
}

// ---------------------------------------------------------------- exponent rule
// Smallest integer e with amax <= 448 * 2^e, for a finite non-negative fp32
// amax; 0 for amax == 0; clamped to [-127, 127].  Integer arithmetic on the
// fp32 encoding: amax = 1.f * 2^E, and 448 = 1.75 * 2^8, so e = E - 8 + [f > 0.75].
__device__ __forceinline__ int roundup_exp(float amax) {
  uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return 0;
  int E;
  uint32_t frac;
  if ((b >> 23) == 0) {             // fp32 subnormal: b * 2^-149, leading one at bit 23 - lz
    const int lz = __clz(b) - 8;
    frac = (b << lz) & 0x7FFFFFu;
    E = -126 - lz;
  } else {
    E = (int)(b >> 23) - 127;
    frac = b & 0x7FFFFFu;
  }
  int e = E - 8 + (frac > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^e as fp32 for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }
// UE8M0 byte -> 2^(b - 127) as fp32 (b = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// 2^x with the MUFU ex2 instruction (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed fp32 pairs (one f32x2 instruction each): (a.x*b.x + c.x, a.y*b.y + c.y),
// (a.x*b.x, a.y*b.y) and (a.x + b.x, a.y + b.y), round to nearest.  The compiler
// intrinsics let the register allocator keep the pairs in aligned registers.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// Two fp32 -> two E4M3 bytes (round to nearest even, saturating); lo in bits 0-7.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// Record a caller's timing event on `s`.  Inside a stream capture the record is
// captured as an event-record node (cudaEventRecordExternal), so every replay of
// the graph records it again and the events time the graph's launches too.
inline void record_timing_event(void* ev, cudaStream_t s) {
  if (!ev) return;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) == cudaSuccess && st == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

}  // namespace flamia
