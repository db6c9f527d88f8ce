// FLAMIA forward attention with two softmax warpgroups per query tile: the
// kernel of the mixed NVFP4/FP8 route (steps a2-a6 of the hot path).
//
// FLAMIA technical review, Algorithm 1 steps 04-08, with the mixed route of
// section 2 ("The mixed route quantizes Q and K again in E4M3 for the gradient
// products"; Korean review section 3.1: only the score operands Q, K are NVFP4):
//   S   = scale * Q~ K~^T from E2M1 codes with an E4M3 scale per 16 elements
//         (block-scaled NVFP4 MMA; no factoring -- section 3 notes that the
//         per-16 scales vary along the reduction),
//   running row max (exact), p = 2^(x - m), l = sum p (unrounded),
//   off-diagonal key tiles: P^ = E4M3(2^8 p), O += P^ V^ with V's token-block
//         scale per 32 keys (MXF8 block-scaled MMA),
//   the diagonal key tile (reading C-8, section 4 "Folding a local scale into
//         the companion operand"): V per key, P~ = 2^8 p 2^eV(j) quantized E4M3
//         with one round-up exponent per (query row, 32-key group) from its own
//         amax; masked keys are 0, so the tile stays prefix-local,
//   O   = bf16(O / l), LSE = m + ln l.
// The same template without MIXED runs the MXFP8 route (E4M3 scores with the
// row and column factors applied after the MMA).
//
// One CTA per (work item, query head); the item's query tiles run one after
// the other.  Roles (384 threads):
//   warp 0      TMA producer (Q tiles once; K and V per (query tile, key tile)
//               pair through a 3-stage ring; the diagonal pair of the mixed
//               route loads the per-token V copy)
//   warp 1      MMA issuer: S(g) two pairs ahead into a double-buffered S,
//               PV(g) once both warpgroups have written P(g)
//   warp 2      TMEM allocator
//   warps 4-7   softmax warpgroup 0: key columns 0-63 of every tile, O columns [0, D/2)
//   warps 8-11  softmax warpgroup 1: key columns 64-127, O columns [D/2, D)
// Both warpgroups hold the same 128 query rows (thread = row); per pair they
// exchange their partial row maxima through shared memory.
// TMEM columns: S [0,128) and [128,256), O [256, 256 + D), scale words from 384:
// score A (Q, per query tile) [384, 400), score B (K, double-buffered)
// [400, 416), PV A (P, one word per warpgroup) [416, 424), PV B (V) [424, 428).
#include "common.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace flamia {

namespace {

constexpr int kCStages = 3;
constexpr int kCThreads = 384;

struct CoopParams {
  const uint8_t* q_scales;    // UE8M0 per (token, head) (E4M3 route)
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint8_t* q4_scales;   // mixed: E4M3 scale codes [T, hq, D/16]
  const uint8_t* k4_scales;   // mixed: [T, hkv, D/16]
  const uint8_t* vt_scales;   // mixed: UE8M0 per token of the per-token V copy
  const int32_t* cu;
  const int* plan;
  int N, T, hq, hkv;
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
};

template <int D, bool MIXED>
struct CoopSmem {
  static constexpr int kQBytes = MIXED ? kTile * D / 2 : kTile * D;   // score operand tiles
  static constexpr int kVBytes = kTile * D;
  static constexpr int kQ = 0;                                   // [2 query tiles]
  static constexpr int kK = kQ + 2 * kQBytes;                    // [kCStages]
  static constexpr int kV = kK + kCStages * kQBytes;             // [kCStages]
  static constexpr int kP = kV + kCStages * kVBytes;             // P^ codes [query][key]
  static constexpr int kTab = kP + kTile * kTile;                // per key tile: K word, V word
  static constexpr int kMaxTabTiles = 2048;
  static constexpr int kX = kTab + kMaxTabTiles * 8;             // row maxima [2 pairs][2 wg][128], sums [2][128]
  static constexpr int kKF = kX + 6 * 128 * 4;                   // mixed: diagonal per-key (eV, 2^-eV) [128][2]
  static constexpr int kBar = kKF + 128 * 2 * 4;
  static constexpr int kBytes = kBar + 256;
  // at least 116 KB so that one CTA (holding all 512 TMEM columns) fits per SM
  static constexpr int kAlloc = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
};

template <int D, bool MIXED>
__global__ void __launch_bounds__(kCThreads, 1)
    attn_fwd_coop_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_vt,
                         const CoopParams p) {
  static_assert(!MIXED || D == 128, "the mixed route is built for head_dim 128");
  using L = CoopSmem<D, MIXED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                    // [kCStages]
  uint64_t* kv_empty = bars + 1 + kCStages;        // [kCStages]
  uint64_t* s_full = bars + 1 + 2 * kCStages;      // [2]
  uint64_t* sf_ready = s_full + 2;                 // [2]
  uint64_t* p_full = sf_ready + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* o_free = p_full + 2;
  uint64_t* drain = p_full + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_full + 4);
  int* status = const_cast<int*>(p.plan) + kPlanStatus;

  const int item_idx = blockIdx.x / p.hq;
  const int h = blockIdx.x % p.hq;
  // the item, its document span and the item count in one round trip: the grid never
  // exceeds the plan capacity, so the first two reads stay inside the plan also for a
  // CTA without an item
  const PlanView pv = plan_view(p.plan, p.T, p.N);
  const int4 item = pv.fwd_items[item_idx];
  const int2 span = pv.fwd_span[item_idx];
  const int n_items = p.plan[kPlanFwdItems];
  if (item_idx >= n_items) return;
  const int t0 = item.y, ntq = item.z;
  const int doc_start = span.x;
  const int doc_len = span.y;
  const int hk = h / (p.hq / p.hkv);
  const int nkv = ntq > 1 ? t0 + 2 : t0 + 1;              // distinct key tiles of the item
  const int G = (t0 + 1) + (ntq > 1 ? t0 + 2 : 0);        // (query tile, key tile) pairs
  auto pair_of = [&](int g, int& w, int& u) {
    if (g <= t0) { w = 0; u = g; } else { w = 1; u = g - (t0 + 1); }
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kCStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&sf_ready[i], 128);
    }
    mbar_init(p_full, 256);
    mbar_init(pv_done, 1);
    mbar_init(o_free, 256);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // K / V token-block scale bytes of every key tile of the item (one byte per
  // 32-key group, 127 past the document end)
  uint32_t* scale_tab = reinterpret_cast<uint32_t*>(smem + L::kTab);
  const bool tab_ok = nkv <= L::kMaxTabTiles;
  if (tab_ok) {
    uint8_t* tb = reinterpret_cast<uint8_t*>(scale_tab);
    for (int i = threadIdx.x; i < nkv * 4; i += kCThreads) {
      const int uu = i >> 2, gg = i & 3;
      const int kl = uu * kTile + gg * 32;
      const int64_t ktok = (int64_t)doc_start + kl;
      const bool kv = kl < doc_len;
      tb[uu * 8 + gg] = kv ? p.k_scales[ktok * p.hkv + hk] : (uint8_t)127;
      tb[uu * 8 + 4 + gg] = kv ? p.v_scales[ktok * p.hkv + hk] : (uint8_t)127;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  constexpr uint32_t kO = 256, kSFQ = 384, kSFK = 400, kPVA = 416, kPVB = 424;
  constexpr uint32_t kLayoutV = D == 128 ? kSwizzle128B : kSwizzle64B;
  constexpr uint32_t kAtomV = 8 * D;
  // score operand layout: E4M3 rows of D bytes, or E2M1 rows of D/2 = 64 bytes
  constexpr uint32_t kRowS = MIXED ? D / 2 : D;
  constexpr uint32_t kLayoutS = kRowS == 128 ? kSwizzle128B : kSwizzle64B;
  constexpr uint32_t kAtomS = 8 * kRowS;

  auto tile_scales = [&](int uu, uint32_t& kw, uint32_t& vw) {
    if (tab_ok) {
      const uint2 kv2 = *reinterpret_cast<const uint2*>(scale_tab + 2 * uu);
      kw = kv2.x;
      vw = kv2.y;
      return;
    }
    kw = 0x7F7F7F7Fu;
    vw = 0x7F7F7F7Fu;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int kl = uu * kTile + g * 32;
      if (kl < doc_len) {
        const int64_t ktok = (int64_t)doc_start + kl;
        kw = (kw & ~(0xFFu << (8 * g))) | ((uint32_t)p.k_scales[ktok * p.hkv + hk] << (8 * g));
        vw = (vw & ~(0xFFu << (8 * g))) | ((uint32_t)p.v_scales[ktok * p.hkv + hk] << (8 * g));
      }
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      if (MIXED) tma_prefetch_desc(&tm_vt);
      mbar_arrive_expect_tx(q_full, ntq * L::kQBytes);
      for (int w = 0; w < ntq; ++w)
        tma_load_3d(smem + L::kQ + w * L::kQBytes, &tm_q, q_full, 0, h, doc_start + (t0 + w) * kTile);
      for (int g = 0; g < G; ++g) {
        int w, u;
        pair_of(g, w, u);
        const int st = g % kCStages;
        if (g >= kCStages && !mbar_wait(&kv_empty[st], ((g / kCStages) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&kv_full[st], L::kQBytes + L::kVBytes);
        tma_load_3d(smem + L::kK + st * L::kQBytes, &tm_k, &kv_full[st], 0, hk, doc_start + u * kTile);
        const CUtensorMap* vmap = (MIXED && u == t0 + w) ? &tm_vt : &tm_v;
        tma_load_3d(smem + L::kV + st * L::kVBytes, vmap, &kv_full[st], 0, hk, doc_start + u * kTile);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sq = smem_u32(smem + L::kQ), sk = smem_u32(smem + L::kK), sv = smem_u32(smem + L::kV),
                     sp = smem_u32(smem + L::kP);
      auto issue_s = [&](int g) {
        int w, u;
        pair_of(g, w, u);
        const uint32_t qa = sq + w * L::kQBytes, ka = sk + (g % kCStages) * L::kQBytes;
        const uint32_t dst = tbase + 128 * (g & 1);
        if constexpr (MIXED) {
#pragma unroll
          for (int s = 0; s < 2; ++s)      // K = 64 E2M1 elements (32 bytes) per instruction
            mma_nvf4(dst, smem_desc(qa + 32 * s, 16, kAtomS, kLayoutS), smem_desc(ka + 32 * s, 16, kAtomS, kLayoutS),
                     idesc_nvf4(128, 128), tbase + kSFQ + 8 * w + 4 * s, tbase + kSFK + 8 * (g & 1) + 4 * s, s > 0);
        } else {
#pragma unroll
          for (int s = 0; s < D / 32; ++s)
            mma_f8(dst, smem_desc(qa + 32 * s, 16, kAtomS, kLayoutS), smem_desc(ka + 32 * s, 16, kAtomS, kLayoutS),
                   idesc_f8(128, 128, 0, 0), s > 0);
        }
      };
      bool ok = mbar_wait(q_full, 0, status);
      for (int g = 0; g < 2 && g < G && ok; ++g) {
        ok = mbar_wait(&kv_full[g % kCStages], (g / kCStages) & 1, status);
        if (ok && MIXED) ok = mbar_wait(&sf_ready[g & 1], (g >> 1) & 1, status);
        if (!ok) break;
        tc_fence_after();
        issue_s(g);
        mma_commit(&s_full[g & 1]);
      }
      for (int g = 0; g < G && ok; ++g) {
        int w, u;
        pair_of(g, w, u);
        ok = mbar_wait(p_full, g & 1, status);
        if (ok && u == 0 && w > 0) ok = mbar_wait(o_free, 0, status);   // epilogue of query tile 0 has read O
        if (!ok) break;
        tc_fence_after();
        const uint32_t va = sv + (g % kCStages) * L::kVBytes;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          // O += P^ V: A = P^ [query][key] K-major; B = V [key][d] MN-major; 32 keys per instruction
          mma_mxf8(tbase + kO, smem_desc(sp + 32 * s, 16, 1024, kSwizzle128B),
                   smem_desc(va + s * 32 * D, kAtomV, kAtomV, kLayoutV), idesc_mxf8(128, D, 0, 1, s, s),
                   tbase + kPVA + 4 * (s >> 1), tbase + kPVB, (u > 0 || s > 0));
        }
        mma_commit(pv_done);
        mma_commit(&kv_empty[g % kCStages]);
        if (g + 2 < G) {
          const int g2 = g + 2;
          ok = mbar_wait(&kv_full[g2 % kCStages], (g2 / kCStages) & 1, status);
          if (ok && MIXED) ok = mbar_wait(&sf_ready[g2 & 1], (g2 >> 1) & 1, status);
          if (!ok) break;
          tc_fence_after();
          issue_s(g2);
          mma_commit(&s_full[g2 & 1]);
        }
      }
      if (!ok) {
        // timed out: make sure nothing issued is still running before TMEM is freed
        mma_commit(drain);
        mbar_wait(drain, 0, status);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax (two warpgroups)
    const int wg = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // query row within the tile (TMEM lane)
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const int kc0 = 64 * wg;                           // first key column of this warpgroup
    constexpr int kOCols = D / 2;                      // O columns per warpgroup
    const int oc0 = kOCols * wg;
    float* xmax = reinterpret_cast<float*>(smem + L::kX);         // [2][2][128]
    float* xsum = xmax + 4 * 128;                                  // [2][128]
    float* kf = reinterpret_cast<float*>(smem + L::kKF);           // [128][2]
    uint8_t* sP = smem + L::kP;

    // score-operand scale words (mixed; warpgroup 0 writes them, replicated over
    // the four lane quarters: lane 32q + l, column c holds row 32c + l)
    auto load_rows4 = [&](const uint8_t* base, int64_t tok0, int H, int hh, uint2 (&w4)[4]) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t tok = tok0 + 32 * c + lane;
        w4[c] = tok < p.T ? *reinterpret_cast<const uint2*>(base + (tok * H + hh) * (D / 16)) : make_uint2(0u, 0u);
      }
    };
    auto store_sf = [&](uint32_t col, const uint2 (&w4)[4]) {
      tmem_st4(lane_base + col, w4[0].x, w4[1].x, w4[2].x, w4[3].x);        // instruction 0: groups 0-3
      tmem_st4(lane_base + col + 4, w4[0].y, w4[1].y, w4[2].y, w4[3].y);    // instruction 1: groups 4-7
    };
    uint2 kpre[4];
    if (MIXED && wg == 0) {
      for (int w = 0; w < ntq; ++w) {
        uint2 q4[4];
        load_rows4(p.q4_scales, (int64_t)doc_start + (t0 + w) * kTile, p.hq, h, q4);
        store_sf(kSFQ + 8 * w, q4);
      }
      for (int g = 0; g < 2 && g < G; ++g) {
        int w, u;
        pair_of(g, w, u);
        load_rows4(p.k4_scales, (int64_t)doc_start + u * kTile, p.hkv, hk, kpre);
        store_sf(kSFK + 8 * g, kpre);
      }
      tmem_st_wait();
      tc_fence_before();
      for (int g = 0; g < 2 && g < G; ++g) mbar_arrive(&sf_ready[g]);
      if (G > 2) {
        int w, u;
        pair_of(2, w, u);
        load_rows4(p.k4_scales, (int64_t)doc_start + u * kTile, p.hkv, hk, kpre);
      }
    }

    float m = -INFINITY, lsum = 0.f, fq = 0.f;
    bool row_valid = false;
    int64_t tok = 0;
    bool ok = true;
    for (int g = 0; g < G; ++g) {
      int w, u;
      pair_of(g, w, u);
      const int t = t0 + w;
      const bool diag = (u == t);
      const int buf = g & 1;
      if (u == 0) {
        const int ql = t * kTile + r;
        row_valid = ql < doc_len;
        tok = (int64_t)doc_start + ql;
        fq = MIXED ? p.scale_log2 : p.scale_log2 * (row_valid ? ue8m0_to_f32(p.q_scales[tok * p.hq + h]) : 1.0f);
        m = -INFINITY;
        lsum = 0.f;
        if (MIXED && r < 64) {
          // per-key V exponents of this query tile's diagonal key tile (this warpgroup's keys)
          const int j = kc0 + r;
          const int kl = t * kTile + j;
          const int vb = kl < doc_len ? p.vt_scales[((int64_t)doc_start + kl) * p.hkv + hk] : 127;
          kf[2 * j] = (float)(vb - 127);
          kf[2 * j + 1] = ue8m0_to_f32((uint32_t)(254 - vb));
        }
      }
      bool okl = mbar_wait(&s_full[buf], (g >> 1) & 1, status);
      float mx = -INFINITY;
      uint32_t kw = 0x7F7F7F7Fu, vw = 0x7F7F7F7Fu;
      if (okl) {
        tc_fence_after();
        if (MIXED && wg == 0 && g + 2 < G) {
          // score B words of pair g + 2 into the buffer S(g) has finished with
          store_sf(kSFK + 8 * buf, kpre);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&sf_ready[buf]);
          if (g + 3 < G) {
            int w3, u3;
            pair_of(g + 3, w3, u3);
            load_rows4(p.k4_scales, (int64_t)doc_start + u3 * kTile, p.hkv, hk, kpre);
          }
        }
        tile_scales(u, kw, vw);
        // pass 1: partial row max of x = S * factor over this warpgroup's 64 keys
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float f = MIXED ? fq : fq * ue8m0_to_f32((kw >> (8 * (2 * wg + c))) & 0xFFu);
          const uint32_t col = 128 * buf + kc0 + 32 * c;
          uint32_t v[32];
          if (!diag) {
            float cm;
            tmem_ld32_max(lane_base + col, v, cm);
            tmem_ld_wait();
            mx = fmaxf(mx, cm * f);
          } else {
            tmem_ld32(lane_base + col, v);
            tmem_ld_wait();
            float b = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) b = (kc0 + 32 * c + j) <= r ? fmaxf(b, __uint_as_float(v[j])) : b;
            mx = fmaxf(mx, b * f);
          }
        }
        xmax[(buf * 2 + wg) * 128 + r] = mx;
        if (g > 0) okl = mbar_wait(pv_done, (g - 1) & 1, status);   // PV(g-1) done: O, P^ and PV words free
      }
      ok = named_bar_and(1, 256, okl);
      if (!ok) break;
      tc_fence_after();
      mx = fmaxf(xmax[(buf * 2) * 128 + r], xmax[(buf * 2 + 1) * 128 + r]);
      const float m_new = fmaxf(m, mx);
      const float alpha = fast_exp2(m - m_new);   // 0 on the first key tile
      if (u > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + kO + oc0 + 32 * c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(lane_base + kO + oc0 + 32 * c, v);
        }
        tmem_st_wait();
      }
      lsum *= alpha;
      const float neg = 8.0f - m_new;
      const bool fold = MIXED && diag;
      uint32_t sfa = 0x7F7F7F7Fu;
      // pass 2: boosted weights 2^(x - m + 8), their E4M3 codes into this warpgroup's half of P^
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int gidx = 2 * wg + c;                 // 32-key group within the tile
        const float f = MIXED ? fq : fq * ue8m0_to_f32((kw >> (8 * gidx)) & 0xFFu);
        uint32_t v[32];
        tmem_ld32(lane_base + 128 * buf + kc0 + 32 * c, v);
        tmem_ld_wait();
        uint32_t packed[8];
        if (!fold) {
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float e0 = fast_exp2(fmaf(__uint_as_float(v[j]), f, neg));
            float e1 = fast_exp2(fmaf(__uint_as_float(v[j + 1]), f, neg));
            if (diag) {
              e0 = (kc0 + 32 * c + j) <= r ? e0 : 0.f;
              e1 = (kc0 + 32 * c + j + 1) <= r ? e1 : 0.f;
            }
            acc += e0 + e1;
            const uint32_t c2 = e4m3x2(e0, e1);
            if (j & 2) packed[j >> 2] |= c2 << 16; else packed[j >> 2] = c2;
          }
          lsum += acc;
        } else {
          // V's per-key exponent folded into the weight; one round-up exponent per 32-key group
          float pf[32];
          float gmax = 0.f, acc = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int kc = kc0 + 32 * c + j;
            float e = fast_exp2(fmaf(__uint_as_float(v[j]), f, neg) + kf[2 * kc]);
            e = kc <= r ? e : 0.f;
            pf[j] = e;
            acc = fmaf(e, kf[2 * kc + 1], acc);
            gmax = fmaxf(gmax, e);
          }
          lsum += acc;
          const int eg = roundup_exp(gmax);
          const float sc = exp2i(-eg);
          sfa = (sfa & ~(0xFFu << (8 * gidx))) | ((uint32_t)(eg + 127) << (8 * gidx));
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            packed[j >> 2] = (uint32_t)e4m3x2(pf[j] * sc, pf[j + 1] * sc) |
                             ((uint32_t)e4m3x2(pf[j + 2] * sc, pf[j + 3] * sc) << 16);
        }
        *reinterpret_cast<uint4*>(sP + swz_offset(r, kc0 + 32 * c, 128)) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        *reinterpret_cast<uint4*>(sP + swz_offset(r, kc0 + 32 * c + 16, 128)) =
            make_uint4(packed[4], packed[5], packed[6], packed[7]);
      }
      m = m_new;
      // PV block-scale words: A = this warpgroup's per-row word (row r at lane r,
      // column base + r / 32); B = V's scale per 32-key group, replicated
      tmem_st1(lane_base + kPVA + 4 * wg + quarter, sfa);
      if (wg == 0) {
        const uint32_t vsf = fold ? 0x7F7F7F7Fu : vw;
        tmem_st4(lane_base + kPVB, vsf, vsf, vsf, vsf);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
      if (diag) {
        // epilogue of query tile t: O / l, LSE
        okl = mbar_wait(pv_done, g & 1, status);
        xsum[wg * 128 + r] = lsum;
        ok = named_bar_and(1, 256, okl);
        if (!ok) break;
        tc_fence_after();
        const float l = xsum[r] + xsum[128 + r];
        const float inv = 1.0f / l;
        __nv_bfloat16* orow = p.out + (tok * p.hq + h) * D + oc0;
        const bool al32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
#pragma unroll 1
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + kO + oc0 + 32 * c, v);
          tmem_ld_wait();
          if (row_valid) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * j]) * inv,
                                                        __uint_as_float(v[2 * j + 1]) * inv);
              pk[j] = *reinterpret_cast<uint32_t*>(&b2);
            }
            __nv_bfloat16* dst = orow + 32 * c;
            if (al32) {                  // two 32-byte stores; 16-byte ones if O is only 16-byte aligned
              st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
              st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            }
          }
        }
        if (wg == 0 && row_valid) p.lse[(int64_t)h * p.T + tok] = (m + __log2f(l) - 8.0f) * 0.69314718055994531f;
        tc_fence_before();
        mbar_arrive(o_free);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool MIXED>
cudaError_t launch_coop_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tvt, const CoopParams& p, int T, int N, cudaStream_t stream) {
  const int64_t max_items = (int64_t)T / (kTile * kItemTiles) + N + 1;
  const int64_t grid = max_items * p.hq;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  constexpr int smem = CoopSmem<D, MIXED>::kAlloc;
  cudaError_t e = prepare_kernel<attn_fwd_coop_kernel<D, MIXED>>(smem);
  if (e != cudaSuccess) return e;
  attn_fwd_coop_kernel<D, MIXED><<<(unsigned)grid, kCThreads, smem, stream>>>(tq, tk, tv, tvt, p);
  return cudaGetLastError();
}

}  // namespace

// Forward of the mixed route (mixed != 0: q4/k4 are the packed E2M1 score
// operands with their E4M3 group scales, vt the per-token V copy) or, with
// mixed == 0, the MXFP8 route on this kernel.  The launch of the rows outside
// every document (O = 0, LSE = +inf) stays with the caller.
cudaError_t launch_fwd_coop(int D, int mixed, const void* qc, const void* qs, const void* kc, const void* ks,
                            const void* vc, const void* vs, const void* q4c, const void* q4s, const void* k4c,
                            const void* k4s, const void* vtc, const void* vts, const int32_t* cu, int N, int T, int hq,
                            int hkv, float scale, const void* plan, void* out, float* lse, cudaStream_t stream) {
  CoopParams p;
  p.q_scales = static_cast<const uint8_t*>(qs);
  p.k_scales = static_cast<const uint8_t*>(ks);
  p.v_scales = static_cast<const uint8_t*>(vs);
  p.q4_scales = static_cast<const uint8_t*>(q4s);
  p.k4_scales = static_cast<const uint8_t*>(k4s);
  p.vt_scales = static_cast<const uint8_t*>(vts);
  p.cu = cu;
  p.plan = static_cast<const int*>(plan);
  p.N = N;
  p.T = T;
  p.hq = hq;
  p.hkv = hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  CUtensorMap tq, tk, tv, tvt;
  if (mixed) {
    if (D != 128) return cudaErrorInvalidValue;
    if (!make_tmap_u8_3d(&tq, q4c, D / 2, hq, T, D / 2, (uint64_t)hq * D / 2, D / 2, kTile) ||
        !make_tmap_u8_3d(&tk, k4c, D / 2, hkv, T, D / 2, (uint64_t)hkv * D / 2, D / 2, kTile) ||
        !make_tmap_u8_3d(&tv, vc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile) ||
        !make_tmap_u8_3d(&tvt, vtc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile))
      return cudaErrorInvalidValue;
    return launch_coop_d<128, true>(tq, tk, tv, tvt, p, T, N, stream);
  }
  if (!make_tmap_u8_3d(&tq, qc, D, hq, T, D, (uint64_t)hq * D, D, kTile) ||
      !make_tmap_u8_3d(&tk, kc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile) ||
      !make_tmap_u8_3d(&tv, vc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile))
    return cudaErrorInvalidValue;
  tvt = tv;
  if (D == 128) return launch_coop_d<128, false>(tq, tk, tv, tvt, p, T, N, stream);
  if (D == 64) return launch_coop_d<64, false>(tq, tk, tv, tvt, p, T, N, stream);
  return cudaErrorInvalidValue;
}

}  // namespace flamia
