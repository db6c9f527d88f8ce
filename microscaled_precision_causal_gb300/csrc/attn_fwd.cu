// FLAMIA forward attention (steps a4-a6 of the hot path): causal, packed
// documents, MXFP8 token-block operands, tcgen05 MMAs with TMEM accumulators.
//
// FLAMIA technical review, Algorithm 1 steps 04-08:
//   S   = (scale * s_Q(i) * s_K(j)) * sum_d c_Q[i,d] c_K[j,d]
//         (section 3, "Factoring the scales out of the score MMA": an E4M3 MMA
//         without block scales, the row/column factors applied afterwards),
//   running row max (exact), p = 2^(x - m), l = sum p (unrounded),
//   P^  = E4M3(2^8 p) (section 5, "A range budget for probability quantization"),
//   O  += P^ V^ with V's token-block scale per 32 keys (MXF8 block-scaled MMA),
//   O   = bf16(O / l), LSE = m + ln l.
//
// The MXFP8 route runs attn_fwd_persist_kernel below: one CTA per SM walks the
// (work item, query head) units in boustrophedon order (Algorithm 2 step 05).  The
// strict options run attn_fwd_kernel: one CTA per unit.  A work item is up to two
// document-local 128-query tiles (Algorithm 2 step 03).  Roles (384 threads):
//   warp 0      TMA producer: both Q tiles once, then K/V tiles through a ring
//   warp 1      MMA issuer (converged warp, one elected lane issues): S_w = Q_w K^T
//               and O_w += P^_w V
//   warp 2      TMEM allocator
//   warps 4-7   softmax warpgroup 0 (query tile t0), thread = query row
//   warps 8-11  softmax warpgroup 1 (query tile t0 + 1)
// The two softmax warpgroups ping-pong: while one converts its score tile the
// tensor core runs the other's PV and next QK^T.
// TMEM columns: S_0 [0,128), O_0 [128,128+D), S_1 [256,384), O_1 [384,384+D).
// The block-scale words of the PV MMA live in the last 8 columns of the
// warpgroup's S region (written after S was read; the next S MMA is issued
// after the PV MMA by the same thread, and tcgen05 MMAs run in issue order).
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace flamia {

namespace {

constexpr int kStages = 3;
constexpr int kThreads = 384;

struct FwdParams {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const int32_t* cu;
  const int* plan;
  int N, T, hq, hkv;
  float scale_log2;          // softmax scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  Window win;                // visible keys (causal: right = 0); the strict kernel is causal only
};

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = kTile * D;          // one Q / K / V code tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;
  static constexpr int kScaleTab = kP + 2 * kTile * kTile;      // per key tile: K word, V word
  static constexpr int kMaxTabTiles = 4096;                      // (strict: 256 bytes per tile, 128 tiles)
  static constexpr int kKeyF = kScaleTab + kMaxTabTiles * 8;     // strict: [wg][2 buffers][3][128] floats
  static constexpr int kBar = kKeyF + 2 * 2 * 3 * 128 * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;           // slack for 1024-byte alignment
};

__device__ __forceinline__ float scale_of(const uint8_t* s, int64_t tok, int H, int h, bool valid) {
  return valid ? ue8m0_to_f32(s[tok * H + h]) : 1.0f;
}

template <int D, bool STRICT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;                 // [kStages]
  uint64_t* kv_empty = bars + 1 + kStages;      // [kStages]
  uint64_t* s_full = bars + 1 + 2 * kStages;    // [2]
  uint64_t* p_full = s_full + 2;                // [2]
  uint64_t* o_full = p_full + 2;                // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_full + 2);
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
  const int nk_w[2] = {t0 + 1, ntq > 1 ? t0 + 2 : 0};
  const int nkv = ntq > 1 ? t0 + 2 : t0 + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // per-key scale bytes (strict) or per-tile scale words of the item's key tiles staged in
  // shared memory: the strict table holds the first kStrictTabTiles tiles and the softmax
  // reads later tiles' bytes from global memory
  constexpr int kStrictTabTiles = L::kMaxTabTiles / 32;
  const bool tab_ok = STRICT ? true : nkv <= L::kMaxTabTiles;
  constexpr int kEarly = kStages;                 // K/V tiles whose loads start in the prologue
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&s_full[w], 1);
      mbar_init(&p_full[w], 128);
      mbar_init(&o_full[w], 1);
    }
    fence_mbar_init();
    {
      // the producer's first loads start before the scale table and the CTA barrier
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(q_full, ntq * L::kTileBytes);
      for (int w = 0; w < ntq; ++w)
        tma_load_3d(smem + L::kQ + w * L::kTileBytes, &tm_q, q_full, 0, h, doc_start + (t0 + w) * kTile);
      for (int u = 0; u < nkv && u < kEarly; ++u) {
        mbar_arrive_expect_tx(&kv_full[u], 2 * L::kTileBytes);
        tma_load_3d(smem + L::kK + u * L::kTileBytes, &tm_k, &kv_full[u], 0, hk, doc_start + u * kTile);
        tma_load_3d(smem + L::kV + u * L::kTileBytes, &tm_v, &kv_full[u], 0, hk, doc_start + u * kTile);
      }
    }
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // K / V block-scale bytes of every key tile of the item (one byte per 32-key
  // group, 127 past the document end), staged once by the two softmax warpgroups
  // after the CTA barrier (while the first tiles load) so the softmax loop reads
  // them from shared memory
  // (each thread's global loads are issued before its shared-memory stores)
  uint32_t* scale_tab = reinterpret_cast<uint32_t*>(smem + L::kScaleTab);
  auto stage_scale_table = [&](int first, int stride) {
    if (STRICT && tab_ok) {
      // strict: per-token scale bytes of every key of the item, 128 K then 128 V per tile
      uint8_t* tb = reinterpret_cast<uint8_t*>(scale_tab);
      for (int i = first; i < min(nkv, kStrictTabTiles) * kTile; i += stride) {
        const int uu = i >> 7, j = i & 127;
        const int kl = uu * kTile + j;
        const int64_t ktok = (int64_t)doc_start + kl;
        const bool kv = kl < doc_len;
        const uint8_t kb = kv ? __ldg(p.k_scales + ktok * p.hkv + hk) : (uint8_t)127;
        const uint8_t vb = kv ? __ldg(p.v_scales + ktok * p.hkv + hk) : (uint8_t)127;
        tb[uu * 256 + j] = kb;
        tb[uu * 256 + 128 + j] = vb;
      }
    }
    if (!STRICT && tab_ok) {
      uint8_t* tb = reinterpret_cast<uint8_t*>(scale_tab);
      for (int i = first; i < nkv * 4; i += stride) {
        const int uu = i >> 2, gg = i & 3;
        const int kl = uu * kTile + gg * 32;
        const int64_t ktok = (int64_t)doc_start + kl;
        const bool kv = kl < doc_len;
        const uint8_t kb = kv ? __ldg(p.k_scales + ktok * p.hkv + hk) : (uint8_t)127;
        const uint8_t vb = kv ? __ldg(p.v_scales + ktok * p.hkv + hk) : (uint8_t)127;
        tb[uu * 8 + gg] = kb;
        tb[uu * 8 + 4 + gg] = vb;
      }
    }
  };
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  constexpr uint32_t kSCol[2] = {0, 256};
  constexpr uint32_t kOCol[2] = {128, 384};
  constexpr uint32_t kRowBytes = D;                 // K-major row of a Q/K/V tile
  constexpr uint32_t kLayout = D == 128 ? kSwizzle128B : kSwizzle64B;
  constexpr uint32_t kAtom = 8 * D;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int u = kEarly; u < nkv; ++u) {      // Q and the first kEarly K/V tiles: prologue
        const int st = u % kStages;
        if (u >= kStages && !mbar_wait(&kv_empty[st], ((u / kStages) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * L::kTileBytes);
        tma_load_3d(smem + L::kK + st * L::kTileBytes, &tm_k, &kv_full[st], 0, hk, doc_start + u * kTile);
        tma_load_3d(smem + L::kV + st * L::kTileBytes, &tm_v, &kv_full[st], 0, hk, doc_start + u * kTile);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The warp runs the loop converged (every lane waits); the elected lane issues
    // the MMAs and the commits.  Every tile sits at a compile-time offset from the
    // aligned SMEM base, so each descriptor is one add on base16 (re-read at every
    // use so that the compiler does not hoist the descriptor words into registers).
    const bool leader = elect_one();
    {
      const uint32_t base16 = (smem_u32(smem) & 0x3FFFFu) >> 4;
      auto b16 = [&]() {
        uint32_t x;
        asm volatile("mov.b32 %0, %1;" : "=r"(x) : "r"(base16));
        return x;
      };
      bool ok = warp_wait(q_full, 0, status);
      auto issue_s = [&](int w, int u) {
        const int st = u % kStages;
#pragma unroll
        for (int s = 0; s < D / 32; ++s)
          if (leader)
            mma_f8(tbase + kSCol[w], sdesc_at(b16(), L::kQ + w * L::kTileBytes + 32 * s, 16, kAtom, kLayout),
                   sdesc_at(b16(), L::kK + st * L::kTileBytes + 32 * s, 16, kAtom, kLayout), idesc_f8(128, 128, 0, 0),
                   s > 0);
      };
      auto issue_pv = [&](int w, int u) {
        const int st = u % kStages;
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (leader)
            mma_mxf8(tbase + kOCol[w], sdesc_at(b16(), L::kP + w * kTile * kTile + 32 * s, 16, 1024, kSwizzle128B),
                     sdesc_at(b16(), L::kV + st * L::kTileBytes + s * 32 * kRowBytes, kAtom, kAtom, kLayout),
                     idesc_mxf8(128, D, 0, 1, s, s), tbase + kSCol[w] + 120, tbase + kSCol[w] + 124, (u > 0 || s > 0));
      };
      if (ok) ok = warp_wait(&kv_full[0], 0, status);
      if (ok) {
        tc_fence_after();
        for (int w = 0; w < ntq; ++w) {
          issue_s(w, 0);
          if (leader) mma_commit(&s_full[w]);
        }
        for (int u = 0; u < nkv && ok; ++u) {
          bool next_loaded = false;
          for (int w = 0; w < ntq && ok; ++w) {
            if (u >= nk_w[w]) continue;
            ok = warp_wait(&p_full[w], u & 1, status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(w, u);
            if (u + 1 < nk_w[w]) {
              if (!next_loaded) {
                const int st = (u + 1) % kStages;
                ok = warp_wait(&kv_full[st], ((u + 1) / kStages) & 1, status);
                if (!ok) break;
                tc_fence_after();
                next_loaded = true;
              }
              issue_s(w, u + 1);
              if (leader) mma_commit(&s_full[w]);
            } else {
              if (leader) mma_commit(&o_full[w]);
            }
          }
          if (leader) mma_commit(&kv_empty[u % kStages]);
        }
      }
      if (!ok && leader) {
        // timed out: make sure nothing we issued is still running before TMEM is freed
        mma_commit(&o_full[0]);
        mbar_wait(&o_full[0], 0, status);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    stage_scale_table(threadIdx.x - 128, 256);
    named_bar_sync(1, 256);
    const int w = (warp - 4) >> 2;        // warpgroup = query tile t0 + w
    if (w < ntq) {
      const int quarter = warp & 3;
      const int r = quarter * 32 + lane;  // row within the tile (= TMEM lane)
      const int t = t0 + w;
      const int qrow_local = t * kTile + r;
      const bool row_valid = qrow_local < doc_len;
      const int64_t tok = (int64_t)doc_start + qrow_local;
      const float fq = p.scale_log2 * scale_of(p.q_scales, tok, p.hq, h, row_valid);
      const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
      const uint32_t s_addr = lane_base + kSCol[w], o_addr = lane_base + kOCol[w];
      uint8_t* sP = smem + L::kP + w * kTile * kTile;
      float m = -INFINITY, lsum = 0.f;
      bool ok = true;
      const int nk = nk_w[w];
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
      float* keyf = reinterpret_cast<float*>(smem + L::kKeyF) + w * (2 * 3 * 128);   // strict only
      for (int u = 0; u < nk; ++u) {
        uint32_t kw = 0, vsf = 0x7F7F7F7Fu;
        float fk[4];
        const float* kf = nullptr;     // strict: per-key s_K, V exponent, 2^-eV of this tile
        if constexpr (STRICT) {
          float* buf = keyf + (u & 1) * (3 * 128);
          int kb = 127, vb = 127;
          if (u < kStrictTabTiles) {
            const uint8_t* tb = reinterpret_cast<const uint8_t*>(scale_tab) + u * 256;
            kb = tb[r];
            vb = tb[128 + r];
          } else if (u * kTile + r < doc_len) {      // past the table: this key's bytes from global memory
            const int64_t ktok = (int64_t)doc_start + u * kTile + r;
            kb = __ldg(p.k_scales + ktok * p.hkv + hk);
            vb = __ldg(p.v_scales + ktok * p.hkv + hk);
          }
          buf[r] = ue8m0_to_f32((uint32_t)kb);
          buf[128 + r] = (float)(vb - 127);
          buf[256 + r] = ue8m0_to_f32((uint32_t)(254 - vb));
          kf = buf;                      // published by the warpgroup barrier below
#pragma unroll
          for (int g = 0; g < 4; ++g) fk[g] = fq;
        } else {
          tile_scales(u, kw, vsf);
#pragma unroll
          for (int g = 0; g < 4; ++g) fk[g] = fq * ue8m0_to_f32((kw >> (8 * g)) & 0xFFu);
        }
        const bool diag = (u == t);
        if constexpr (STRICT) {
          // warpgroup-wide: publishes the per-key factors and leaves together on a timeout
          ok = named_bar_and(2 + w, 128, mbar_wait(&s_full[w], u & 1, status));
        } else {
          ok = __all_sync(0xffffffffu, mbar_wait(&s_full[w], u & 1, status));
        }
        if (!ok) break;
        tc_fence_after();
        // pass 1: row max of x = S * log2(e) over visible keys.  The column factor
        // is a positive power of two times a constant, so max(v * f) = f * max(v).
        float mx = -INFINITY;
        if (STRICT) {
          // per-key column factors: x_j = dot_j * s_K(j) * fq
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];
            tmem_ld32(s_addr + 32 * g, v);
            tmem_ld_wait();
            float b = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float x = __uint_as_float(v[j]) * kf[32 * g + j];
              b = (!diag || (g * 32 + j) <= r) ? fmaxf(b, x) : b;
            }
            mx = fmaxf(mx, b * fq);
          }
        } else if (!diag) {
          // fused TMEM load + row max (all keys visible)
          float cm[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];               // the values are not needed here, only their max
            tmem_ld32_max(s_addr + 32 * g, v, cm[g]);
            tmem_ld_wait();               // before the registers can be reused
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) mx = fmaxf(mx, cm[g] * fk[g]);
        } else {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];
            tmem_ld32(s_addr + 32 * g, v);
            tmem_ld_wait();
            float b = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) b = (g * 32 + j) <= r ? fmaxf(b, __uint_as_float(v[j])) : b;
            mx = fmaxf(mx, b * fk[g]);
          }
        }
        const float m_new = fmaxf(m, mx);
        const float alpha = fast_exp2(m - m_new);   // 0 on the first tile
        // rescale the running O row when the max moved (warp-uniform decision)
        if (u > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(o_addr + 32 * c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st32(o_addr + 32 * c, v);
          }
          tmem_st_wait();
        }
        lsum *= alpha;
        const float neg = 8.0f - m_new;
        if constexpr (STRICT) {
          // pass 2 (strict): V's per-key scale folded into the boosted weight,
          // pf_j = 2^(x_j - m + 8 + eV_j); one round-up exponent per 32-key group;
          // the normaliser accumulates pf_j * 2^-eV_j (= the unfolded boosted weight)
          uint32_t sfa = 0;
          float lacc = 0.f;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];
            tmem_ld32(s_addr + 32 * g, v);
            tmem_ld_wait();
            float pf[32];
            float gmax = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int kc = g * 32 + j;
              const float x = __uint_as_float(v[j]) * kf[kc] * fq;
              float e = fast_exp2(x + neg + kf[128 + kc]);
              e = (!diag || kc <= r) ? e : 0.f;
              pf[j] = e;
              lacc = fmaf(e, kf[256 + kc], lacc);
              gmax = fmaxf(gmax, e);
            }
            const int eg = roundup_exp(gmax);
            const float sc = exp2i(-eg);
            sfa |= (uint32_t)(eg + 127) << (8 * g);
            uint32_t packed[8];
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              packed[j >> 2] = (uint32_t)e4m3x2(pf[j] * sc, pf[j + 1] * sc) |
                               ((uint32_t)e4m3x2(pf[j + 2] * sc, pf[j + 3] * sc) << 16);
            *reinterpret_cast<uint4*>(sP + swz_offset(r, 32 * g, 128)) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4*>(sP + swz_offset(r, 32 * g + 16, 128)) =
                make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
          lsum += lacc;
          // A scale of row r is read from lane r, column (base + r / 32): this warp's quarter
          tmem_st1(s_addr + 120 + quarter, sfa);
        } else {
        // pass 2: boosted weights 2^(x - m + 8), their E4M3 codes into the P tile (the
        // loop is built twice: the causal mask only on the diagonal tile)
        float2 acc2 = make_float2(0.f, 0.f);
        auto pass2 = [&](auto diag_tile) {
          constexpr bool kDiag = decltype(diag_tile)::value;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t v[32];
          tmem_ld32(s_addr + 32 * g, v);
          tmem_ld_wait();
          uint32_t packed[8];
          const float2 f2 = make_float2(fk[g], fk[g]), n2 = make_float2(neg, neg);
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            float2 x0 = ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), f2, n2);
            float2 x1 = ffma2(make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])), f2, n2);
            float2 p0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
            float2 p1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
            if (kDiag) {
              const int kc = g * 32 + j;
              p0.x = kc <= r ? p0.x : 0.f;
              p0.y = kc + 1 <= r ? p0.y : 0.f;
              p1.x = kc + 2 <= r ? p1.x : 0.f;
              p1.y = kc + 3 <= r ? p1.y : 0.f;
            }
            acc2 = fadd2(acc2, fadd2(p0, p1));
            packed[j >> 2] = (uint32_t)e4m3x2(p0.x, p0.y) | ((uint32_t)e4m3x2(p1.x, p1.y) << 16);
          }
          *reinterpret_cast<uint4*>(sP + swz_offset(r, 32 * g, 128)) =
              make_uint4(packed[0], packed[1], packed[2], packed[3]);
          *reinterpret_cast<uint4*>(sP + swz_offset(r, 32 * g + 16, 128)) =
              make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
        };
        if (diag) pass2(std::true_type{});
        else pass2(std::false_type{});
        lsum += acc2.x + acc2.y;
        }
        m = m_new;
        // block-scale words of the PV MMA: P^ scale 1.0 (strict: per-row group
        // exponents, written above), V scale per 32-key group (strict: 1.0)
        if (!STRICT) tmem_st4(s_addr + 120, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        tmem_st4(s_addr + 124, vsf, vsf, vsf, vsf);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[w]);
      }
      // warpgroup-wide, so that the four warps leave together on a timeout
      ok = named_bar_and(2 + w, 128, ok && mbar_wait(&o_full[w], 0, status));
      if (ok) {
        tc_fence_after();
        // O = bf16(acc / l) straight from registers: 32 columns per TMEM load, written as
        // two 32-byte stores of the thread's row (16-byte ones if O is only 16-byte
        // aligned); the SM's store path drains them while the warpgroup leaves
        const float inv = 1.0f / lsum;
        const bool al32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
        __nv_bfloat16* orow = p.out + (tok * p.hq + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(o_addr + 32 * c, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * j]) * inv,
                                                      __uint_as_float(v[2 * j + 1]) * inv);
            pk[j] = *reinterpret_cast<uint32_t*>(&b2);
          }
          if (row_valid) {
            __nv_bfloat16* dst = orow + 32 * c;
            if (al32) {
              st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
              st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
        if (row_valid) p.lse[(int64_t)h * p.T + tok] = (m + __log2f(lsum) - 8.0f) * 0.69314718055994531f;
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

// Persistent forward of the MXFP8 route: one CTA per SM walks the (work item,
// query head) units of the cost-sorted work list in boustrophedon order -- in
// round r, CTA c takes unit r G + c when r is even and r G + G - 1 - c when r is
// odd (G CTAs) -- the assignment of the review's Algorithm 2 (step 05).  Nothing
// drains between units: the producer loads the next unit's Q tiles into the
// second Q buffer and its K/V tiles into the ring while the current unit still
// runs, the MMA warp issues the next unit's first QK^T as soon as its tiles have
// landed, and a warpgroup's epilogue (O = acc / l, LSE) overlaps the other
// warpgroup's last tiles and the next unit's first score MMAs.  A warpgroup reads
// its O accumulator before it hands in the first P^ tile of its next unit, so the
// first PV MMA of that unit (which overwrites O) never races the epilogue.
// Roles and TMEM columns are those of attn_fwd_kernel; the K/V block-scale words
// of the next tile are loaded into registers one tile ahead.
// Register split (setmaxnreg): the control warpgroup (producer, MMA warp) keeps 120
// registers, the two softmax warpgroups take 192; the shares add up to the launch
// allocation of 168 per thread, and the launch is refused with any other allocation
// (the increase could then never be granted).
constexpr int kPersistLaunchRegs = (65536 / kThreads) & ~7;
constexpr int kPersistRegCtl = 120;
constexpr int kPersistRegSoftmax = 192;
static_assert(kPersistRegCtl * 128 + kPersistRegSoftmax * 256 <= kPersistLaunchRegs * kThreads, "register split");

constexpr int kClcSlots = 4;     // answers of dynamic work requests in flight or unread

template <int D>
struct PersistSmem {
  static constexpr int kTileBytes = kTile * D;
  static constexpr int kQ = 0;                                   // [2 buffers][2 query tiles]
  static constexpr int kK = kQ + 4 * kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;            // [2 warpgroups]
  static constexpr int kMaxTabTiles = 1024;                       // per key tile: K word, V word
  static constexpr int kTab = kP + 2 * kTile * kTile;             // [2 warpgroups][kMaxTabTiles]
  static constexpr int kBar = kTab + 2 * kMaxTabTiles * 8;
  static constexpr int kClc = kBar + 256;                         // cancel answer (16 B), unit ring
  static constexpr int kBytes = kClc + 16 + 4 * kClcSlots;
  static constexpr int kAlloc = kBytes + 1024;
};

// One unit of the forward work: query tiles t0 (.. t0 + ntq - 1) of a document for
// query head h.  The query tile of warpgroup w sees key tiles [klo(w), khi(w)]; the
// unit loads the union [ulo, ulo + nkv) once, in increasing order.
struct FwdUnit {
  int h, hk, t0, ntq, doc_start, doc_len, nkv, ulo;
  int klo0, klo1, khi0, khi1;
  __device__ __forceinline__ int klo(int w) const { return w ? klo1 : klo0; }
  __device__ __forceinline__ int khi(int w) const { return w ? khi1 : khi0; }
  __device__ __forceinline__ int nk(int w) const { return w < ntq ? khi(w) - klo(w) + 1 : 0; }
};

template <bool WIN>
__device__ __forceinline__ FwdUnit fwd_unit(const PlanView& pv, int i, int hq, int hkv, Window win) {
  FwdUnit U;
  const int item_idx = i / hq;
  U.h = i % hq;
  U.hk = U.h / (hq / hkv);
  const int4 item = pv.fwd_items[item_idx];
  const int2 span = pv.fwd_span[item_idx];
  U.t0 = item.y;
  U.ntq = item.z;
  U.doc_start = span.x;
  U.doc_len = span.y;
  const int nt = (U.doc_len + kTile - 1) / kTile;
  U.klo0 = WIN ? win_klo(U.t0, win) : 0;
  U.khi0 = WIN ? win_khi(U.t0, nt, win) : U.t0;
  U.klo1 = U.ntq > 1 ? (WIN ? win_klo(U.t0 + 1, win) : 0) : U.klo0;
  U.khi1 = U.ntq > 1 ? (WIN ? win_khi(U.t0 + 1, nt, win) : U.t0 + 1) : U.khi0;
  U.ulo = U.klo0;                         // the later query tile's range starts and ends no earlier
  U.nkv = (U.ntq > 1 ? U.khi1 : U.khi0) - U.ulo + 1;
  return U;
}


// The CTA's sequence of units.  Static: the boustrophedon rounds over G = gridDim.x
// persistent CTAs.  Dynamic (DYN, Algorithm 2 steps 07 and 09): the grid has a CTA
// per possible unit, in the work list's cost order; a running CTA first takes the
// unit of its own index, and the producer, right after issuing the last K/V load of
// a unit, asks the hardware for the next CTA that has not started yet and takes over
// its unit (cluster launch control).  The answer lands in a ring slot that every
// role decodes; the MMA warp and the eight softmax warps hand the slot back.  A CTA
// stops at the first request that cancels nothing, or cancels a CTA past the last
// unit (those CTAs have no work; the ones never cancelled start and leave at once).
// The CTA's sequence of units.  Static: the boustrophedon rounds over G = gridDim.x
// persistent CTAs.  Dynamic (DYN, Algorithm 2 steps 07 and 09): the grid has a CTA
// per possible unit.  A CTA that starts draws a ticket from the plan's counter; right
// after issuing the last K/V load of a unit the producer asks the hardware to cancel
// the launch of a CTA that has not started yet (cluster launch control) and, if one
// was cancelled, draws the next ticket in its stead.  Ticket n is unit n of the
// cost-sorted list: the hardware hands out cancelled CTAs only roughly in index
// order (measured: up to about a wave out of place), so the tickets keep the units
// in cost order.  Every CTA below the unit count either starts or is cancelled, and
// each contributes a ticket, so the tickets cover every unit; each is run by the CTA
// that drew it, and one past the last unit ends a CTA.
// The producer puts each next unit into a ring slot; the MMA warp and the eight
// softmax warps read it and hand the slot back.
// A consumer warp's wait for the unit in slot (k - 1) % kClcSlots (out of line:
// inlined into the softmax loop it raises register pressure across the whole loop).
// Returns the unit, -1 when there is none, or -2 when the wait expired.
__device__ __noinline__ int wait_next_unit(uint64_t* full, uint64_t* empty, const int* unit_slot, int k, bool arrive,
                                           int* status) {
  const int sl = (k - 1) % kClcSlots;
  if (!__all_sync(0xffffffffu, mbar_wait(&full[sl], ((k - 1) / kClcSlots) & 1, status))) return -2;
  const int x = unit_slot[sl];
  __syncwarp();
  if (arrive) mbar_arrive(&empty[sl]);
  return x;
}

template <bool DYN>
struct UnitSeq {
  int c, G, n_units;
  int first;           // dynamic: the ticket drawn at the start
  int* unit_slot;      // [kClcSlots]
  uint64_t* full;      // [kClcSlots] unit published
  uint64_t* empty;     // [kClcSlots] unit read by the MMA warp and the softmax warps
  // unit number k of this CTA (k = 0, 1, ...), or -1 when there is none (ok turns
  // false when a wait expired).  A consumer is a whole converged warp (MMA warp: the
  // elected lane arrives; softmax warp: lane 0) and hands the slot back; the producer
  // (one thread) takes units 1, 2, ... from next().
  __device__ __forceinline__ int unit(int k, bool arrive, bool& ok, int* status) const {
    if constexpr (!DYN) {
      const int r = k;
      if ((int64_t)r * G >= n_units) return -1;
      const int i = r * G + ((r & 1) ? G - 1 - c : c);
      return i < n_units ? i : -1;
    } else {
      if (k == 0) return first < n_units ? first : -1;
      const int x = wait_next_unit(full, empty, unit_slot, k, arrive, status);
      ok = x != -2;
      return x < 0 ? -1 : x;
    }
  }
  // producer, after the last K/V load of unit k: unit k + 1, or -1
  __device__ __forceinline__ int next(int k, uint8_t* resp, uint64_t* clc_bar, int* ticket, bool& ok,
                                      int* status) const {
    const int sl = k % kClcSlots;
    if (k >= kClcSlots && !mbar_wait(&empty[sl], ((k / kClcSlots) - 1) & 1, status)) {
      ok = false;
      return -1;
    }
    fence_proxy_async_smem();        // the last answer was read before the next one lands
    mbar_arrive_expect_tx(clc_bar, 16);
    clc_try_cancel(resp, clc_bar);
    if (!mbar_wait(clc_bar, k & 1, status)) {
      ok = false;
      return -1;
    }
    int x = clc_cancelled_x(resp) >= 0 ? atomicAdd(ticket, 1) : -1;
    if (x >= n_units) x = -1;
    unit_slot[sl] = x;
    mbar_arrive(&full[sl]);
    return x;
  }
};

// WIN: a call with a window other than causal (noncausal, sliding); the causal
// builds carry none of its code.  DYN: dynamic work acquisition (UnitSeq).
template <int D, bool WIN = false, bool DYN = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = PersistSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bars + 0;                  // [2 Q buffers]
  uint64_t* q_empty = bars + 2;                 // [2]
  uint64_t* kv_full = bars + 4;                 // [kStages]
  uint64_t* kv_empty = kv_full + kStages;       // [kStages]
  uint64_t* s_full = kv_empty + kStages;        // [2 warpgroups]
  uint64_t* p_full = s_full + 2;                // [2]
  uint64_t* o_full = p_full + 2;                // [2]
  uint64_t* drain = o_full + 2;
  uint64_t* clc_full = drain + 1;               // [kClcSlots]
  uint64_t* clc_empty = clc_full + kClcSlots;   // [kClcSlots]
  uint64_t* clc_bar = clc_empty + kClcSlots;    // the cancel answer landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(clc_bar + 1);
  int* first_slot = reinterpret_cast<int*>(tmem_slot + 1);
  int* unit_slot = reinterpret_cast<int*>(smem + L::kClc + 16);   // [kClcSlots], after the answer
  int* status = const_cast<int*>(p.plan) + kPlanStatus;
  int* ticket = const_cast<int*>(p.plan) + kPlanFwdTicket;

  const PlanView pv = plan_view(p.plan, p.T, p.N);
  const int n_units = p.plan[kPlanFwdItems] * p.hq;
  // dynamic: a CTA past the last unit leaves before any set-up without a ticket (a CTA
  // below it contributes one ticket, drawn here or by the CTA that cancelled it, so
  // the tickets still cover every unit)
  if (DYN && (int)blockIdx.x >= n_units) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    if (DYN) *first_slot = atomicAdd(ticket, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kClcSlots; ++i) {
      mbar_init(&clc_full[i], 1);
      mbar_init(&clc_empty[i], 9);
    }
    mbar_init(clc_bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const UnitSeq<DYN> seq{(int)blockIdx.x, (int)gridDim.x, n_units, DYN ? *first_slot : 0, unit_slot, clc_full,
                         clc_empty};
  constexpr uint32_t kSCol[2] = {0, 256};
  constexpr uint32_t kOCol[2] = {128, 384};
  constexpr uint32_t kRowBytes = D;
  constexpr uint32_t kLayout = D == 128 ? kSwizzle128B : kSwizzle64B;
  constexpr uint32_t kAtom = 8 * D;
  if (warp < 4) setmaxnreg_dec<kPersistRegCtl>();
  else setmaxnreg_inc<kPersistRegSoftmax>();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int qn = 0;        // units loaded so far (Q buffer qn & 1)
      int kvc = 0;       // K/V tiles loaded so far (ring stage kvc % kStages)
      bool ok = true;
      int nxt = -1;
      for (int r = 0; ok; ++r) {
        const int i = (DYN && r > 0) ? nxt : seq.unit(r, false, ok, status);
        if (i < 0) break;
        const FwdUnit U = fwd_unit<WIN>(pv, i, p.hq, p.hkv, p.win);
        const int qb = qn & 1;
        if (qn >= 2 && !mbar_wait(&q_empty[qb], ((qn >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&q_full[qb], U.ntq * L::kTileBytes);
        for (int w = 0; w < U.ntq; ++w)
          tma_load_3d(smem + L::kQ + (2 * qb + w) * L::kTileBytes, &tm_q, &q_full[qb], 0, U.h,
                      U.doc_start + (U.t0 + w) * kTile);
        ++qn;
        for (int u = 0; u < U.nkv; ++u, ++kvc) {
          const int st = kvc % kStages;
          if (kvc >= kStages && !mbar_wait(&kv_empty[st], ((kvc / kStages) - 1) & 1, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kv_full[st], 2 * L::kTileBytes);
          const int ku = U.ulo + u;
          tma_load_3d(smem + L::kK + st * L::kTileBytes, &tm_k, &kv_full[st], 0, U.hk, U.doc_start + ku * kTile);
          tma_load_3d(smem + L::kV + st * L::kTileBytes, &tm_v, &kv_full[st], 0, U.hk, U.doc_start + ku * kTile);
        }
        if (DYN && ok) nxt = seq.next(r, smem + L::kClc, clc_bar, ticket, ok, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    const uint32_t base16 = (smem_u32(smem) & 0x3FFFFu) >> 4;
    auto b16 = [&]() {
      uint32_t x;
      asm volatile("mov.b32 %0, %1;" : "=r"(x) : "r"(base16));
      return x;
    };
    auto issue_s = [&](int w, int qb, int st) {
#pragma unroll
      for (int s = 0; s < D / 32; ++s)
        if (leader)
          mma_f8(tbase + kSCol[w], sdesc_at(b16(), L::kQ + (2 * qb + w) * L::kTileBytes + 32 * s, 16, kAtom, kLayout),
                 sdesc_at(b16(), L::kK + st * L::kTileBytes + 32 * s, 16, kAtom, kLayout), idesc_f8(128, 128, 0, 0),
                 s > 0);
    };
    auto issue_pv = [&](int w, int st, bool acc) {
#pragma unroll
      for (int s = 0; s < 4; ++s)
        if (leader)
          mma_mxf8(tbase + kOCol[w], sdesc_at(b16(), L::kP + w * kTile * kTile + 32 * s, 16, 1024, kSwizzle128B),
                   sdesc_at(b16(), L::kV + st * L::kTileBytes + s * 32 * kRowBytes, kAtom, kAtom, kLayout),
                   idesc_mxf8(128, D, 0, 1, s, s), tbase + kSCol[w] + 120, tbase + kSCol[w] + 124, acc || s > 0);
    };
    int qn = 0, kvc = 0;
    int pcnt0 = 0, pcnt1 = 0;   // P^ tiles handed in by each warpgroup so far
    bool ok = true;
    int i = seq.unit(0, leader, ok, status);
    for (int r = 0; i >= 0 && ok; i = seq.unit(++r, leader, ok, status)) {
      const FwdUnit U = fwd_unit<WIN>(pv, i, p.hq, p.hkv, p.win);
      const int qb = qn & 1;
      ok = warp_wait(&q_full[qb], (qn >> 1) & 1, status) &&
           warp_wait(&kv_full[kvc % kStages], (kvc / kStages) & 1, status);
      if (!ok) break;
      tc_fence_after();
      for (int w = 0; w < U.ntq; ++w) {
        if (U.klo(w) != U.ulo) continue;         // its first key tile comes later
        issue_s(w, qb, kvc % kStages);
        if (leader) mma_commit(&s_full[w]);
      }
      for (int uu = 0; uu < U.nkv && ok; ++uu) {
        const int u = U.ulo + uu;                // key tile (document-local index)
        const int st = (kvc + uu) % kStages;
        const int st1 = (kvc + uu + 1) % kStages;
        bool next_loaded = false;
        auto load_next = [&]() {
          if (!next_loaded) {
            ok = warp_wait(&kv_full[st1], ((kvc + uu + 1) / kStages) & 1, status);
            if (ok) tc_fence_after();
            next_loaded = true;
          }
          return ok;
        };
        for (int w = 0; w < U.ntq && ok; ++w) {
          if (u < U.klo(w) || u > U.khi(w)) continue;
          ok = warp_wait(&p_full[w], (w ? pcnt1 : pcnt0) & 1, status);
          if (w) ++pcnt1;
          else ++pcnt0;
          if (!ok) break;
          tc_fence_after();
          issue_pv(w, st, u > U.klo(w));
          if (u + 1 <= U.khi(w)) {
            if (!load_next()) break;
            issue_s(w, qb, st1);
            if (leader) mma_commit(&s_full[w]);
          } else {
            if (leader) mma_commit(&o_full[w]);
          }
        }
        // a warpgroup whose range starts at the next key tile gets its first S now
        for (int w = 1; w < U.ntq && ok; ++w) {
          if (U.klo(w) != u + 1) continue;
          if (!load_next()) break;
          issue_s(w, qb, st1);
          if (leader) mma_commit(&s_full[w]);
        }
        if (leader) mma_commit(&kv_empty[st]);
      }
      if (leader) mma_commit(&q_empty[qb]);
      kvc += U.nkv;
      ++qn;
    }
    if (!ok && leader) {
      // timed out: make sure nothing we issued is still running before TMEM is freed
      mma_commit(drain);
      mbar_wait(drain, 0, status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int w = (warp - 4) >> 2;        // warpgroup = query tile t0 + w of each unit
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;    // row within the tile (= TMEM lane)
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_addr = lane_base + kSCol[w], o_addr = lane_base + kOCol[w];
    uint8_t* sP = smem + L::kP + w * kTile * kTile;
    const bool al32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
    int scnt = 0, ocnt = 0;               // S tiles and units of this warpgroup so far
    bool ok = true;
    // static order: the Q scale byte of this thread's row and its two first K/V table
    // entries (units of up to 64 key tiles) of the warpgroup's next unit, loaded before
    // this unit's epilogue so that their latency overlaps it
    uint32_t pre_kv = 0, pre_q = 0;
    int pre_unit = -1;
    for (int rr = 0; ok; ++rr) {
      const int i = seq.unit(rr, lane == 0, ok, status);
      if (i < 0) break;
      const FwdUnit U = fwd_unit<WIN>(pv, i, p.hq, p.hkv, p.win);
      if (w >= U.ntq) continue;
      const int t = U.t0 + w;
      const int qrow_local = t * kTile + r;
      const bool row_valid = qrow_local < U.doc_len;
      const int64_t tok = (int64_t)U.doc_start + qrow_local;
      const bool pre = !DYN && pre_unit == i;
      const float fq = p.scale_log2 * (pre ? (row_valid ? ue8m0_to_f32(pre_q) : 1.0f)
                                           : scale_of(p.q_scales, tok, p.hq, U.h, row_valid));
      const int nk = U.nk(w), klo = U.klo(w);
      // K and V block-scale bytes of every key tile of the unit (one per 32-key group,
      // 127 past the document end), staged in this warpgroup's own table (tiles past
      // its capacity read them from global memory); each thread's loads come before
      // its stores.  The warpgroup barrier of the previous epilogue separates the last
      // reads of the old table from these stores.
      uint32_t* tab = reinterpret_cast<uint32_t*>(smem + L::kTab) + w * (2 * L::kMaxTabTiles);
      uint8_t* tb = reinterpret_cast<uint8_t*>(tab);
      const int ntab = min(nk, L::kMaxTabTiles);
      auto scale_bytes = [&](int uu, int g, uint32_t& kb, uint32_t& vb) {
        const int kl = uu * kTile + g * 32;
        const bool kv = kl < U.doc_len;
        const int64_t ktok = (int64_t)U.doc_start + kl;
        kb = kv ? __ldg(p.k_scales + ktok * p.hkv + U.hk) : 127u;
        vb = kv ? __ldg(p.v_scales + ktok * p.hkv + U.hk) : 127u;
      };
      if (pre && ntab * 4 <= 256) {
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const int e = r + 128 * q2;
          if (e < ntab * 4) {
            tb[(e >> 2) * 8 + (e & 3)] = (uint8_t)(pre_kv >> (16 * q2));
            tb[(e >> 2) * 8 + 4 + (e & 3)] = (uint8_t)(pre_kv >> (16 * q2 + 8));
          }
        }
      } else {
        for (int e = r; e < ntab * 4; e += 128) {
          uint32_t kb, vb;
          scale_bytes(klo + (e >> 2), e & 3, kb, vb);
          tb[(e >> 2) * 8 + (e & 3)] = (uint8_t)kb;
          tb[(e >> 2) * 8 + 4 + (e & 3)] = (uint8_t)vb;
        }
      }
      named_bar_sync(2 + w, 128);
      float m = -INFINITY, lsum = 0.f;
      for (int uu = 0; uu < nk; ++uu) {
        const int u = klo + uu;                // key tile (document-local index)
        uint32_t kw = 0, vsf = 0;
        if (uu < ntab) {
          const uint2 kv2 = *reinterpret_cast<const uint2*>(tab + 2 * uu);
          kw = kv2.x;
          vsf = kv2.y;
        } else {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t kb, vb;
            scale_bytes(u, g, kb, vb);
            kw |= kb << (8 * g);
            vsf |= vb << (8 * g);
          }
        }
        float fk[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) fk[g] = fq * ue8m0_to_f32((kw >> (8 * g)) & 0xFFu);
        // a tile with a hidden pair (causal: the diagonal one) or keys past the document
        // end takes the masked variants, where this row sees the tile's keys [klim, khim]
        const bool diag = WIN ? win_masked(t, u, U.doc_len, p.win) : u == t;
        auto key_bounds = [&](int& klim, int& khim) {
          if constexpr (WIN) {
            const int qi = t * kTile + r;
            klim = p.win.left < 0 ? 0 : qi - p.win.left - u * kTile;
            khim = min(U.doc_len - 1 - u * kTile, p.win.right < 0 ? kTile : qi + p.win.right - u * kTile);
          } else {                             // causal: the keys up to the query
            klim = 0;
            khim = r;
          }
        };
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[w], scnt & 1, status));
        ++scnt;
        if (!ok) break;
        tc_fence_after();
        // pass 1: row max of x = S * log2(e) over visible keys (the column factor is a
        // positive power of two times a constant, so max(v * f) = f * max(v))
        float mx = -INFINITY;
        if (!diag) {
          float cm[4];
          {                                     // the four loads in flight together (values unused)
            uint32_t v0[32], v1[32], v2[32], v3[32];
            tmem_ld32_max(s_addr, v0, cm[0]);
            tmem_ld32_max(s_addr + 32, v1, cm[1]);
            tmem_ld32_max(s_addr + 64, v2, cm[2]);
            tmem_ld32_max(s_addr + 96, v3, cm[3]);
            tmem_ld_wait();
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) mx = fmaxf(mx, cm[g] * fk[g]);
        } else {
          int klim, khim;
          key_bounds(klim, khim);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];
            tmem_ld32(s_addr + 32 * g, v);
            tmem_ld_wait();
            float b = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              b = (g * 32 + j >= klim && g * 32 + j <= khim) ? fmaxf(b, __uint_as_float(v[j])) : b;
            mx = fmaxf(mx, b * fk[g]);
          }
        }
        const float m_new = fmaxf(m, mx);
        // 0 on the first tile; 1 while the row has seen no key (a window that starts
        // further right), where m - m_new would be -inf - -inf
        const float alpha = (WIN && m_new == -INFINITY) ? 1.0f : fast_exp2(m - m_new);
        // rescale the running O row when the max moved (warp-uniform decision)
        if (uu > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t v[32];
            tmem_ld32(o_addr + 32 * cc, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            tmem_st32(o_addr + 32 * cc, v);
          }
          tmem_st_wait();
        }
        lsum *= alpha;
        const float neg = 8.0f - m_new;
        // pass 2: boosted weights 2^(x - m + 8) and their E4M3 codes into the P tile
        // (built twice: the causal mask only on the diagonal tile)
        float2 acc2 = make_float2(0.f, 0.f);
        auto pass2 = [&](auto diag_tile) {
          constexpr bool kDiag = decltype(diag_tile)::value;
          int klim = 0, khim = 0;
          if constexpr (kDiag) key_bounds(klim, khim);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];
            tmem_ld32(s_addr + 32 * g, v);
            tmem_ld_wait();
            uint32_t packed[8];
            const float2 f2 = make_float2(fk[g], fk[g]), n2 = make_float2(neg, neg);
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float2 x0 = ffma2(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), f2, n2);
              float2 x1 = ffma2(make_float2(__uint_as_float(v[j + 2]), __uint_as_float(v[j + 3])), f2, n2);
              float2 p0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
              float2 p1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
              if (kDiag) {
                const int kc = g * 32 + j;
                p0.x = (kc >= klim && kc <= khim) ? p0.x : 0.f;
                p0.y = (kc + 1 >= klim && kc + 1 <= khim) ? p0.y : 0.f;
                p1.x = (kc + 2 >= klim && kc + 2 <= khim) ? p1.x : 0.f;
                p1.y = (kc + 3 >= klim && kc + 3 <= khim) ? p1.y : 0.f;
              }
              acc2 = fadd2(acc2, fadd2(p0, p1));
              packed[j >> 2] = (uint32_t)e4m3x2(p0.x, p0.y) | ((uint32_t)e4m3x2(p1.x, p1.y) << 16);
            }
            *reinterpret_cast<uint4*>(sP + swz_offset(r, 32 * g, 128)) =
                make_uint4(packed[0], packed[1], packed[2], packed[3]);
            *reinterpret_cast<uint4*>(sP + swz_offset(r, 32 * g + 16, 128)) =
                make_uint4(packed[4], packed[5], packed[6], packed[7]);
          }
        };
        if (diag) pass2(std::true_type{});
        else pass2(std::false_type{});
        lsum += acc2.x + acc2.y;
        m = m_new;
        // block-scale words of the PV MMA: P^ scale 1.0, V's token-block scales
        tmem_st4(s_addr + 120, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
        tmem_st4(s_addr + 124, vsf, vsf, vsf, vsf);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[w]);
      }
      if constexpr (!DYN) {
        // the next unit of this warpgroup in the static order (if it takes part in it)
        pre_unit = -1;
        bool tmp_ok = true;
        const int i2 = seq.unit(rr + 1, false, tmp_ok, status);
        if (i2 >= 0) {
          const FwdUnit U2 = fwd_unit<WIN>(pv, i2, p.hq, p.hkv, p.win);
          if (w < U2.ntq) {
            pre_unit = i2;
            const int q2l = (U2.t0 + w) * kTile + r;
            const bool v2 = q2l < U2.doc_len;
            pre_q = v2 ? __ldg(p.q_scales + ((int64_t)U2.doc_start + q2l) * p.hq + U2.h) : 127u;
            pre_kv = 0;
            const int ntab2 = min(U2.nk(w), L::kMaxTabTiles), klo2 = U2.klo(w);
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
              const int e = r + 128 * q2;
              if (e < ntab2 * 4) {
                const int kl = (klo2 + (e >> 2)) * kTile + (e & 3) * 32;
                const bool kv = kl < U2.doc_len;
                const int64_t ktok = (int64_t)U2.doc_start + kl;
                const uint32_t kb = kv ? __ldg(p.k_scales + ktok * p.hkv + U2.hk) : 127u;
                const uint32_t vb = kv ? __ldg(p.v_scales + ktok * p.hkv + U2.hk) : 127u;
                pre_kv |= (kb | vb << 8) << (16 * q2);
              }
            }
          }
        }
      }
      // warpgroup-wide, so that the four warps leave together on a timeout
      ok = named_bar_and(2 + w, 128, ok && mbar_wait(&o_full[w], ocnt & 1, status));
      ++ocnt;
      if (!ok) break;
      tc_fence_after();
      // O = bf16(acc / l) straight from registers (two 32-byte stores per 32 columns;
      // 16-byte ones if O is only 16-byte aligned).  These TMEM loads complete before
      // this warpgroup hands in the first P^ tile of its next unit, which is what the
      // next unit's first (overwriting) PV MMA waits for.
      const float inv = 1.0f / lsum;
      __nv_bfloat16* orow = p.out + (tok * p.hq + U.h) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(o_addr + 32 * cc, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * j]) * inv, __uint_as_float(v[2 * j + 1]) * inv);
          pk[j] = *reinterpret_cast<uint32_t*>(&b2);
        }
        if (row_valid) {
          __nv_bfloat16* dst = orow + 32 * cc;
          if (al32) {
            st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
            st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      }
      if (row_valid) p.lse[(int64_t)U.h * p.T + tok] = (m + __log2f(lsum) - 8.0f) * 0.69314718055994531f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// Rows outside every document: O = 0, LSE = +inf.
template <int D>
__global__ void fwd_tail_kernel(const int* plan, int T, int hq, __nv_bfloat16* out, float* lse) {
  if (blockIdx.x == 0 && threadIdx.x == 0) const_cast<int*>(plan)[kPlanFwdTicket] = 0;   // for the next forward
  const int valid = plan[kPlanValid];
  const int64_t n = (int64_t)(T - valid) * hq;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = valid + i / hq;
    const int h = (int)(i % hq);
    uint4* dst = reinterpret_cast<uint4*>(out + (row * hq + h) * D);
#pragma unroll
    for (int j = 0; j < D / 8; ++j) dst[j] = make_uint4(0, 0, 0, 0);
    lse[(int64_t)h * T + row] = INFINITY;
  }
}

template <int D, bool STRICT>
cudaError_t launch_fwd_d(const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                         const void* vs, const int32_t* cu, int N, int T, int hq, int hkv, float scale,
                         const void* plan, void* out, float* lse, cudaStream_t stream, void* const* ev, Window win,
                         bool dynamic) {
  CUtensorMap tq, tk, tv;
  if (!make_tmap_u8_3d(&tq, qc, D, hq, T, D, (uint64_t)hq * D, D, kTile) ||
      !make_tmap_u8_3d(&tk, kc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile) ||
      !make_tmap_u8_3d(&tv, vc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.q_scales = static_cast<const uint8_t*>(qs);
  p.k_scales = static_cast<const uint8_t*>(ks);
  p.v_scales = static_cast<const uint8_t*>(vs);
  p.cu = cu;
  p.plan = static_cast<const int*>(plan);
  p.N = N;
  p.T = T;
  p.hq = hq;
  p.hkv = hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.win = win;
  const int64_t max_items = (int64_t)T / (kTile * kItemTiles) + N + 1;
  const int64_t grid = max_items * hq;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaError_t e;
  if constexpr (STRICT) {
    constexpr int smem = FwdSmem<D>::kAlloc;
    e = prepare_kernel<attn_fwd_kernel<D, STRICT>>(smem);
    if (e != cudaSuccess) return e;
    if (ev) record_timing_event(ev[0], stream);
    attn_fwd_kernel<D, STRICT><<<(unsigned)grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  } else {
    // persistent, static order: one CTA per SM (fewer when there are fewer units than
    // SMs); dynamic order (causal calls only): a CTA per possible unit
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = PersistSmem<D>::kAlloc;
    int regs = 0;
    const bool causal = win.left < 0 && win.right == 0;
    const bool dyn = causal && dynamic;
    if (dyn) {
      e = prepare_kernel<attn_fwd_persist_kernel<D, false, true>>(smem, &regs);
    } else {
      e = causal ? prepare_kernel<attn_fwd_persist_kernel<D, false>>(smem, &regs)
                 : prepare_kernel<attn_fwd_persist_kernel<D, true>>(smem, &regs);
    }
    if (e != cudaSuccess) return e;
    if (regs != kPersistLaunchRegs) return cudaErrorInvalidConfiguration;
    const unsigned pgrid = (unsigned)(grid < sms ? grid : sms);
    if (ev) record_timing_event(ev[0], stream);
    if (dyn) {
      attn_fwd_persist_kernel<D, false, true><<<(unsigned)grid, kThreads, smem, stream>>>(tq, tk, tv, p);
    } else {
      if (causal) attn_fwd_persist_kernel<D, false><<<pgrid, kThreads, smem, stream>>>(tq, tk, tv, p);
      else attn_fwd_persist_kernel<D, true><<<pgrid, kThreads, smem, stream>>>(tq, tk, tv, p);
    }
  }
  e = cudaGetLastError();
  if (ev) record_timing_event(ev[1], stream);
  if (e != cudaSuccess) return e;
  fwd_tail_kernel<D><<<152, 256, 0, stream>>>(static_cast<const int*>(plan), T, hq, static_cast<__nv_bfloat16*>(out),
                                              lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tail(int D, const void* plan, int T, int hq, void* out, float* lse, cudaStream_t stream) {
  if (D == 128)
    fwd_tail_kernel<128><<<152, 256, 0, stream>>>(static_cast<const int*>(plan), T, hq,
                                                  static_cast<__nv_bfloat16*>(out), lse);
  else if (D == 64)
    fwd_tail_kernel<64><<<152, 256, 0, stream>>>(static_cast<const int*>(plan), T, hq,
                                                 static_cast<__nv_bfloat16*>(out), lse);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_fwd(int D, const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                       const void* vs, const int32_t* cu, int N, int T, int hq, int hkv, float scale,
                       const void* plan, void* out, float* lse, cudaStream_t stream, void* const* ev, bool strict,
                       Window win, bool dynamic) {
#define FLAMIA_FWD_ARGS qc, qs, kc, ks, vc, vs, cu, N, T, hq, hkv, scale, plan, out, lse, stream, ev, win, dynamic
  if (strict && (win.left >= 0 || win.right != 0)) return cudaErrorInvalidValue;   // the strict kernel is causal
  if (D == 128 && strict) return launch_fwd_d<128, true>(FLAMIA_FWD_ARGS);
  if (D == 128) return launch_fwd_d<128, false>(FLAMIA_FWD_ARGS);
  if (D == 64 && strict) return launch_fwd_d<64, true>(FLAMIA_FWD_ARGS);
  if (D == 64) return launch_fwd_d<64, false>(FLAMIA_FWD_ARGS);
#undef FLAMIA_FWD_ARGS
  return cudaErrorInvalidValue;
}

}  // namespace flamia
