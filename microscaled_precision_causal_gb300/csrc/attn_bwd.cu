// FLAMIA backward attention (steps a8-a12 of the hot path) plus the dQ boost
// and dQ finalisation kernels.
//
// FLAMIA technical review, Algorithm 1 steps 10-16 (and section 7, "Softmax
// and TMEM resources": token scales are applied by the compute warps after the
// feature-axis MMAs, so dP needs no TMEM scale operands):
//   S^T  = K Q^T            (unscaled E4M3 MMA, factors s_K(j) s_Q(i) scale after)
//   P    = 2^(x - LSE*log2 e)      (exactly the forward's tiles and masks)
//   dP^T = V dO^T           (unscaled E4M3 MMA, factors s_V(j) s_dO(i) after)
//   dS   = P o (dP - D)
//   dS^  = E4M3 with one round-up exponent per document-local 32x32 block
//          (section 3: the 32x32 square serves both contraction axes)
//   dV  += E4M3(2^8 P)^T dO^ / 2^8     (MXF8, dO's scale per 32 queries)
//   dK  += dS^^T Q^                    (MXF8, dS block and Q scales per 32 queries)
//   dQp  = dS^ K^                      (MXF8, same dS codes read transposed; at
//                                       d = 128 computed as dQp^T = K^T dS^^T in two
//                                       64-query halves)
//   dQacc += fp16(c * dQp)             (section 4, boosted FP16 partials; staged in
//                                       shared memory, added into the accumulator
//                                       with bulk fp16 reduce copies)
//
// One CTA per (document-local 128-key tile, kv head); it visits every query
// head of the kv head's group and every query tile at or after the key tile.
// Roles (896 threads at d = 128, 768 with the strict options, 512 at d = 64):
//   warp 0      TMA producer (K, V once; Q and dO codes per step)
//   warp 1      MMA issuer (a converged warp; one elected lane issues)
//   warp 2      TMEM allocator
//   warp 3      per-query row data of the next steps (LSE, D, chunk scales) into SMEM
//   warps 4..   compute warpgroups (four at d = 128, two at d = 64): each owns
//               32 of the 128 query columns of a step and 32 of the head-dim
//               columns of the dK / dV accumulators
//   last WGs    dQ readout (two at d = 128): TMEM -> fp16 staging -> bulk reduce
//               into the accumulator
// Thread = key row while building P^ and dS^ codes.  TMEM: S^T [0,128), dP^T
// [128,256), dV [256, 256+D), dK [384, 384+D).  P^ (dV's A operand) goes to TMEM
// into S^T columns its warpgroup has read (default and mixed routes) or to SMEM
// (strict).  At d = 128 the dQ^T halves take dP^T's first 64 columns once dS^ is
// built; at d = 64 the dQ partial has [320, 384).  Block-scale words: dV's in
// S^T's columns [0, 8) ([104, 112) strict), written once S^T has been read; dK's
// and dQ's in dP^T's columns [104, 124) (at d = 64 dQ's in [448, 456)), written
// once dP^T has been read.  Per step the MMA warp issues dV(k) as soon as P^ is
// written, then S^T(k+1) (the exponentials of the next step overlap the dS^ work
// of this one), then dK(k), dQ(k) and dP^T(k+1) once the dQ columns have been
// read.  The mixed route's S~ MMA (NVFP4) takes its scale words from dP^T's
// columns [64, 80), written by the readout warpgroups once dP^T has been read.  dK
// and dV are staged as bf16 and
// leave by TMA stores (a document's partial last tile by row stores).
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.h"

namespace flamia {

namespace {

constexpr int kQStages = 2;
// Compute warpgroups: each owns 32 of the 128 query columns of a step (as 4 / kWG
// chunks of 32) and 32 of the head-dim columns of dQ / dK / dV.
// Warpgroups: 0 = control (TMA producer, MMA issuer, TMEM allocator, row data),
// 1 .. kWG = compute (P^ and dS^), then kRO dQ readout warpgroups (two at d = 128
// outside the strict options, each reading 32 of a dQ^T half's 64 columns).  The
// control and readout warpgroups hand registers to the compute warpgroups
// (setmaxnreg); the per-role totals fit the launch allocation:
// kRegCtl x 128 + kRegRead x 128 kRO + kRegHigh x kCompute <= kLaunchRegs x kThreads.
template <int D, bool STRICT = false>
struct BwdShape {
  static constexpr int kWG = D == 128 ? 4 : 2;
  static constexpr int kChunksPerWG = 4 / kWG;
  static constexpr int kCols = D / kWG;                     // head-dim columns per slice (32)
  static constexpr int kCompute = 128 * kWG;
  static constexpr int kRO = D == 128 && !STRICT ? 2 : 1;
  static constexpr int kThreads = 128 + kCompute + 128 * kRO;
  static constexpr int kLaunchRegs = (65536 / kThreads) & ~7;   // 72 / 80 at d = 128, 128 at d = 64
  static constexpr int kRegCtl = D == 128 ? 48 : 64;
  static constexpr int kRegRead = D == 128 ? (kRO == 2 ? 48 : 80) : 64;
  static constexpr int kRegHigh = D == 128 ? 88 : 192;
  static_assert(kRegCtl * 128 + kRegRead * 128 * kRO + kRegHigh * kCompute <= kLaunchRegs * kThreads,
                "register split");
};

struct BwdParams {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint8_t* do_scales;
  const float* lse;        // [hq, T]
  const float* dvec;       // [hq, T]
  const float* boost;      // [N, hq]
  const int32_t* cu;
  const int* plan;
  int N, T, hq, hkv;
  float scale_log2;        // softmax scale * log2(e)
  float scale;
  const uint8_t* q4_scales;   // mixed route: E4M3 scale codes [T, hq, D/16] of the NVFP4 score operands
  const uint8_t* k4_scales;   // [T, hkv, D/16]
  __half* dq_acc;          // fp16 accumulator chunks (dq_chunk_elems layout)
  __nv_bfloat16* dk;       // [T, hkv, D]
  __nv_bfloat16* dv;
  float* dbg;              // diagnostic build only: fp32 P and dS, [2, hq, T, T]
  Window win;              // visible keys (causal: right = 0); strict and mixed are causal only
};

template <int D, bool MIXED>
struct BwdSmem {
  static constexpr int kTileBytes = kTile * D;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                  // [kQStages]
  static constexpr int kDO = kQ + kQStages * kTileBytes;      // [kQStages]
  static constexpr int kPt = kDO + kQStages * kTileBytes;     // P^ codes, [key][query] (strict route)
  static constexpr int kDS = kPt + kTile * kTile;             // dS^ codes, [key][query]
  static constexpr int kRow = kDS + kTile * kTile;            // per-query data, 2 buffers
  // per-query row data: -lse2[128], -D[128], chunk scale bytes[8] (4 words reserved),
  // then (strict) s_Q[128] and s_dO[128] as floats
  static constexpr int kRowBuf = (128 * 2 + 4 + 128 * 2) * 4;
  static constexpr int kE = kRow + 2 * kRowBuf;               // 16 block exponents (+ strict per-row exponents)
  static constexpr int kStageBytes = kTile * BwdShape<D>::kCols * 2;   // one warpgroup's fp16 slice of the dQ tile
  static constexpr int kStage = (kE + 64 + 1024 + 1023) & ~1023;   // [warpgroup][2 buffers]
  static_assert(D != 128 || 2 * BwdShape<D>::kWG * kStageBytes == 2 * 32768, "two 32 KB dQ^T staging buffers");
  static constexpr int kScoreBytes = kTile * D / 2;           // mixed route: one E2M1 score-operand tile
  static constexpr int kK4 = kStage + 2 * BwdShape<D>::kWG * kStageBytes;
  static constexpr int kQ4 = kK4 + (MIXED ? kScoreBytes : 0);          // [kQStages]
  static constexpr int kBar = kQ4 + (MIXED ? kQStages * kScoreBytes : 0);
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = kBytes + 1024;
};

// DBG: a diagnostic build that also writes the fp32 P and dS of every visible pair
// (default route, small problems); the production builds carry none of its code.
// WIN: a call with a window other than causal (noncausal, sliding); the causal
// builds carry none of its code.  ROT: Q and K were rotated by H / 2^k before
// quantization (H the +-1 Hadamard matrix, k = ceil(log2(D) / 2)); dK is rotated
// back by the same map in the epilogue (dQ in its finalise kernel).
template <int D, bool STRICT, bool MIXED, bool DBG = false, bool WIN = false, bool ROT = false>
__global__ void __launch_bounds__(BwdShape<D, STRICT>::kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_q4, const __grid_constant__ CUtensorMap tm_k4,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const BwdParams p) {
  static_assert(!(STRICT && MIXED), "the strict options and the mixed route are separate");
  static_assert(!MIXED || D == 128, "the mixed route is built for head_dim 128");
  static_assert(!DBG || (!STRICT && !MIXED), "the diagnostic build covers the default route");
  static_assert(!WIN || (!STRICT && !MIXED), "the strict options and the mixed route are causal");
  static_assert(!ROT || (!STRICT && !MIXED && !DBG), "the rotation is built for the MXFP8 route");
  using L = BwdSmem<D, MIXED>;
  using Shape = BwdShape<D, STRICT>;
  constexpr int kWG = Shape::kWG, kCPW = Shape::kChunksPerWG, kCols = Shape::kCols;
  constexpr int kCompute = Shape::kCompute, kRO = Shape::kRO;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bars + 0;
  uint64_t* qd_full = bars + 1;              // [kQStages]
  uint64_t* qd_empty = bars + 1 + kQStages;  // [kQStages]
  uint64_t* row_full = bars + 1 + 2 * kQStages;   // [2]
  uint64_t* row_empty = row_full + 2;             // [2]
  uint64_t* s_full = row_empty + 2;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* dq_full = s_full + 3;
  uint64_t* dq_empty = s_full + 4;
  uint64_t* acc_full = s_full + 5;
  uint64_t* sf_ready = s_full + 6;            // mixed: score scale words of step 0 written
  uint64_t* pt_full = s_full + 7;             // P^ tile and the dV scale words written (every compute thread;
                                              // strict: warpgroup 0 after a barrier of all of them)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 8);
  int* status = const_cast<int*>(p.plan) + kPlanStatus;

  const int n_items = p.plan[kPlanBwdItems];
  const int item_idx = blockIdx.x / p.hkv;
  const int hk = blockIdx.x % p.hkv;
  if (item_idx >= n_items) return;
  const PlanView pv = plan_view(p.plan, p.T, p.N);
  const int4 item = pv.bwd_items[item_idx];
  const int2 span = pv.bwd_span[item_idx];      // loaded alongside the item (no dependent load)
  const int doc = item.x, u = item.y;
  const int doc_start = span.x;
  const int doc_len = span.y;
  const int nt = (doc_len + kTile - 1) / kTile;
  const int g = p.hq / p.hkv;
  // the query tiles that see this key tile under the call's window (causal: u .. nt - 1)
  const int tlo = WIN ? win_tlo(u, p.win) : u;
  const int qtiles = WIN ? win_thi(u, nt, p.win) - tlo + 1 : nt - u;
  const int nsteps = g * qtiles;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&row_full[i], 32);
      mbar_init(&row_empty[i], kCompute);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, kCompute);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128 * kRO);
    mbar_init(acc_full, 1);
    mbar_init(sf_ready, 128 * kRO);
    mbar_init(pt_full, STRICT ? 128 : kCompute);
    fence_mbar_init();
    // the producer's first loads (K, V and the first kQStages steps' Q, dO) start
    // before the TMEM allocation and the CTA barrier
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    mbar_arrive_expect_tx(kv_full, 2 * L::kTileBytes + (MIXED ? L::kScoreBytes : 0));
    tma_load_3d(smem + L::kK, &tm_k, kv_full, 0, hk, doc_start + u * kTile);
    tma_load_3d(smem + L::kV, &tm_v, kv_full, 0, hk, doc_start + u * kTile);
    if (MIXED) tma_load_3d(smem + L::kK4, &tm_k4, kv_full, 0, hk, doc_start + u * kTile);
    for (int k = 0; k < nsteps && k < kQStages; ++k) {
      const int h = hk * g + k / qtiles, t = tlo + k % qtiles;
      mbar_arrive_expect_tx(&qd_full[k], 2 * L::kTileBytes + (MIXED ? L::kScoreBytes : 0));
      tma_load_3d(smem + L::kQ + k * L::kTileBytes, &tm_q, &qd_full[k], 0, h, doc_start + t * kTile);
      tma_load_3d(smem + L::kDO + k * L::kTileBytes, &tm_do, &qd_full[k], 0, h, doc_start + t * kTile);
      if (MIXED) tma_load_3d(smem + L::kQ4 + k * L::kScoreBytes, &tm_q4, &qd_full[k], 0, h, doc_start + t * kTile);
    }
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool compute_wg = warp >= 4 && warp < 4 + 4 * kWG;
  const uint32_t tbase = *tmem_slot;
  constexpr uint32_t kS = 0, kP = 128, kDV = 256, kDK = 384;
  // dQ: at d = 128 (default and mixed routes) dQ^T = K^T dS^T in two 64-query halves
  // into the first 64 dP columns (TMEM is full: S, dP, dV, dK); at d = 64 the
  // query-major dQ partial sits in free columns.  Block-scale words: dV's in the S
  // columns (written after P), dK's and dQ's in the dP columns (written after dS),
  // so S of the next step can be issued right after dV.
  constexpr bool kDQT = D == 128 && !STRICT;
  constexpr uint32_t kDQ = D == 128 ? kP : 320;
  // dV: A 4 words, B 4 words; default and mixed routes: in S columns only warpgroup 0
  // reads (it writes them right after its own S load, so no barrier of all the compute
  // warpgroups is needed before dV)
  constexpr uint32_t kSFV = STRICT ? kS + 104 : kS;
  // P^ as dV's A operand: default and mixed routes in TMEM, 8 columns per 32-query chunk c at
  // kPtCol + 32 c, inside the S^T columns that chunk's warpgroup has itself just read (the
  // next step's S^T, issued after dV, overwrites them); the strict route stages it in SMEM
  constexpr bool kPtT = !STRICT;
  constexpr uint32_t kPtCol = kS + 16;
  constexpr uint32_t kSFK = kP + 104;       // dK: A 4, B 4
  constexpr uint32_t kSFQ = D == 128 ? kP + 112 : 448;   // dQ: A 4, B 4 (d = 128: B lo 4, B hi 4)
  constexpr uint32_t kLayout = D == 128 ? kSwizzle128B : kSwizzle64B;
  constexpr uint32_t kAtom = 8 * D;
  float* rowbuf = reinterpret_cast<float*>(smem + L::kRow);

  if (warp < 4) {
  setmaxnreg_dec<Shape::kRegCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int k = kQStages; k < nsteps; ++k) {     // K, V and the first kQStages steps: prologue
        const int st = k % kQStages;
        if (!mbar_wait(&qd_empty[st], ((k / kQStages) - 1) & 1, status)) break;
        const int h = hk * g + k / qtiles, t = tlo + k % qtiles;
        mbar_arrive_expect_tx(&qd_full[st], 2 * L::kTileBytes + (MIXED ? L::kScoreBytes : 0));
        tma_load_3d(smem + L::kQ + st * L::kTileBytes, &tm_q, &qd_full[st], 0, h, doc_start + t * kTile);
        tma_load_3d(smem + L::kDO + st * L::kTileBytes, &tm_do, &qd_full[st], 0, h, doc_start + t * kTile);
        if (MIXED)
          tma_load_3d(smem + L::kQ4 + st * L::kScoreBytes, &tm_q4, &qd_full[st], 0, h, doc_start + t * kTile);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The warp runs the loop converged (every lane waits); the elected lane issues
    // the MMAs and the commits (a commit tracks the MMAs of its own thread).
    const bool leader = elect_one();
    {
      // operand descriptors: every tile sits at a compile-time offset from the aligned
      // SMEM base, so each descriptor is one add on base16
      constexpr uint32_t kDS64 = kDQT ? kSwizzle64B : kSwizzle128B;
      constexpr uint32_t kDSR = kDQT ? 512 : 1024;       // dS^ 8-row group stride
      const uint32_t base16 = (smem_u32(smem) & 0x3FFFFu) >> 4;
      // base16 re-read at every use, so that the compiler does not hoist the ~20
      // descriptor words out of the step loop into the issuer's few registers
      auto b16 = [&]() {
        uint32_t x;
        asm volatile("mov.b32 %0, %1;" : "=r"(x) : "r"(base16));
        return x;
      };
      auto k_kmaj = [&](uint32_t o) { return sdesc_at(b16(), L::kK + o, 16, kAtom, kLayout); };        // S^T: A
      auto k_mn = [&](uint32_t o) { return sdesc_at(b16(), L::kK + o, kAtom, kAtom, kLayout); };       // dQ: B, dQ^T: A
      auto v_kmaj = [&](uint32_t o) { return sdesc_at(b16(), L::kV + o, 16, kAtom, kLayout); };        // dP^T: A
      auto q_kmaj = [&](uint32_t o) { return sdesc_at(b16(), L::kQ + o, 16, kAtom, kLayout); };        // S^T: B
      auto q_mn = [&](uint32_t o) { return sdesc_at(b16(), L::kQ + o, kAtom, kAtom, kLayout); };       // dK: B
      auto do_kmaj = [&](uint32_t o) { return sdesc_at(b16(), L::kDO + o, 16, kAtom, kLayout); };      // dP^T: B
      auto do_mn = [&](uint32_t o) { return sdesc_at(b16(), L::kDO + o, kAtom, kAtom, kLayout); };     // dV: B
      auto pt_kmaj = [&](uint32_t o) { return sdesc_at(b16(), L::kPt + o, 16, 1024, kSwizzle128B); };  // dV: A
      // dS^: dK's A (keys x queries, K-major) and dQ's operand read query-major (at d = 128
      // two 64-query SW64 tiles, the B operands of the dQ^T halves)
      auto ds_kmaj = [&](uint32_t o) { return sdesc_at(b16(), L::kDS + o, 16, kDSR, kDS64); };
      auto ds_mn = [&](uint32_t o) { return sdesc_at(b16(), L::kDS + o, kDSR, kDSR, kDS64); };
      auto issue_s = [&](int st) {
        if constexpr (MIXED) {
          // S^T = K~ Q~^T from the NVFP4 copies (64 E2M1 elements per instruction); the
          // scale words sit in dP columns 64-71 (K~) and 72-79 (Q~): the dQ^T halves do not
          // use them, and they are free once the compute warps have read dP^T
#pragma unroll
          for (int s = 0; s < 2; ++s)
            if (leader) mma_nvf4(tbase + kS, sdesc_at(b16(), L::kK4 + 32 * s, 16, 8 * 64, kSwizzle64B),
                     sdesc_at(b16(), L::kQ4 + st * L::kScoreBytes + 32 * s, 16, 8 * 64, kSwizzle64B),
                     idesc_nvf4(128, 128), tbase + kP + 64 + 4 * s, tbase + kP + 72 + 4 * s, s > 0);
        } else {
#pragma unroll
          for (int s = 0; s < D / 32; ++s)
            if (leader) mma_f8(tbase + kS, k_kmaj(32 * s), q_kmaj(st * L::kTileBytes + 32 * s), idesc_f8(128, 128, 0, 0), s > 0);
        }
      };
      auto issue_dp = [&](int st) {
#pragma unroll
        for (int s = 0; s < D / 32; ++s)
          if (leader) mma_f8(tbase + kP, v_kmaj(32 * s), do_kmaj(st * L::kTileBytes + 32 * s), idesc_f8(128, 128, 0, 0), s > 0);
      };
      // dP^T for the queries of one 64-query half qh (columns kP + 64 qh ..)
      auto issue_dp_half = [&](int st, int qh) {
#pragma unroll
        for (int s = 0; s < D / 32; ++s)
          if (leader)
            mma_f8(tbase + kP + 64 * qh, v_kmaj(32 * s), do_kmaj(st * L::kTileBytes + qh * 64 * D + 32 * s),
                   idesc_f8(128, 64, 0, 0), s > 0);
      };
      // dQ^T = K^T dS^T per 64-query half (A: K keys x d read d-major; B: the half's
      // dS^ tile, queries contiguous)
      auto issue_dqt = [&](int hf) {
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (leader) mma_mxf8(tbase + kDQ, k_mn(s * 32 * D), ds_mn(hf * 8192 + s * 32 * 64), idesc_mxf8(128, 64, 1, 1, s, s),
                   tbase + kSFQ, tbase + kSFQ + 4 + 4 * hf, s > 0);
        if (leader) mma_commit(dq_full);
      };
      bool ok = warp_wait(kv_full, 0, status) && warp_wait(&qd_full[0], 0, status);
      if (ok && MIXED) ok = warp_wait(sf_ready, 0, status);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        if (leader) mma_commit(s_full);
        issue_dp(0);
        if (leader) mma_commit(dp_full);
      }
      bool acc_committed = false;
      for (int k = 0; k < nsteps && ok; ++k) {
        const int st = k % kQStages;
        const int st1 = (k + 1) % kQStages;
        const bool more = k + 1 < nsteps;
        // dV as soon as P^ is in SMEM; then (not mixed) S of the next step, which runs
        // while the compute warpgroups build dS^
        ok = warp_wait(pt_full, k & 1, status);
        if (!ok) break;
        tc_fence_after();
        {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            // dV += P^^T dO (A: keys x queries K-major; B: dO queries x d, MN-major)
            if (leader) {
              if constexpr (kPtT)
                mma_mxf8_ta(tbase + kDV, tbase + kPtCol + 32 * s, do_mn(st * L::kTileBytes + s * 32 * D),
                            idesc_mxf8(128, D, 0, 1, s, s), tbase + kSFV, tbase + kSFV + 4, (k > 0 || s > 0));
              else
                mma_mxf8(tbase + kDV, pt_kmaj(32 * s), do_mn(st * L::kTileBytes + s * 32 * D), idesc_mxf8(128, D, 0, 1, s, s),
                         tbase + kSFV, tbase + kSFV + 4, (k > 0 || s > 0));
            }
        }
        if (more) {
          // mixed route: the next step's score scale words are written by the readout
          // warpgroups once this step's dP^T has been read (the compute warps' hand-in)
          ok = (!MIXED || warp_wait(sf_ready, (k + 1) & 1, status)) &&
               warp_wait(&qd_full[st1], ((k + 1) / kQStages) & 1, status);
          if (!ok) break;
          tc_fence_after();
          issue_s(st1);
          if (leader) mma_commit(s_full);
        }
        ok = warp_wait(p_full, k & 1, status);
        if (!ok) break;
        tc_fence_after();
        // the low dQ^T half goes first so that its readout overlaps dK; the high half
        // follows once the readout released the columns
        if (kDQT) issue_dqt(0);
        {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            // dK += dS^^T Q (A: dS^ keys x queries K-major)
            if (leader) mma_mxf8(tbase + kDK, ds_kmaj(kDQT ? (s >> 1) * 8192 + 32 * (s & 1) : 32 * s), q_mn(st * L::kTileBytes + s * 32 * D),
                     idesc_mxf8(128, D, 0, 1, s, s), tbase + kSFK, tbase + kSFK + 4, (k > 0 || s > 0));
        }
        if (leader) mma_commit(&qd_empty[st]);             // Q and dO of this step are no longer read
        // last step: dK and dV are complete once the MMAs so far are, so the compute
        // warpgroups' epilogue starts while the last dQ partial is computed and read
        if (!more) {
          if (leader) mma_commit(acc_full);
          acc_committed = true;
        }
        if (kDQT) {
          ok = warp_wait(dq_empty, 0, status);
          if (!ok) break;
          tc_fence_after();
          issue_dqt(1);
          // the next step's dP^T for queries 64..127 goes into the columns the dQ^T halves
          // do not use (the scale words there were read by the dK and dQ^T MMAs issued
          // before it), so only the other half waits for the readout of the high half
          if (!MIXED && more) issue_dp_half(st1, 1);
        } else if (!STRICT) {
          if (k > 0) {                         // the previous partial has been read
            ok = warp_wait(dq_empty, (k - 1) & 1, status);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int s = 0; s < 4; ++s)
            // dQ partial = dS^ K (A: the dS^ tile read query-major; B: K keys x d, MN-major)
            if (leader) mma_mxf8(tbase + kDQ, ds_mn(s * 32 * 128), k_mn(s * 32 * D), idesc_mxf8(128, D, 1, 1, s, s),
                     tbase + kSFQ, tbase + kSFQ + 4, s > 0);
          if (leader) mma_commit(dq_full);
        }
        if (more) {
          if (kDQT) {                          // dP of the next step goes where the dQ^T halves were
            ok = warp_wait(dq_empty, 1, status);
            if (!ok) break;
            tc_fence_after();
          }
          if (kDQT && !MIXED) issue_dp_half(st1, 0);
          else issue_dp(st1);
          if (leader) mma_commit(dp_full);
        }
      }
      if (!ok && leader) {
        // a wait ran out: commit (unless the last step did) and wait, so that nothing
        // of ours still reads SMEM or TMEM
        if (!acc_committed) mma_commit(acc_full);
        mbar_wait(acc_full, 0, status);
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ per-query row data
    // Every global load of a step is issued into registers before the wait for the
    // buffer and before any shared-memory store, so the latencies overlap each other
    // and the wait instead of queueing behind stores the compiler cannot reorder.
    for (int k = 0; k < nsteps; ++k) {
      const int b = k & 1;
      const int h = hk * g + k / qtiles, t = tlo + k % qtiles;
      float lv[4], dv[4], sqv[4], sdv[4];
      uint8_t scb = 127;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ql = t * kTile + q * 32 + lane;
        const bool qv = ql < doc_len;
        const int64_t qtok = (int64_t)doc_start + ql;
        lv[q] = qv ? __ldg(p.lse + (int64_t)h * p.T + qtok) : 0.f;
        dv[q] = qv ? __ldg(p.dvec + (int64_t)h * p.T + qtok) : 0.f;
        if (STRICT) {
          sqv[q] = qv ? ue8m0_to_f32(__ldg(p.q_scales + qtok * p.hq + h)) : 1.0f;
          sdv[q] = qv ? ue8m0_to_f32(__ldg(p.do_scales + qtok * p.hq + h)) : 1.0f;
        }
      }
      if (lane < 8) {
        const int ql = t * kTile + (lane & 3) * 32;
        const uint8_t* src = lane < 4 ? p.q_scales : p.do_scales;
        if (ql < doc_len) scb = __ldg(src + ((int64_t)doc_start + ql) * p.hq + h);
      }
      if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(&row_empty[b], ((k >> 1) - 1) & 1, status))) break;
      float* rb = rowbuf + b * (L::kRowBuf / 4);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = q * 32 + lane;
        const bool qv = t * kTile + i < doc_len;
        // the P boost 2^8 rides in the exponent; dP - D is scaled by 2^-8 to compensate
        rb[i] = qv ? fmaf(-lv[q], 1.4426950408889634f, 8.0f) : -INFINITY;
        rb[128 + i] = qv ? -dv[q] * (1.0f / 256.0f) : 0.f;
        if (STRICT) {
          rb[260 + i] = sqv[q];
          rb[388 + i] = sdv[q];
        }
      }
      if (lane < 8) reinterpret_cast<uint8_t*>(rb + 256)[lane] = scb;
      mbar_arrive(&row_full[b]);
    }
  }
  } else if (compute_wg) {
    // ------------------------------------------------------------ compute (warps 4 .. 4 + 4 kWG - 1)
    setmaxnreg_inc<Shape::kRegHigh>();
    const int wg = (warp - 4) >> 2;                    // query columns [32 kCPW wg, 32 kCPW (wg + 1))
    const int quarter = warp & 3;
    const int j = quarter * 32 + lane;                 // key row (TMEM lane) for S / dP; query row for dQ
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const bool key_valid = u * kTile + j < doc_len;
    const int64_t ktok = (int64_t)doc_start + u * kTile + j;
    const float sk_row = key_valid ? ue8m0_to_f32(p.k_scales[ktok * p.hkv + hk]) : 1.0f;
    const float sv_row = key_valid ? ue8m0_to_f32(p.v_scales[ktok * p.hkv + hk]) : 1.0f;
    uint32_t ksf = 0;   // K block scales per 32-key group (dQ MMA, B operand)
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) {
      const int kl = u * kTile + gg * 32;
      const uint32_t b = kl < doc_len ? p.k_scales[((int64_t)doc_start + kl) * p.hkv + hk] : 127u;
      ksf |= b << (8 * gg);
    }
    uint8_t* Esm = smem + L::kE;
    uint8_t* sPt = smem + L::kPt;
    uint8_t* sDS = smem + L::kDS;
    // diagnostic build: row j's 32 values of query chunk c (slice 0 = P, 1 = dS)
    auto dbg_store = [&](int which, int kstep, int c, const float* vals, float mul) {
      const int h = hk * g + kstep / qtiles, tq = tlo + kstep % qtiles;
      if (!key_valid) return;
#pragma unroll 1
      for (int i = 0; i < 32; ++i) {
        const int ql = tq * kTile + 32 * c + i;
        if (ql < doc_len) p.dbg[(((int64_t)which * p.hq + h) * p.T + doc_start + ql) * p.T + ktok] = vals[i] * mul;
      }
    };
    bool ok = true;
    for (int k = 0; k < nsteps; ++k) {
      const int t = tlo + k % qtiles;
      // tiles with a hidden pair (causal: the diagonal one) or keys past the document end
      // take the masked variant of the weight loop
      const bool diag = WIN ? win_masked(t, u, doc_len, p.win) : t == u;
      const int b = k & 1;
      const float* rb = rowbuf + b * (L::kRowBuf / 4);
      const uint8_t* cs = reinterpret_cast<const uint8_t*>(rb + 256);
      // default and mixed routes: per warp, since no warpgroup needs another's data before
      // the barrier that closes dS^ (the block exponents of the last step were all read
      // before every compute thread handed in that step, which the dP^T this step waits
      // for follows); the strict options keep the warpgroups in step here, which measured
      // faster for their per-key folds
      if constexpr (STRICT)
        ok = named_bar_and(1, kCompute, mbar_wait(&row_full[b], (k >> 1) & 1, status) && mbar_wait(s_full, k & 1, status));
      else
        ok = __all_sync(0xffffffffu, mbar_wait(&row_full[b], (k >> 1) & 1, status) && mbar_wait(s_full, k & 1, status));
      if (!ok) {
        // a warp whose wait ran out still meets the barrier that closes dS^ (with a false
        // vote), so that the other compute warps learn of it there and none is left waiting
        if constexpr (!STRICT) named_bar_and(1, kCompute, false);
        break;
      }
      tc_fence_after();
      // 2^8 P = 2^(x - LSE log2 e + 8) for this warpgroup's query chunks
      float pr[kCPW][32];
#pragma unroll
      for (int cc = 0; cc < kCPW; ++cc) {
        const int c = kCPW * wg + cc;
        uint32_t vs[32];
        tmem_ld32(lane_base + kS + 32 * c, vs);
        tmem_ld_wait();
        if (!STRICT && wg == 0 && cc == 0) {
          // scale words of dV += P^^T dO into columns this warpgroup has just read: A = P^
          // (1.0), B = dO per query chunk
          const uint32_t bw = (uint32_t)cs[4] | (uint32_t)cs[5] << 8 | (uint32_t)cs[6] << 16 | (uint32_t)cs[7] << 24;
          tmem_st4(lane_base + kSFV + 0, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          tmem_st4(lane_base + kSFV + 4, bw, bw, bw, bw);
        }
        const float fS = MIXED ? p.scale_log2 : p.scale_log2 * sk_row * (STRICT ? 1.0f : ue8m0_to_f32(cs[c]));
        const float2 fS2 = make_float2(fS, fS);
        const float4* nl4 = reinterpret_cast<const float4*>(rb + 32 * c);   // -LSE * log2(e)
        const float4* sq4 = reinterpret_cast<const float4*>(rb + 260 + 32 * c);   // strict: s_Q per query
        uint32_t pk[8];
        // the causal mask only on the diagonal tile: the loop is built twice
        auto p_math = [&](auto diag_tile) {
          constexpr bool kDiag = decltype(diag_tile)::value;
          // windowed calls, masked variant: this key row is seen by the tile's queries
          // [qlim, qhim] (causal calls: the queries at or after the key)
          int qlim = 0, qhim = 0;
          if constexpr (kDiag && WIN) {
            const int kj = u * kTile + j;
            qlim = !key_valid ? kTile : (p.win.right < 0 ? 0 : kj - p.win.right - t * kTile);
            qhim = !key_valid ? -1 : (p.win.left < 0 ? kTile : kj + p.win.left - t * kTile);
          }
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 nl = nl4[i >> 2];
          float2 d0 = make_float2(__uint_as_float(vs[i]), __uint_as_float(vs[i + 1]));
          float2 d1 = make_float2(__uint_as_float(vs[i + 2]), __uint_as_float(vs[i + 3]));
          if (STRICT) {
            const float4 sq = sq4[i >> 2];
            d0 = fmul2(d0, make_float2(sq.x, sq.y));
            d1 = fmul2(d1, make_float2(sq.z, sq.w));
          }
          float2 x0 = ffma2(d0, fS2, make_float2(nl.x, nl.y));
          float2 x1 = ffma2(d1, fS2, make_float2(nl.z, nl.w));
          float2 p0 = make_float2(fast_exp2(x0.x), fast_exp2(x0.y));
          float2 p1 = make_float2(fast_exp2(x1.x), fast_exp2(x1.y));
          if (kDiag) {
            const int il = 32 * c + i;
            if constexpr (WIN) {
              p0.x = (il >= qlim && il <= qhim) ? p0.x : 0.f;
              p0.y = (il + 1 >= qlim && il + 1 <= qhim) ? p0.y : 0.f;
              p1.x = (il + 2 >= qlim && il + 2 <= qhim) ? p1.x : 0.f;
              p1.y = (il + 3 >= qlim && il + 3 <= qhim) ? p1.y : 0.f;
            } else {
              p0.x = il >= j ? p0.x : 0.f;
              p0.y = il + 1 >= j ? p0.y : 0.f;
              p1.x = il + 2 >= j ? p1.x : 0.f;
              p1.y = il + 3 >= j ? p1.y : 0.f;
            }
          }
          pr[cc][i] = p0.x; pr[cc][i + 1] = p0.y; pr[cc][i + 2] = p1.x; pr[cc][i + 3] = p1.y;
          if (!STRICT) pk[i >> 2] = (uint32_t)e4m3x2(p0.x, p0.y) | ((uint32_t)e4m3x2(p1.x, p1.y) << 16);
        }
        };
        if (diag) p_math(std::true_type{});
        else p_math(std::false_type{});
        if constexpr (DBG) dbg_store(0, k, c, pr[cc], 1.0f / 256.0f);
        if (STRICT) {
          // dV operand with dO's per-token scale folded in: 2^8 P s_dO(i), one round-up
          // exponent per (key row, 32-query chunk)
          const float4* sd4 = reinterpret_cast<const float4*>(rb + 388 + 32 * c);
          float pf[32];
          float gmax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 sd = sd4[i >> 2];
            const float2 a0 = fmul2(make_float2(pr[cc][i], pr[cc][i + 1]), make_float2(sd.x, sd.y));
            const float2 a1 = fmul2(make_float2(pr[cc][i + 2], pr[cc][i + 3]), make_float2(sd.z, sd.w));
            pf[i] = a0.x; pf[i + 1] = a0.y; pf[i + 2] = a1.x; pf[i + 3] = a1.y;
            gmax = fmax3(gmax, fmaxf(a0.x, a0.y), fmaxf(a1.x, a1.y));
          }
          const int ev = roundup_exp(gmax);
          const float sc = exp2i(-ev);
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            pk[i >> 2] = (uint32_t)e4m3x2(pf[i] * sc, pf[i + 1] * sc) | ((uint32_t)e4m3x2(pf[i + 2] * sc, pf[i + 3] * sc) << 16);
          Esm[64 + j * 4 + c] = (uint8_t)(ev + 127);
        }
        if constexpr (kPtT) {
          tmem_st8(lane_base + kPtCol + 32 * c, pk);    // key row j of chunk c: 32 codes, query order
        } else {
          *reinterpret_cast<uint4*>(sPt + swz_offset(j, 32 * c, 128)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(sPt + swz_offset(j, 32 * c + 16, 128)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if constexpr (!kPtT) fence_proxy_async_smem();   // P^ and its row exponents, published below
      if constexpr (STRICT) {
        ok = named_bar_and(1, kCompute, mbar_wait(dp_full, k & 1, status));
        if (!ok) break;
        tc_fence_after();
        if (wg == 0) {
          // scale words of dV += P^^T dO (S^T has been read by every warpgroup): A = P^'s
          // per-key-row exponents, B = 1.0 (dO's per-token scales are folded into P^)
          tmem_st1(lane_base + kSFV + quarter, *reinterpret_cast<const uint32_t*>(Esm + 64 + j * 4));
          tmem_st4(lane_base + kSFV + 4, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(pt_full);
        }
      } else {
        // every compute thread hands in its part of P^ (warpgroup 0 also the scale words)
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(pt_full);
        ok = __all_sync(0xffffffffu, mbar_wait(dp_full, k & 1, status));
        if (!ok) {
          named_bar_and(1, kCompute, false);   // meets the barrier that closes dS^ (false vote)
          break;
        }
        tc_fence_after();
      }
#pragma unroll
      for (int cc = 0; cc < kCPW; ++cc) {
        const int c = kCPW * wg + cc;
        uint32_t vp[32];
        tmem_ld32(lane_base + kP + 32 * c, vp);
        tmem_ld_wait();
        if (kDQT && wg == kWG - 1) {
          // the scale words that do not depend on this step's dS^ exponents, into dP columns
          // this warpgroup has just read: dK's B (Q per query chunk), dQ^T's A (K's blocks)
          const uint32_t bq = *reinterpret_cast<const uint32_t*>(cs);
          tmem_st4(lane_base + kSFK + 4, bq, bq, bq, bq);
          tmem_st4(lane_base + kSFQ, ksf, ksf, ksf, ksf);
        }
        const float fP = (1.0f / 256.0f) * sv_row * (STRICT ? 1.0f : ue8m0_to_f32(cs[4 + c]));
        const float2 fP2 = make_float2(fP, fP);
        const float4* nd4 = reinterpret_cast<const float4*>(rb + 128 + 32 * c);   // -D
        const float4* sd4 = reinterpret_cast<const float4*>(rb + 388 + 32 * c);   // strict: s_dO
        const float4* sq4 = reinterpret_cast<const float4*>(rb + 260 + 32 * c);   // strict: s_Q
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 nd = nd4[i >> 2];
          float2 v0 = make_float2(__uint_as_float(vp[i]), __uint_as_float(vp[i + 1]));
          float2 v1 = make_float2(__uint_as_float(vp[i + 2]), __uint_as_float(vp[i + 3]));
          if (STRICT) {
            const float4 sd = sd4[i >> 2];
            v0 = fmul2(v0, make_float2(sd.x, sd.y));
            v1 = fmul2(v1, make_float2(sd.z, sd.w));
          }
          const float2 t0 = ffma2(v0, fP2, make_float2(nd.x, nd.y));
          const float2 t1 = ffma2(v1, fP2, make_float2(nd.z, nd.w));
          float2 d0 = fmul2(make_float2(pr[cc][i], pr[cc][i + 1]), t0);
          float2 d1 = fmul2(make_float2(pr[cc][i + 2], pr[cc][i + 3]), t1);
          if (STRICT) {     // dK operand: Q's per-token scale folded into dS
            const float4 sq = sq4[i >> 2];
            d0 = fmul2(d0, make_float2(sq.x, sq.y));
            d1 = fmul2(d1, make_float2(sq.z, sq.w));
          }
          pr[cc][i] = d0.x; pr[cc][i + 1] = d0.y; pr[cc][i + 2] = d1.x; pr[cc][i + 3] = d1.y;
          amax = fmax3(amax, fabsf(d0.x), fabsf(d0.y));
          amax = fmax3(amax, fabsf(d1.x), fabsf(d1.y));
        }
        if constexpr (DBG) dbg_store(1, k, c, pr[cc], 1.0f);
        // 32 x 32 block: the warp's 32 key rows (non-negative floats order like their bit
        // patterns, so one warp-wide integer maximum)
        if (!STRICT) amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
        const int e = roundup_exp(amax);
        const float sc = exp2i(-e);
        const float2 sc2 = make_float2(sc, sc);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float2 q0 = fmul2(make_float2(pr[cc][i], pr[cc][i + 1]), sc2);
          const float2 q1 = fmul2(make_float2(pr[cc][i + 2], pr[cc][i + 3]), sc2);
          pk[i >> 2] = (uint32_t)e4m3x2(q0.x, q0.y) | ((uint32_t)e4m3x2(q1.x, q1.y) << 16);
        }
        // d = 128 (not strict): two 64-query SW64 tiles, the B operands of the dQ^T halves
        uint8_t* dsrow = kDQT ? sDS + (c >> 1) * 8192 + swz_offset(j, 32 * (c & 1), 64) : sDS + swz_offset(j, 32 * c, 128);
        uint8_t* dsrow2 = kDQT ? sDS + (c >> 1) * 8192 + swz_offset(j, 32 * (c & 1) + 16, 64)
                               : sDS + swz_offset(j, 32 * c + 16, 128);
        *reinterpret_cast<uint4*>(dsrow) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(dsrow2) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        if (STRICT) Esm[576 + j * 4 + c] = (uint8_t)(e + 127);
        else if (lane == 0) Esm[quarter * 4 + c] = (uint8_t)(e + 127);
      }
      fence_proxy_async_smem();              // this thread's dS^ codes, for the MMAs
      // all block exponents written; S^T and dP^T fully read (default and mixed routes: a
      // vote, since a warp whose wait ran out meets this barrier with false)
      if constexpr (STRICT) {
        named_bar_sync(1, kCompute);
      } else {
        ok = named_bar_and(1, kCompute, true);
        if (!ok) break;
      }
      if (STRICT) {
        // A-operand scales are per key row: row j's word sits in lane j, column
        // (base + j / 32), i.e. this warp's quarter; B operands (dO, Q) are folded.
        if (wg == 1 % kWG) {      // dK: A per key row, B (Q) folded
          tmem_st1(lane_base + kSFK + quarter, *reinterpret_cast<const uint32_t*>(Esm + 576 + j * 4));
          tmem_st4(lane_base + kSFK + 4, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&row_empty[b]);
        mbar_arrive(p_full);
        continue;                            // dQ comes from the deterministic dQ kernel
      }
      if constexpr (kDQT) {
        // the exponent-dependent words of dK and dQ^T, one group per warpgroup: E holds
        // one byte per (key block, query chunk), word b = key block b's four chunks
        const uint4 e4 = *reinterpret_cast<const uint4*>(Esm);
        if (wg == 1) {                        // dK: A row = key in block b, byte = query chunk
          tmem_st4(lane_base + kSFK, e4.x, e4.y, e4.z, e4.w);
        } else if (wg != 3) {
          // dQ^T: B row = query, one word per query chunk c holding its four key blocks'
          // bytes (the 4 x 4 byte transpose of E); warpgroup 2 the low half, 0 the high
          const uint32_t lo = __byte_perm(e4.x, e4.y, wg == 2 ? 0x5140 : 0x7362);
          const uint32_t hi = __byte_perm(e4.z, e4.w, wg == 2 ? 0x5140 : 0x7362);
          const uint32_t c0 = __byte_perm(lo, hi, 0x5410), c1 = __byte_perm(lo, hi, 0x7632);
          tmem_st4(lane_base + kSFQ + (wg == 2 ? 4 : 8), c0, c1, c0, c1);
        }
        tmem_st_wait();
      } else {
        // block-scale words of the dK and dQ MMAs (dV's were written after P^), one
        // operand pair per warpgroup
        const uint8_t* E = Esm;               // E[key block][query chunk]
        const int pair0 = wg, pair1 = wg + kWG;   // pairs 0 = dV, 1 = dK, 2 = dQ
#pragma unroll
        for (int pi = 0; pi < 2; ++pi) {
          const int pair = pi == 0 ? pair0 : pair1;
          if (pair == 0 || pair > 2) continue;
          uint32_t a[4], bw;
          if (pair == 1) {          // dK: A row = key in block cc, byte = query chunk; B = Q per query chunk
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              a[cc] = (uint32_t)E[cc * 4 + 0] | (uint32_t)E[cc * 4 + 1] << 8 | (uint32_t)E[cc * 4 + 2] << 16 |
                      (uint32_t)E[cc * 4 + 3] << 24;
            bw = (uint32_t)cs[0] | (uint32_t)cs[1] << 8 | (uint32_t)cs[2] << 16 | (uint32_t)cs[3] << 24;
          } else {                  // dQ: A row = query in chunk cc, byte = key block; B = K per key block
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              a[cc] = (uint32_t)E[0 * 4 + cc] | (uint32_t)E[1 * 4 + cc] << 8 | (uint32_t)E[2 * 4 + cc] << 16 |
                      (uint32_t)E[3 * 4 + cc] << 24;
            bw = ksf;
          }
          if (pair == 1) {
            tmem_st4(lane_base + kSFK, a[0], a[1], a[2], a[3]);
            tmem_st4(lane_base + kSFK + 4, bw, bw, bw, bw);
          } else if (kDQT) {
            // dQ^T: A = K^T (every d row: K's block scales), B = the half's dS^T rows
            // (query n of half hf: the word of query chunk 2 hf + n / 32)
            tmem_st4(lane_base + kSFQ, bw, bw, bw, bw);
            tmem_st4(lane_base + kSFQ + 4, a[0], a[1], a[0], a[1]);
            tmem_st4(lane_base + kSFQ + 8, a[2], a[3], a[2], a[3]);
          } else {
            tmem_st4(lane_base + kSFQ, a[0], a[1], a[2], a[3]);
            tmem_st4(lane_base + kSFQ + 4, bw, bw, bw, bw);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&row_empty[b]);
      mbar_arrive(p_full);
    }
    if (ok) ok = named_bar_and(1, kCompute, mbar_wait(acc_full, 0, status));
    if (ok) {
      tc_fence_after();
      // dV and dK tiles: each thread stages its row's slice as bf16 in the (now idle) Q
      // and dO buffers, as 64-column boxes of 128 rows x 128 bytes (16-byte unit c of
      // row j at position c XOR (j mod 8), the 128-byte swizzle); a full tile leaves by
      // TMA stores of those boxes, the last, partial tile of a document by coalesced
      // row stores of its rows (a box would write into the next document)
      constexpr int kRowB = D * 2, kUnits = kRowB / 16;
      static_assert(kQStages * L::kTileBytes == kTile * kRowB, "a stage pair holds one bf16 tile");
      auto stg_off = [](int r, int unit) { return (unit >> 3) * (kTile * 128) + r * 128 + (((unit & 7) ^ (r & 7)) << 4); };
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = (which == 0 ? kDV : kDK) + wg * kCols;
        float mul = which == 0 ? (1.0f / 256.0f) : p.scale;
        uint8_t* stg = smem + (which == 0 ? L::kQ : L::kDO);
        uint32_t v[32];
        if (ROT && which == 1) {
          // rotated operands: this warpgroup's 32 columns of dK_rot H / 2^k.  H = H_kWG x
          // H_32: combine the row's kWG slices with the signs of H_kWG's row wg, then
          // the 32-point butterflies (strides 1 .. 16) in registers.
          float acc[32];
#pragma unroll 1
          for (int s2 = 0; s2 < kWG; ++s2) {
            tmem_ld32(lane_base + kDK + s2 * kCols, v);
            tmem_ld_wait();
            const float sg = (__popc(wg & s2) & 1) ? -1.0f : 1.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = s2 == 0 ? sg * __uint_as_float(v[i]) : fmaf(sg, __uint_as_float(v[i]), acc[i]);
          }
#pragma unroll
          for (int st = 1; st < 32; st <<= 1)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (!(i & st)) {
                const float a = acc[i], b = acc[i + st];
                acc[i] = a + b;
                acc[i + st] = a - b;
              }
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(acc[i]);
          mul *= D == 128 ? 0.0625f : 0.125f;   // 2^-k
        } else {
          tmem_ld32(lane_base + col, v);
          tmem_ld_wait();
        }
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * q]) * mul, __uint_as_float(v[2 * q + 1]) * mul);
          pk[q] = *reinterpret_cast<uint32_t*>(&b2);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int unit = (wg * kCols * 2) / 16 + q;
          *reinterpret_cast<uint4*>(stg + stg_off(j, unit)) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();              // the staged tiles, for the TMA stores
      named_bar_sync(1, kCompute);
      const int rows = min(kTile, doc_len - u * kTile);
      const int64_t row0 = (int64_t)doc_start + u * kTile;
      if (rows == kTile) {
        if (threadIdx.x == 128) {
#pragma unroll
          for (int hb = 0; hb < D / 64; ++hb) {
            tma_store_3d(&tm_dv, smem + L::kQ + hb * (kTile * 128), 64 * hb, hk, (int)row0);
            tma_store_3d(&tm_dk, smem + L::kDO + hb * (kTile * 128), 64 * hb, hk, (int)row0);
          }
          bulk_commit();
          bulk_wait_read<0>();               // the buffers stay valid until the stores have read them
        }
      } else {
        for (int idx = threadIdx.x - 128; idx < 2 * rows * kUnits; idx += kCompute) {
          const int which = idx >= rows * kUnits;
          const int rem = idx - which * rows * kUnits;
          const int r = rem / kUnits, unit = rem % kUnits;
          const uint4 val = *reinterpret_cast<const uint4*>(smem + (which == 0 ? L::kQ : L::kDO) + stg_off(r, unit));
          __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + ((row0 + r) * p.hkv + hk) * D + unit * 8;
          *reinterpret_cast<uint4*>(dst) = val;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ readout (the last warpgroup)
    if constexpr (Shape::kRegRead < Shape::kLaunchRegs) setmaxnreg_dec<Shape::kRegRead>();
    else setmaxnreg_inc<Shape::kRegRead>();
    const int ro = (warp - 4 - 4 * kWG) >> 2;         // readout warpgroup
    // Per step: wait for the dQ partial, read it slice by slice (32 head-dim columns,
    // thread = query row), release the TMEM columns, stage c * partial as fp16 in the
    // slice's swizzled SMEM buffer and reduce each slice into its accumulator chunk
    // with one bulk fp16 reduce-add (rows past the document end are staged as zeros).
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;                 // query row of the dQ partial (TMEM lane)
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    const bool elected = ro == 0 && (threadIdx.x & 127) == 0;
    // mixed route: scale words of the score MMA, written into dP columns before every
    // score MMA, replicated over the four lane quarters (lane 32q + l, column c holds
    // row 32c + l); per row and instruction one word of four E4M3 scales.  Readout
    // warpgroup 0 holds the K~ rows' words (A, fixed, columns 64-71), warpgroup 1 the
    // Q~ rows' words of the next step's query tile (B, columns 72-79).  They are
    // written once the compute warps have handed in the step (its dP^T read), so the
    // next score MMA goes out before this step's dQ^T.
    uint2 sfw[4] = {};
    auto load_sf_rows = [&](const uint8_t* base, int64_t tok0, int H, int hh_) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t tok = tok0 + 32 * c + lane;
        sfw[c] = tok < p.T ? *reinterpret_cast<const uint2*>(base + (tok * H + hh_) * (D / 16)) : make_uint2(0u, 0u);
      }
    };
    auto step_qsf = [&](int kk) {       // warpgroup 1: the Q~ rows of step kk
      load_sf_rows(p.q4_scales, (int64_t)doc_start + (tlo + kk % qtiles) * kTile, p.hq, hk * g + kk / qtiles);
    };
    auto store_score_sf = [&]() {
      tmem_st4(lane_base + kP + 64 + 8 * ro, sfw[0].x, sfw[1].x, sfw[2].x, sfw[3].x);
      tmem_st4(lane_base + kP + 64 + 8 * ro + 4, sfw[0].y, sfw[1].y, sfw[2].y, sfw[3].y);
    };
    if (MIXED) {
      if (ro == 0) load_sf_rows(p.k4_scales, (int64_t)doc_start + u * kTile, p.hkv, hk);
      else step_qsf(0);
      store_score_sf();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(sf_ready);
      if (ro == 1 && nsteps > 1) step_qsf(1);
    }
    constexpr int kRowBytes = kCols * 2;               // 64: one staged row of fp16
    constexpr int kChunks = kRowBytes / 16;            // 16-byte units per staged row
    bool ok = true;
    for (int k = 0; k < nsteps && !STRICT; ++k) {
      const int hh = k / qtiles, t = tlo + k % qtiles;
      const int h = hk * g + hh;
      const float cb = p.boost[(int64_t)doc * p.hq + h];
      const int qvalid = doc_len - t * kTile;          // query rows of the tile inside the document
      if (MIXED && k + 1 < nsteps) {
        // the next step's score scale words, once this step's dP^T has been read
        ok = named_bar_and(6, 128 * kRO, mbar_wait(p_full, k & 1, status));
        if (!ok) break;
        tc_fence_after();
        store_score_sf();                      // warpgroup 1: the Q~ rows of step k + 1
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(sf_ready);
      }
      if constexpr (kDQT) {
        // dQ^T: thread = head-dim row d = i; per 64-query half this warpgroup reads its
        // 32 query columns and packs them into four 16-byte units of the staged chunk
        // (queries past the document end as 0)
        uint8_t* srow = smem + L::kStage + (k & 1) * (2 * 16384) + i * 128;
        const uint32_t sw = (uint32_t)(i & 7);
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          ok = named_bar_and(6, 128 * kRO, mbar_wait(dq_full, hf, status));
          if (!ok) break;
          tc_fence_after();
          uint32_t v[32];
          tmem_ld32(lane_base + kDQ + 32 * ro, v);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(dq_empty);             // the columns are in registers
          const int nq = qvalid - hf * 64 - 32 * ro;   // valid queries among the 32
          const float2 cb2 = make_float2(cb, cb);
          auto stage = [&](auto tail) {                  // built twice: the mask only at a document end
            constexpr bool kTail = decltype(tail)::value;
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int q = 8 * uu + 2 * e;
                float2 f = fmul2(make_float2(__uint_as_float(v[q]), __uint_as_float(v[q + 1])), cb2);
                if (kTail) {
                  f.x = q < nq ? f.x : 0.f;
                  f.y = q + 1 < nq ? f.y : 0.f;
                }
                __half2 h2 = __floats2half2_rn(f.x, f.y);
                w[e] = *reinterpret_cast<uint32_t*>(&h2);
              }
              const uint32_t unit = (uint32_t)(4 * ro + uu);
              *reinterpret_cast<uint4*>(srow + hf * 16384 + ((unit ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          };
          if (nq < 32) stage(std::true_type{});
          else stage(std::false_type{});
        }
        if (!ok) break;
      } else {
        const bool qv = i < qvalid;
        const float2 cb2 = make_float2(qv ? cb : 0.f, qv ? cb : 0.f);
        ok = named_bar_and(6, 128, mbar_wait(dq_full, k & 1, status));
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kWG; ++c) {
          uint32_t v[32];
          tmem_ld32(lane_base + kDQ + 32 * c, v);
          tmem_ld_wait();
          if (c == kWG - 1) {                // the whole partial is in registers or SMEM
            tc_fence_before();
            mbar_arrive(dq_empty);
          }
          uint8_t* sbk = smem + L::kStage + (2 * c + (k & 1)) * L::kStageBytes;
#pragma unroll
          for (int c16 = 0; c16 < kChunks; ++c16) {
            uint32_t hw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = fmul2(make_float2(__uint_as_float(v[8 * c16 + 2 * q]), __uint_as_float(v[8 * c16 + 2 * q + 1])), cb2);
              __half2 h2 = __floats2half2_rn(f.x, f.y);
              hw[q] = *reinterpret_cast<uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(sbk + dq_chunk_byte(i, 16 * c16)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          }
        }
      }
      if (MIXED && ro == 1 && k + 2 < nsteps) step_qsf(k + 2);
      fence_proxy_async_smem();
      named_bar_sync(6, 128 * kRO);
      if (elected) {
        // bulk fp16 reduce-adds of the staged tile (d = 128: one 32 KB chunk; d = 64: one
        // per slice); the wait leaves at most this step's copies reading shared memory,
        // so the other buffer is free next step
        const int64_t tile = pv.tile_prefix[doc] + t;
        if constexpr (kDQT) {
          bulk_reduce_add_f16(p.dq_acc + dqt_chunk_elems(tile, h, p.hq),
                              smem_u32(smem + L::kStage + (k & 1) * (2 * 16384)), 2 * 16384);
        } else {
          for (int c = 0; c < kWG; ++c)
            bulk_reduce_add_f16(p.dq_acc + dq_chunk_elems(tile, h, c, p.hq, D),
                                smem_u32(smem + L::kStage + (2 * c + (k & 1)) * L::kStageBytes), L::kStageBytes);
        }
        bulk_commit();
        bulk_wait_read<1>();
      }
    }
    // shared memory stays valid until the copies have read it; their global adds
    // complete before the kernel does (the finalize kernel runs after it)
    if (elected) bulk_wait_read<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// dQ boost of (document, query head) from the maxima the backward prep folded in
// (review section 4, "Forward locality and backward locality differ"; reading
// C-10): c = 2^floor(log2(2^headroom / M)), M = 2 max ||dO^_i|| max ||V^_j|| max |K^_jd|.
__global__ void boost_from_max_kernel(const float* maxima, const int* plan, int N, int hq, int headroom,
                                      float* boost) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N * hq || (plan[kPlanStatus] & FLAMIA_DEV_BAD_CU_SEQLENS)) return;
  boost[i] = dq_boost_from_maxima(maxima[3 * i], maxima[3 * i + 1], maxima[3 * i + 2], headroom);
}

// dQ = bf16(scale * acc / c), read from the accumulator chunks one (document
// tile, query head) at a time; then the rows outside every document of dQ, dK
// and dV are zeroed.
template <int D, bool ROT = false>
__global__ void __launch_bounds__(256) dq_finalize_kernel(const __half* acc, const int32_t* cu, const int* plan,
                                                          const float* boost, int N, int T, int hq, int hkv,
                                                          float scale, __nv_bfloat16* dq, __nv_bfloat16* dk,
                                                          __nv_bfloat16* dv) {
  const bool bad = plan[kPlanStatus] & FLAMIA_DEV_BAD_CU_SEQLENS;
  const int valid = bad ? 0 : plan[kPlanValid];
  const int ntiles = bad ? 0 : plan[kPlanTiles];
  const PlanView pv = plan_view(plan, T, N);
  constexpr int kVec = 8, kVpr = D / kVec;             // 16-byte vectors per row
  const int64_t units = (int64_t)ntiles * hq;
  for (int64_t un = blockIdx.x; un < units; un += gridDim.x) {
    const int tile = (int)(un / hq), h = (int)(un % hq);
    const int doc = upper_doc(pv.tile_prefix, N, tile);
    const int t = tile - pv.tile_prefix[doc];
    const int s0 = cu[doc];
    const int rows = min(kTile, cu[doc + 1] - s0 - t * kTile);
    const float mul = scale / boost[(int64_t)doc * hq + h];
    if constexpr (ROT) {
      // rotated operands: thread = query row, the row's D values through the D-point
      // butterflies (strides 1 .. D / 2), times 2^-k
      for (int r = threadIdx.x; r < rows; r += blockDim.x) {
        float z[D];
#pragma unroll
        for (int c = 0; c < D; c += kVec) {
          const __half* chunk = acc + dq_chunk_elems(tile, h, c / 32, hq, D);
          const uint4 in = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(chunk) +
                                                           dq_chunk_byte(r, (c % 32) * 2));
          const __half2* hv = reinterpret_cast<const __half2*>(&in);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(hv[q]);
            z[c + 2 * q] = f.x;
            z[c + 2 * q + 1] = f.y;
          }
        }
#pragma unroll
        for (int st = 1; st < D; st <<= 1)
#pragma unroll
          for (int i = 0; i < D; ++i)
            if (!(i & st)) {
              const float a = z[i], b = z[i + st];
              z[i] = a + b;
              z[i + st] = a - b;
            }
        const float m2 = mul * (D == 128 ? 0.0625f : 0.125f);
#pragma unroll
        for (int c = 0; c < D; c += kVec) {
          uint4 out;
          uint32_t* ov = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(z[c + 2 * q] * m2, z[c + 2 * q + 1] * m2);
            ov[q] = *reinterpret_cast<uint32_t*>(&b2);
          }
          *reinterpret_cast<uint4*>(dq + (((int64_t)s0 + t * kTile + r) * hq + h) * D + c) = out;
        }
      }
      continue;
    }
    for (int i = threadIdx.x; i < rows * kVpr; i += blockDim.x) {
      const int r = i / kVpr, col = (i % kVpr) * kVec;
      const __half* chunk = acc + dq_chunk_elems(tile, h, col / 32, hq, D);
      const uint4 in = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(chunk) +
                                                       dq_chunk_byte(r, (col % 32) * 2));
      const __half2* hv = reinterpret_cast<const __half2*>(&in);
      uint4 out;
      uint32_t* ov = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(hv[q]);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * mul, f.y * mul);
        ov[q] = *reinterpret_cast<uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(dq + (((int64_t)s0 + t * kTile + r) * hq + h) * D + col) = out;
    }
  }
  // rows outside every document
  const int64_t tq = (int64_t)(T - valid) * hq * kVpr, tk = (int64_t)(T - valid) * hkv * kVpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < tq + 2 * tk;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < tq) reinterpret_cast<uint4*>(dq)[(int64_t)valid * hq * kVpr + i] = make_uint4(0, 0, 0, 0);
    else if (i < tq + tk) reinterpret_cast<uint4*>(dk)[(int64_t)valid * hkv * kVpr + (i - tq)] = make_uint4(0, 0, 0, 0);
    else reinterpret_cast<uint4*>(dv)[(int64_t)valid * hkv * kVpr + (i - tq - tk)] = make_uint4(0, 0, 0, 0);
  }
}

// d = 128 (default and mixed routes): as dq_finalize_kernel for the head-dim-major
// dQ^T chunks, transposed through shared memory.  Persistent CTAs walk the
// (document tile, query head) chunks; each 32 KB chunk is copied into one of two
// shared-memory buffers with cp.async while the previous one is converted, so two
// chunks per CTA are in flight.  Thread = (query row q, head-dim half): it gathers
// the row's 64 values from the chunk (a warp reads 32 consecutive queries of one
// head-dim row, 64 contiguous bytes) and writes them as 32-byte stores of the
// row-major dQ row (16-byte ones if dQ is only 16-byte aligned).
constexpr int kDqtFinalizeSmem = 2 * 32768;

template <bool ROT = false>
__global__ void __launch_bounds__(256) dqt_finalize_kernel(const __half* acc, const int32_t* cu, const int* plan,
                                                           const float* boost, int N, int T, int hq, int hkv,
                                                           float scale, __nv_bfloat16* dq, __nv_bfloat16* dk,
                                                           __nv_bfloat16* dv) {
  constexpr int D = 128;
  extern __shared__ __align__(16) uint8_t fsm[];
  const bool bad = plan[kPlanStatus] & FLAMIA_DEV_BAD_CU_SEQLENS;
  const int valid = bad ? 0 : plan[kPlanValid];
  const int ntiles = bad ? 0 : plan[kPlanTiles];
  const PlanView pv = plan_view(plan, T, N);
  const int64_t units = (int64_t)ntiles * hq;
  const bool al32 = (reinterpret_cast<uintptr_t>(dq) & 31) == 0;
  auto issue = [&](int64_t un, int buf) {      // this thread's eight 16-byte pieces of the chunk
    const uint8_t* src = reinterpret_cast<const uint8_t*>(acc + dqt_chunk_elems(un / hq, (int)(un % hq), hq));
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int off = (k * 256 + (int)threadIdx.x) * 16;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(fsm + buf * 32768 + off)),
                   "l"(src + off)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  const int q = threadIdx.x & 127, half = threadIdx.x >> 7;
  // a unit's rows and scale; looked up for the next unit while its chunk is in flight
  struct Meta {
    int64_t row0;         // first token of the tile
    int rows, h;
    float mul;
  };
  auto meta = [&](int64_t un) {
    Meta m;
    const int tile = (int)(un / hq);
    m.h = (int)(un % hq);
    const int doc = upper_doc(pv.tile_prefix, N, tile);
    const int t = tile - pv.tile_prefix[doc];
    const int s0 = cu[doc];
    m.row0 = (int64_t)s0 + t * kTile;
    m.rows = min(kTile, cu[doc + 1] - s0 - t * kTile);
    m.mul = scale / boost[(int64_t)doc * hq + m.h];
    return m;
  };
  int buf = 0;
  Meta cur{};
  if ((int64_t)blockIdx.x < units) {
    issue(blockIdx.x, 0);
    cur = meta(blockIdx.x);
  }
  for (int64_t un = blockIdx.x; un < units; un += gridDim.x, buf ^= 1) {
    const bool more = un + gridDim.x < units;
    Meta nxt{};
    if (more) {
      issue(un + gridDim.x, buf ^ 1);   // that buffer was released by the barrier closing the last pass
      nxt = meta(un + gridDim.x);
    }
    if (more) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int rows = cur.rows, h = cur.h;
    if (q < rows) {
      const float mul = cur.mul;
      const uint8_t* base = fsm + buf * 32768 + (q >> 6) * 16384 + (q & 7) * 2;
      const int unit = (q & 63) >> 3;
      __nv_bfloat16* orow = dq + ((cur.row0 + q) * hq + h) * D + half * 64;
      auto val = [&](int d) {
        return __half2float(*reinterpret_cast<const __half*>(base + d * 128 + ((unit ^ (d & 7)) << 4)));
      };
      // rotated operands: this thread's half of the row times H / 16 (H = H_2 x H_64: the
      // half's sign on the other half, then the 64-point butterflies, strides 1 .. 32)
      float z[ROT ? 64 : 1];
      if constexpr (ROT) {
#pragma unroll
        for (int c = 0; c < 64; ++c) z[c] = half ? val(c) - val(c + 64) : val(c) + val(c + 64);
#pragma unroll
        for (int st = 1; st < 64; st <<= 1)
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (!(i & st)) {
              const float a = z[i], b = z[i + st];
              z[i] = a + b;
              z[i + st] = a - b;
            }
      }
      const float m2 = ROT ? mul * 0.0625f : mul;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int d = half * 64 + c * 16 + 2 * j;
          const float a = ROT ? z[ROT ? c * 16 + 2 * j : 0] : val(d);
          const float b = ROT ? z[ROT ? c * 16 + 2 * j + 1 : 0] : val(d + 1);
          __nv_bfloat162 b2 = __floats2bfloat162_rn(a * m2, b * m2);
          pk[j] = *reinterpret_cast<uint32_t*>(&b2);
        }
        __nv_bfloat16* dst = orow + c * 16;
        if (al32) {
          st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
        } else {
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
    __syncthreads();
    cur = nxt;
  }
  constexpr int kVpr = D / 8;
  const int64_t tq = (int64_t)(T - valid) * hq * kVpr, tk = (int64_t)(T - valid) * hkv * kVpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < tq + 2 * tk;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < tq) reinterpret_cast<uint4*>(dq)[(int64_t)valid * hq * kVpr + i] = make_uint4(0, 0, 0, 0);
    else if (i < tq + tk) reinterpret_cast<uint4*>(dk)[(int64_t)valid * hkv * kVpr + (i - tq)] = make_uint4(0, 0, 0, 0);
    else reinterpret_cast<uint4*>(dv)[(int64_t)valid * hkv * kVpr + (i - tq - tk)] = make_uint4(0, 0, 0, 0);
  }
}

// Strict causal dQ boost ([EN] section 4, "the causal accumulator scale combines
// ||dO_i|| with running maxima of key and value magnitudes"): per query row,
// M_i = 2 ||dO^_i|| max_{j<=i} ||V^_j|| max_{j<=i,d} |K^_jd| over the document and
// c_i = 2^floor(log2(2^headroom / M_i)) (1 where M_i = 0).  One CTA per
// (document, query head), a chunked prefix-max scan over the document's tokens.
__global__ void __launch_bounds__(256) causal_boost_kernel(const int32_t* cu, const int* plan, const float2* st_do,
                                                           const float2* st_k, const float2* st_v, int T, int hq,
                                                           int hkv, int headroom, float* cvec) {
  const int doc = blockIdx.x, h = blockIdx.y;
  const int hk = h / (hq / hkv);
  if (plan[kPlanStatus] & FLAMIA_DEV_BAD_CU_SEQLENS) return;
  const int s0 = cu[doc], s1 = cu[doc + 1];
  __shared__ float wv[8], wk[8];
  __shared__ float carry[2];
  if (threadIdx.x == 0) carry[0] = carry[1] = 0.f;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = s0; base < s1; base += 256) {
    const int t = base + threadIdx.x;
    const bool in = t < s1;
    float v = in ? st_v[(int64_t)t * hkv + hk].x : 0.f;
    float k = in ? st_k[(int64_t)t * hkv + hk].y : 0.f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float pv = __shfl_up_sync(0xffffffffu, v, o), pk = __shfl_up_sync(0xffffffffu, k, o);
      if (lane >= o) { v = fmaxf(v, pv); k = fmaxf(k, pk); }
    }
    if (lane == 31) { wv[warp] = v; wk[warp] = k; }
    __syncthreads();
    float cv = carry[0], ck = carry[1];
    for (int w = 0; w < warp; ++w) { cv = fmaxf(cv, wv[w]); ck = fmaxf(ck, wk[w]); }
    v = fmaxf(v, cv);
    k = fmaxf(k, ck);
    if (in) {
      const double M = 2.0 * (double)st_do[(int64_t)t * hq + h].x * (double)v * (double)k;
      double cb = 1.0;
      if (M > 0.0 && M < 1e300) {
        const double target = ldexp(1.0, headroom);
        int e = (int)floor(log2(target / M));
        while (ldexp(M, e) > target) --e;
        while (ldexp(M, e + 1) <= target) ++e;
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
        cb = ldexp(1.0, e);
      }
      cvec[(int64_t)h * T + t] = (float)cb;
    }
    __syncthreads();
    if (threadIdx.x == 255) { carry[0] = v; carry[1] = k; }
    __syncthreads();
  }
}

// Rows outside every document: dQ, dK and dV are zero.
template <int D>
__global__ void bwd_tail_kernel(const int* plan, int T, int hq, int hkv, __nv_bfloat16* dq, __nv_bfloat16* dk,
                                __nv_bfloat16* dv) {
  const bool bad = plan[kPlanStatus] & FLAMIA_DEV_BAD_CU_SEQLENS;
  const int valid = bad ? 0 : plan[kPlanValid];
  const int64_t nq = (int64_t)(T - valid) * hq * (D / 8), nk = (int64_t)(T - valid) * hkv * (D / 8);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nq + 2 * nk; i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nq) reinterpret_cast<uint4*>(dq)[(int64_t)valid * hq * (D / 8) + i] = make_uint4(0, 0, 0, 0);
    else if (i < nq + nk) reinterpret_cast<uint4*>(dk)[(int64_t)valid * hkv * (D / 8) + (i - nq)] = make_uint4(0, 0, 0, 0);
    else reinterpret_cast<uint4*>(dv)[(int64_t)valid * hkv * (D / 8) + (i - nq - nk)] = make_uint4(0, 0, 0, 0);
  }
}

// Deterministic dQ (strict options): one CTA per (forward work item, query head)
// processes the item's query tiles one after another; for each, the visible key
// tiles in increasing order.  Two compute warpgroups share each (query tile, key
// tile) pair: warpgroup g takes key columns [64 g, 64 g + 64) of S and dP and the
// head-dim columns [D/2 g, D/2 (g + 1)) of the dQ accumulator.  Thread = query row
// of its warpgroup.  Per key tile: S = Q K^T and
// dP = dO V^T (unscaled E4M3 MMAs), P = 2^(x - LSE log2 e), dS = P o (dP - D),
// the K fold dS'' = dS s_K(j) quantized with one round-up exponent per (query
// row, 32-key block) (the strict per-row dS exponent), dQ partial = dS'' K^ codes
// (MXF8 MMA), then acc = fp16(acc + fp16(c_i * partial)) in registers in the
// fixed key-tile order; finally dQ = bf16(scale * acc / c_i).
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 2 TMEM
// allocator, warp 3 per-key factors (s_K, s_V) into SMEM, warps 4-11 compute.
// TMEM: S [0,128), dP [128,256), dQ partial [256, 256 + D).  The dQ MMA's four
// instructions (one per 32-key block) take their A scale words from separate
// columns, written by the warpgroup that owns the block into the dP columns it has
// itself read (warpgroup 0: dP columns 0-7 and the B words in 8-11; warpgroup 1:
// 64-71).
constexpr int kDqStages = 4;     // K/V ring: each pair loads a new key tile
constexpr int kDqKd = 4;         // per-key factor buffers
constexpr int kDqThreads = 384;

struct DqParams {
  const uint8_t* q_scales;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  const uint8_t* do_scales;
  const float* lse;
  const float* dvec;
  const float* cvec;       // [hq, T] causal boosts
  const int32_t* cu;
  const int* plan;
  int N, T, hq, hkv;
  float scale_log2, scale;
  __nv_bfloat16* dq;
};

template <int D>
struct DqSmem {
  static constexpr int kTileBytes = kTile * D;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTileBytes;
  static constexpr int kK = kDO + kTileBytes;                  // [kDqStages]
  static constexpr int kV = kK + kDqStages * kTileBytes;       // [kDqStages]
  static constexpr int kDS = kV + kDqStages * kTileBytes;      // dS'' codes, [query][key]
  static constexpr int kKD = kDS + kTile * kTile;              // per-key factors [kDqKd buffers][2][128] floats
  static constexpr int kBar = kKD + kDqKd * 2 * 128 * 4;
  static constexpr int kBytes = kBar + 256;
  // at least 116 KB so that one CTA (holding all 512 TMEM columns) fits per SM
  static constexpr int kAlloc = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
};

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
    attn_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const DqParams p) {
  using L = DqSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* qd_full = bars + 0;
  uint64_t* qd_empty = bars + 1;
  uint64_t* kv_full = bars + 2;                 // [kDqStages]
  uint64_t* kv_empty = bars + 2 + kDqStages;    // [kDqStages]
  uint64_t* kd_full = bars + 2 + 2 * kDqStages; // [kDqKd]
  uint64_t* kd_empty = kd_full + kDqKd;         // [kDqKd]
  uint64_t* s_full = kd_empty + kDqKd;
  uint64_t* p_full = s_full + 1;
  uint64_t* dq_full = s_full + 2;
  uint64_t* dq_empty = s_full + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 4);
  int* status = const_cast<int*>(p.plan) + kPlanStatus;

  const int n_items = p.plan[kPlanFwdItems];
  const int item_idx = blockIdx.x / p.hq;
  const int h = blockIdx.x % p.hq;
  if (item_idx >= n_items) return;
  const PlanView pv = plan_view(p.plan, p.T, p.N);
  const int4 item = pv.fwd_items[item_idx];
  const int2 span = pv.fwd_span[item_idx];      // loaded alongside the item (no dependent load)
  const int t0 = item.y, ntq = item.z;
  const int doc_start = span.x;
  const int doc_len = span.y;
  const int hk = h / (p.hq / p.hkv);
  // pairs (query tile w, key tile u), w-major, u = 0 .. t0 + w
  const int npairs = ntq == 1 ? t0 + 1 : 2 * t0 + 3;
  auto pair_of = [&](int k, int& w, int& u) {
    if (k <= t0) { w = 0; u = k; } else { w = 1; u = k - (t0 + 1); }
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    mbar_init(qd_empty, 1);
    for (int i = 0; i < kDqStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < kDqKd; ++i) {
      mbar_init(&kd_full[i], 32);
      mbar_init(&kd_empty[i], 256);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 256);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  constexpr uint32_t kS = 0, kP = 128, kDQ = 256;
  // scale words of the dQ MMA: A of key block s (byte s, replicated), B (1.0)
  auto a_sf = [](int s) -> uint32_t { return kP + 64 * (s >> 1) + 4 * (s & 1); };
  constexpr uint32_t kSFB = kP + 8;
  constexpr uint32_t kLayout = D == 128 ? kSwizzle128B : kSwizzle64B;
  constexpr uint32_t kAtom = 8 * D;
  float* kdbuf = reinterpret_cast<float*>(smem + L::kKD);

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      for (int k = 0; k < npairs && ok; ++k) {
        int w, u;
        pair_of(k, w, u);
        if (u == 0) {     // a new query tile: Q and dO codes
          if (w == 1) ok = mbar_wait(qd_empty, 0, status);
          if (!ok) break;
          mbar_arrive_expect_tx(qd_full, 2 * L::kTileBytes);
          tma_load_3d(smem + L::kQ, &tm_q, qd_full, 0, h, doc_start + (t0 + w) * kTile);
          tma_load_3d(smem + L::kDO, &tm_do, qd_full, 0, h, doc_start + (t0 + w) * kTile);
        }
        const int st = k % kDqStages;
        if (k >= kDqStages && !mbar_wait(&kv_empty[st], ((k / kDqStages) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * L::kTileBytes);
        tma_load_3d(smem + L::kK + st * L::kTileBytes, &tm_k, &kv_full[st], 0, hk, doc_start + u * kTile);
        tma_load_3d(smem + L::kV + st * L::kTileBytes, &tm_v, &kv_full[st], 0, hk, doc_start + u * kTile);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sq = smem_u32(smem + L::kQ), sdo = smem_u32(smem + L::kDO), sk = smem_u32(smem + L::kK),
                     sv = smem_u32(smem + L::kV), sds = smem_u32(smem + L::kDS);
      bool ok = true;
      for (int k = 0; k < npairs && ok; ++k) {
        int w, u;
        pair_of(k, w, u);
        const int st = k % kDqStages;
        if (u == 0) ok = mbar_wait(qd_full, w, status);
        if (ok) ok = mbar_wait(&kv_full[st], (k / kDqStages) & 1, status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = sk + st * L::kTileBytes, va = sv + st * L::kTileBytes;
#pragma unroll
        for (int s = 0; s < D / 32; ++s) {
          mma_f8(tbase + kS, smem_desc(sq + 32 * s, 16, kAtom, kLayout), smem_desc(ka + 32 * s, 16, kAtom, kLayout),
                 idesc_f8(128, 128, 0, 0), s > 0);
          mma_f8(tbase + kP, smem_desc(sdo + 32 * s, 16, kAtom, kLayout), smem_desc(va + 32 * s, 16, kAtom, kLayout),
                 idesc_f8(128, 128, 0, 0), s > 0);
        }
        mma_commit(s_full);
        ok = mbar_wait(p_full, k & 1, status);
        if (ok && k > 0) ok = mbar_wait(dq_empty, (k - 1) & 1, status);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          // dQ partial = dS'' K (A: queries x keys, K-major; B: K keys x d, MN-major)
          mma_mxf8(tbase + kDQ, smem_desc(sds + 32 * s, 16, 1024, kSwizzle128B),
                   smem_desc(ka + s * 32 * D, kAtom, kAtom, kLayout), idesc_mxf8(128, D, 0, 1, s, s),
                   tbase + a_sf(s), tbase + kSFB, s > 0);
        }
        mma_commit(dq_full);
        mma_commit(&kv_empty[st]);
        if (u == t0 + w) mma_commit(qd_empty);     // last key tile of this query tile
      }
      if (!ok) {
        mma_commit(dq_full);
        mbar_wait(dq_full, 0, status);
      }
    }
  } else if (warp == 3) {
    // per-key factors s_K(j), s_V(j) of each key tile; a pair's global loads are all
    // issued into registers before the wait for the buffer and the shared-memory stores,
    // so that their latencies overlap instead of queueing behind stores the compiler
    // cannot reorder them past
    for (int k = 0; k < npairs; ++k) {
      int w, u;
      pair_of(k, w, u);
      const int b = k % kDqKd;
      uint32_t ks[4], vs[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kl = u * kTile + q * 32 + lane;
        const int64_t ktok = (int64_t)doc_start + kl;
        ks[q] = kl < doc_len ? __ldg(p.k_scales + ktok * p.hkv + hk) : 127u;   // 127: 2^0 past the end
        vs[q] = kl < doc_len ? __ldg(p.v_scales + ktok * p.hkv + hk) : 127u;
      }
      if (k >= kDqKd && !__all_sync(0xffffffffu, mbar_wait(&kd_empty[b], ((k / kDqKd) - 1) & 1, status))) break;
      float* kd = kdbuf + b * 256;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        kd[q * 32 + lane] = ue8m0_to_f32(ks[q]);
        kd[128 + q * 32 + lane] = ue8m0_to_f32(vs[q]);
      }
      mbar_arrive(&kd_full[b]);
    }
  } else if (warp >= 4) {
    const int g = (warp - 4) >> 2;                   // warpgroup: key columns [64 g, 64 g + 64), dQ half g
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;               // query row within the tile (TMEM lane)
    const uint32_t lane_base = tbase + ((uint32_t)(quarter * 32) << 16);
    uint8_t* sDS = smem + L::kDS;
    constexpr int kHalf = D / 2;                      // head-dim columns of this warpgroup's dQ half
    bool ok = true;
    __half2 acc[kHalf / 2];
    float nl = 0.f, nd = 0.f, fq = 0.f, sdo = 0.f, cb = 1.f;
    bool qv = false;
    int64_t qtok = 0;
    for (int k = 0; k < npairs; ++k) {
      int w, u;
      pair_of(k, w, u);
      const int t = t0 + w;
      if (u == 0) {
        const int ql = t * kTile + i;
        qv = ql < doc_len;
        qtok = (int64_t)doc_start + ql;
        nl = qv ? -p.lse[(int64_t)h * p.T + qtok] * 1.4426950408889634f : -INFINITY;
        nd = qv ? -p.dvec[(int64_t)h * p.T + qtok] : 0.f;
        fq = qv ? p.scale_log2 * ue8m0_to_f32(p.q_scales[qtok * p.hq + h]) : 0.f;
        sdo = qv ? ue8m0_to_f32(p.do_scales[qtok * p.hq + h]) : 0.f;
        cb = qv ? p.cvec[(int64_t)h * p.T + qtok] : 1.f;
#pragma unroll
        for (int c = 0; c < kHalf / 2; ++c) acc[c] = __floats2half2_rn(0.f, 0.f);
      }
      const bool diag = (u == t);
      const int b = k % kDqKd;
      const float* kd = kdbuf + b * 256;
      ok = named_bar_and(1, 256, mbar_wait(s_full, k & 1, status) && mbar_wait(&kd_full[b], (k / kDqKd) & 1, status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * g + cc;                     // 32-key block
        float ds[32];
        float amax = 0.f;
        {
          uint32_t vs[32], vp[32];
          tmem_ld32(lane_base + kS + 32 * c, vs);
          tmem_ld32(lane_base + kP + 32 * c, vp);
          tmem_ld_wait();
#pragma unroll
          for (int jh = 0; jh < 32; ++jh) {
            const int jj = jh;
            const int j = 32 * c + jj;
            const float sk = kd[j];
            const float x = __uint_as_float(vs[jh]) * (fq * sk) + nl;
            const bool vis = !diag || j <= i;
            const float pr = vis ? fast_exp2(x) : 0.f;
            const float dp = __uint_as_float(vp[jh]) * (sdo * kd[128 + j]) + nd;
            const float v = pr * dp * sk;              // K fold
            ds[jj] = v;
            amax = fmaxf(amax, fabsf(v));
          }
        }
        const int e = roundup_exp(amax);
        const float sc = exp2i(-e);
        uint32_t pk[8];
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4)
          pk[jj >> 2] = (uint32_t)e4m3x2(ds[jj] * sc, ds[jj + 1] * sc) | ((uint32_t)e4m3x2(ds[jj + 2] * sc, ds[jj + 3] * sc) << 16);
        *reinterpret_cast<uint4*>(sDS + swz_offset(i, 32 * c, 128)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(sDS + swz_offset(i, 32 * c + 16, 128)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        // A scale of row i for key block c: lane i, column (a_sf(c) + i / 32), the
        // exponent in every byte (the instruction reads byte c)
        tmem_st1(lane_base + a_sf(c) + quarter, (uint32_t)(e + 127) * 0x01010101u);
      }
      if (g == 0) tmem_st4(lane_base + kSFB, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);   // B: K codes, 1.0
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&kd_empty[b]);
      mbar_arrive(p_full);
      ok = named_bar_and(1, 256, mbar_wait(dq_full, k & 1, status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      {
        uint32_t v[kHalf];                             // the partial's columns, one TMEM round trip
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c)
          tmem_ld32(lane_base + kDQ + kHalf * g + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < kHalf / 2; ++q) {
          const __half2 hpart = __floats2half2_rn(__uint_as_float(v[2 * q]) * cb, __uint_as_float(v[2 * q + 1]) * cb);
          acc[q] = __hadd2(acc[q], hpart);
        }
      }
      tc_fence_before();
      mbar_arrive(dq_empty);
      if (u == t && qv) {          // last key tile of this query tile: dQ = bf16(scale * acc / c_i)
        const float mul = p.scale / cb;
        __nv_bfloat16* orow = p.dq + (qtok * p.hq + h) * D + kHalf * g;
#pragma unroll
        for (int c = 0; c < kHalf / 8; ++c) {
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __half22float2(acc[4 * c + q]);
            __nv_bfloat162 b2 = __floats2bfloat162_rn(f.x * mul, f.y * mul);
            o[q] = *reinterpret_cast<uint32_t*>(&b2);
          }
          reinterpret_cast<uint4*>(orow)[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
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

template <int D, bool STRICT, bool MIXED, bool DBG = false, bool WIN = false, bool ROT = false>
cudaError_t launch_bwd_d(const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                         const void* vs, const void* doc_codes, const void* dos, const float* lse, const float* dvec,
                         const float* boost, const int32_t* cu, int N, int T, int hq, int hkv, float scale,
                         const void* plan, void* dq_acc, void* dq, void* dk, void* dv, cudaStream_t stream,
                         void* const* ev, const void* q4c, const void* q4s, const void* k4c, const void* k4s,
                         float* dbg, Window win) {
  CUtensorMap tq, tk, tv, tdo, tq4, tk4, tdk, tdv;
  if (!make_tmap_bf16_3d(&tdk, dk, D, hkv, T, D * 2, (uint64_t)hkv * D * 2, 64, kTile) ||
      !make_tmap_bf16_3d(&tdv, dv, D, hkv, T, D * 2, (uint64_t)hkv * D * 2, 64, kTile))
    return cudaErrorInvalidValue;
  if (!make_tmap_u8_3d(&tq, qc, D, hq, T, D, (uint64_t)hq * D, D, kTile) ||
      !make_tmap_u8_3d(&tk, kc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile) ||
      !make_tmap_u8_3d(&tv, vc, D, hkv, T, D, (uint64_t)hkv * D, D, kTile) ||
      !make_tmap_u8_3d(&tdo, doc_codes, D, hq, T, D, (uint64_t)hq * D, D, kTile))
    return cudaErrorInvalidValue;
  if (MIXED) {
    if (!make_tmap_u8_3d(&tq4, q4c, D / 2, hq, T, D / 2, (uint64_t)hq * D / 2, D / 2, kTile) ||
        !make_tmap_u8_3d(&tk4, k4c, D / 2, hkv, T, D / 2, (uint64_t)hkv * D / 2, D / 2, kTile))
      return cudaErrorInvalidValue;
  } else {
    tq4 = tq;
    tk4 = tk;
  }
  BwdParams p;
  p.q_scales = static_cast<const uint8_t*>(qs);
  p.k_scales = static_cast<const uint8_t*>(ks);
  p.v_scales = static_cast<const uint8_t*>(vs);
  p.do_scales = static_cast<const uint8_t*>(dos);
  p.lse = lse;
  p.dvec = dvec;
  p.boost = boost;
  p.cu = cu;
  p.plan = static_cast<const int*>(plan);
  p.N = N;
  p.T = T;
  p.hq = hq;
  p.hkv = hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.scale = scale;
  p.q4_scales = static_cast<const uint8_t*>(q4s);
  p.k4_scales = static_cast<const uint8_t*>(k4s);
  p.dq_acc = static_cast<__half*>(dq_acc);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dbg = dbg;
  p.win = win;
  const int64_t max_items = (int64_t)T / kTile + N + 1;
  const int64_t grid = max_items * hkv;
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  constexpr int smem = BwdSmem<D, MIXED>::kAlloc;
  int regs = 0;
  cudaError_t e = prepare_kernel<attn_bwd_kernel<D, STRICT, MIXED, DBG, WIN, ROT>>(smem, &regs);
  if (e != cudaSuccess) return e;
  // the warpgroups' register split (setmaxnreg) assumes this launch allocation;
  // with any other the increase could never be granted, so refuse to launch
  if (regs != BwdShape<D, STRICT>::kLaunchRegs) return cudaErrorInvalidConfiguration;
  if (ev) record_timing_event(ev[0], stream);
  attn_bwd_kernel<D, STRICT, MIXED, DBG, WIN, ROT>
      <<<(unsigned)grid, BwdShape<D, STRICT>::kThreads, smem, stream>>>(tq, tk, tv, tdo, tq4, tk4, tdk, tdv, p);
  e = cudaGetLastError();
  if (ev) record_timing_event(ev[1], stream);
  if (e != cudaSuccess) return e;
  if (ev) record_timing_event(ev[2], stream);
  if (!STRICT && D == 128) {
    e = prepare_kernel<dqt_finalize_kernel<ROT>>(kDqtFinalizeSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    dqt_finalize_kernel<ROT><<<3 * sms, 256, kDqtFinalizeSmem, stream>>>(static_cast<const __half*>(dq_acc), cu, p.plan,
                                                                    boost, N, T, hq, hkv, scale,
                                                                    static_cast<__nv_bfloat16*>(dq), p.dk, p.dv);
  } else if (!STRICT) {
    dq_finalize_kernel<D, ROT><<<4 * 152, 256, 0, stream>>>(static_cast<const __half*>(dq_acc), cu, p.plan, boost, N, T, hq,
                                                       hkv, scale, static_cast<__nv_bfloat16*>(dq), p.dk, p.dv);
  } else {
    DqParams dp;
    dp.q_scales = p.q_scales;
    dp.k_scales = p.k_scales;
    dp.v_scales = p.v_scales;
    dp.do_scales = p.do_scales;
    dp.lse = lse;
    dp.dvec = dvec;
    dp.cvec = boost;
    dp.cu = cu;
    dp.plan = p.plan;
    dp.N = N;
    dp.T = T;
    dp.hq = hq;
    dp.hkv = hkv;
    dp.scale_log2 = p.scale_log2;
    dp.scale = scale;
    dp.dq = static_cast<__nv_bfloat16*>(dq);
    constexpr int dsmem = DqSmem<D>::kAlloc;
    e = prepare_kernel<attn_dq_kernel<D>>(dsmem);
    if (e != cudaSuccess) return e;
    const int64_t dgrid = ((int64_t)T / (kTile * kItemTiles) + N + 1) * hq;
    if (dgrid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    attn_dq_kernel<D><<<(unsigned)dgrid, kDqThreads, dsmem, stream>>>(tq, tk, tv, tdo, dp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_tail_kernel<D><<<152, 256, 0, stream>>>(p.plan, T, hq, hkv, static_cast<__nv_bfloat16*>(dq), p.dk, p.dv);
  }
  e = cudaGetLastError();
  if (ev) record_timing_event(ev[3], stream);
  return e;
}

}  // namespace

cudaError_t launch_boost(const int32_t* cu, int N, const void* plan, const float* st_do, const float* st_k,
                         const float* st_v, int T, int hq, int hkv, int headroom, float* boost, bool causal,
                         const float* maxima, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (causal)
    causal_boost_kernel<<<dim3(N, hq), 256, 0, s>>>(cu, static_cast<const int*>(plan),
                                                    reinterpret_cast<const float2*>(st_do),
                                                    reinterpret_cast<const float2*>(st_k),
                                                    reinterpret_cast<const float2*>(st_v), T, hq, hkv, headroom, boost);
  else
    boost_from_max_kernel<<<(N * hq + 255) / 256, 256, 0, s>>>(maxima, static_cast<const int*>(plan), N, hq, headroom,
                                                               boost);
  return cudaGetLastError();
}

cudaError_t launch_bwd(int D, const void* qc, const void* qs, const void* kc, const void* ks, const void* vc,
                       const void* vs, const void* doc_codes, const void* dos, const float* lse, const float* dvec,
                       const float* boost, const int32_t* cu, int N, int T, int hq, int hkv, float scale,
                       const void* plan, void* dq_acc, void* dq, void* dk, void* dv, cudaStream_t stream,
                       void* const* ev, bool strict, const void* q4c, const void* q4s, const void* k4c,
                       const void* k4s, float* dbg, Window win, bool rot) {
#define FLAMIA_BWD_ARGS qc, qs, kc, ks, vc, vs, doc_codes, dos, lse, dvec, boost, cu, N, T, hq, hkv, scale, plan, \
                        dq_acc, dq, dk, dv, stream, ev, q4c, q4s, k4c, k4s, dbg, win
  const bool mixed = q4c != nullptr;
  if ((strict || mixed) && (win.left >= 0 || win.right != 0)) return cudaErrorInvalidValue;   // causal only
  if (dbg && (mixed || strict)) return cudaErrorInvalidValue;
  const bool causal = win.left < 0 && win.right == 0;
  if (dbg && !causal) return cudaErrorInvalidValue;
  if (dbg && D == 128) return launch_bwd_d<128, false, false, true>(FLAMIA_BWD_ARGS);
  if (dbg && D == 64) return launch_bwd_d<64, false, false, true>(FLAMIA_BWD_ARGS);
  if (rot && (mixed || strict || dbg)) return cudaErrorInvalidValue;
  if (rot && D == 128)
    return causal ? launch_bwd_d<128, false, false, false, false, true>(FLAMIA_BWD_ARGS)
                  : launch_bwd_d<128, false, false, false, true, true>(FLAMIA_BWD_ARGS);
  if (rot && D == 64)
    return causal ? launch_bwd_d<64, false, false, false, false, true>(FLAMIA_BWD_ARGS)
                  : launch_bwd_d<64, false, false, false, true, true>(FLAMIA_BWD_ARGS);
  if (!causal && D == 128) return launch_bwd_d<128, false, false, false, true>(FLAMIA_BWD_ARGS);
  if (!causal && D == 64) return launch_bwd_d<64, false, false, false, true>(FLAMIA_BWD_ARGS);
  if (D == 128 && mixed) return launch_bwd_d<128, false, true>(FLAMIA_BWD_ARGS);
  if (mixed) return cudaErrorInvalidValue;
  if (D == 128 && strict) return launch_bwd_d<128, true, false>(FLAMIA_BWD_ARGS);
  if (D == 128) return launch_bwd_d<128, false, false>(FLAMIA_BWD_ARGS);
  if (D == 64 && strict) return launch_bwd_d<64, true, false>(FLAMIA_BWD_ARGS);
  if (D == 64) return launch_bwd_d<64, false, false>(FLAMIA_BWD_ARGS);
#undef FLAMIA_BWD_ARGS
  return cudaErrorInvalidValue;
}

}  // namespace flamia
