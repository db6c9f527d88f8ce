// Token-block MXFP8 quantizer (step a1 of the hot path) and its fused
// backward-prep variant (step a7).
//
// FLAMIA technical review section 3 ("Why one shared exponent can serve two
// reductions"): one UE8M0 exponent per document-local block of <= 32
// consecutive tokens x the whole head dimension; section 4: the exponent is
// the smallest with amax <= 448 * 2^e (round-up rule, never clamps); section
// 6: blocks are local to each document and the scale metadata is dense (one
// byte per token).  The per-token variant is the strict option of section 4.
//
// Bandwidth-bound: one warp per (block, head); each lane moves 16 bytes per
// load (coalesced 128-bit accesses along head_dim); amax is a warp-shuffle
// max; codes come from the saturating round-to-nearest-even cvt to E4M3.
//
// The backward-prep variant (review Algorithm 1 step 09) encodes dO once and,
// in the same pass, computes D_i = dO^_i . O_i from the saved bf16 O and
// zeroes the fp16 dQ accumulator rows it owns.
//
// The rotated variant (review section 3, "Rotation, range, and the
// alternative"; Korean review section 3.4: rotation, block statistics, codes
// and scales in one pass) first multiplies each token row by H / 2^k (H the
// +-1 Sylvester Hadamard matrix, k = ceil(log2(d) / 2)) with the fast
// Walsh-Hadamard butterflies in fp32, strides 1, 2, ..., d/2 in increasing
// order: inside a lane's 16-byte vectors, then across the row's lanes
// (shuffles), then across the lane's vectors.
#include <cuda_fp4.h>

#include "common.cuh"
#include "ptx.cuh"

namespace flamia {

namespace {

// Launch shape: the plain quantizer holds its block in registers between the two
// passes (4 warps, 3 blocks per SM); the backward prep streams dO and O and keeps
// more warps in flight instead, re-reading the block from L1/L2 in pass 2.
// The rotated variant streams its block twice (one unit per warp, more warps in
// flight) instead of holding it next to the rotation's working values.
template <bool WITH_D, bool ROT = false>
struct QShape {
  static constexpr int kWarps = WITH_D || ROT ? 8 : 4;
  static constexpr int kMinBlocks = WITH_D || ROT ? 4 : 3;
};

// One launch quantizes up to three tensors of the same documents (Q, K and V of a
// training call): job i owns the work units [jobs[i-1].end, jobs[i].end).
struct QJob {
  const __nv_bfloat16* x;     // bf16 [T, H, D]
  uint8_t* codes;             // E4M3 [T, H, D]
  uint8_t* scales;            // UE8M0 [T, H]
  float2* stats;              // [T, H] row statistics, or null
  int H;
  int64_t end;                // one past the job's last work unit (cumulative over the jobs)
};
struct QJobs {
  QJob j[3];
};

template <int D, bool PER_TOKEN, bool STATS, bool WITH_D, bool ROT = false>
__global__ void __launch_bounds__(QShape<WITH_D, ROT>::kWarps * 32, QShape<WITH_D, ROT>::kMinBlocks)
    quantize_kernel(const QJobs jobs, int T, const int32_t* __restrict__ cu, int N, const int* __restrict__ plan,
                    const __nv_bfloat16* __restrict__ o, float* __restrict__ dvec, __half* __restrict__ dq_acc,
                    const float2* __restrict__ k_stats, const float2* __restrict__ v_stats, int hkv,
                    float* __restrict__ maxima, int64_t nwork) {
  // Each lane owns 32 elements of a row as four 16-byte vectors, vector j at column
  // j * 8 kLpr + 8 (lane % kLpr): a load instruction reads kRpi rows x 16 kLpr
  // contiguous bytes, and per-row reductions take log2(kLpr) shuffle levels.
  constexpr int kLpr = D / 32;         // lanes per token row
  constexpr int kRpi = 32 / kLpr;      // rows per iteration
  constexpr int kIters = 32 / kRpi;    // 32 rows per warp
  const int lane = threadIdx.x & 31;
  constexpr int kWarps = QShape<WITH_D, ROT>::kWarps;
  constexpr bool kHold = !PER_TOKEN && !WITH_D && !ROT;   // block held in registers for pass 2
  static_assert(!ROT || (!PER_TOKEN && !WITH_D), "the rotation is fused into the token-block quantizer of Q and K");
  const PlanView pv = plan_view(plan, T, N);
  const int valid = plan[kPlanValid];
  const int nblk = plan[kPlanBlocks];
  const int sub = lane / kLpr;            // row within an iteration
  const int seg = lane % kLpr;
  auto col_of = [&](int j) { return j * 8 * kLpr + 8 * seg; };

  // Work unit gw = (32-row block, head); the warps walk the units with a grid stride.
  // Rows [r0, r0 + nrows); tail rows (no document) get zeros.
  struct QUnit {
    int h, r0, nrows, doc, dq_row0, job;
    bool tail, skip;
    int64_t dq_tile0;     // backward prep: accumulator tile of the block's document tile
  };
  auto unit_setup = [&](int64_t gw) {
    QUnit U;
    U.job = gw < jobs.j[0].end ? 0 : (gw < jobs.j[1].end ? 1 : 2);
    const int64_t local = gw - (U.job ? jobs.j[U.job - 1].end : 0);
    const int Hj = jobs.j[U.job].H;
    U.h = (int)(local % Hj);
    const int64_t unit = local / Hj;
    U.tail = false;
    U.skip = gw >= nwork;
    U.dq_tile0 = 0;
    U.dq_row0 = 0;
    U.doc = -1;
    U.r0 = 0;
    U.nrows = 0;
    if (U.skip) return U;
    if (PER_TOKEN) {
      U.r0 = (int)(unit * 32);
      U.skip = U.r0 >= T;
      U.nrows = min(32, T - U.r0);
    } else if (unit < nblk) {
      U.doc = upper_doc(pv.blk_prefix, N, (int)unit);
      const int s0 = cu[U.doc], s1 = cu[U.doc + 1];
      U.r0 = s0 + ((int)unit - pv.blk_prefix[U.doc]) * kBlock;
      U.nrows = min(kBlock, s1 - U.r0);
      U.dq_tile0 = pv.tile_prefix[U.doc] + (U.r0 - s0) / kTile;
      U.dq_row0 = (U.r0 - s0) % kTile;
    } else {
      U.r0 = valid + (int)(unit - nblk) * 32;
      U.skip = U.r0 >= T;
      U.nrows = min(32, T - U.r0);
      U.tail = true;
    }
    return U;
  };
  auto live_u = [&](const QUnit& U, int r) { return r < U.nrows && !U.tail && (!PER_TOKEN || U.r0 + r < valid); };
  // register-held variant: the next unit's block is prefetched into this lane's own
  // shared-memory slots (16 x 16 bytes, zero-filled where no row) with cp.async
  __shared__ uint4 pf_buf[kHold ? kWarps : 1][kHold ? kIters * 4 : 1][32];
  auto prefetch = [&](const QUnit& U) {
#pragma unroll
    for (int it = 0; it < kIters; ++it)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = it * kRpi + sub;
        const bool lv = !U.skip && live_u(U, r);
        const QJob& J = jobs.j[U.job];
        const __nv_bfloat16* src = J.x + ((int64_t)(lv ? U.r0 + r : 0) * J.H + U.h) * D + col_of(j);
        const uint32_t dst = smem_u32(&pf_buf[kHold ? (threadIdx.x >> 5) : 0][kHold ? it * 4 + j : 0][lane]);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(lv ? 16 : 0) : "memory");
      }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  const int64_t stride = (int64_t)gridDim.x * kWarps;
  int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  QUnit nextU;
  if constexpr (kHold) {
    nextU = unit_setup(gw);
    prefetch(nextU);
  }
  for (; gw < nwork; gw += stride) {
  // (the other variants launch one warp per unit and leave after one pass)
  const QUnit U = kHold ? nextU : unit_setup(gw);
  uint4 w[kHold ? kIters : 1][4];
  if constexpr (kHold) {
    nextU = unit_setup(gw + stride);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
    for (int it = 0; it < kIters; ++it)
#pragma unroll
      for (int j = 0; j < 4; ++j) w[kHold ? it : 0][j] = pf_buf[kHold ? (threadIdx.x >> 5) : 0][kHold ? it * 4 + j : 0][lane];
    if (!nextU.skip) prefetch(nextU);          // this lane's slots were just read
  }
  if (U.skip) continue;
  const QJob& J = jobs.j[U.job];
  const __nv_bfloat16* __restrict__ x = J.x;
  uint8_t* __restrict__ codes = J.codes;
  uint8_t* __restrict__ scales = J.scales;
  float2* __restrict__ stats = J.stats;
  const int H = J.H;
  const bool with_stats = STATS && stats != nullptr;     // uniform over the warp
  const int h = U.h, r0 = U.r0, nrows = U.nrows, doc = U.doc, dq_row0 = U.dq_row0;
  const bool tail = U.tail;
  const int64_t dq_tile0 = U.dq_tile0;
  auto live = [&](int r) { return live_u(U, r); };
  auto load8 = [&](const __nv_bfloat16* base, int r, int j) {
    return live(r) ? __ldg(reinterpret_cast<const uint4*>(base + ((int64_t)(r0 + r) * H + h) * D + col_of(j)))
                   : make_uint4(0, 0, 0, 0);
  };
  // the row's 32 values of this lane rotated by H / 2^k (fp32 butterflies, strides
  // 1, 2, 4 in the vectors, 8 .. 4 kLpr across the lanes, 8 kLpr, 16 kLpr across vectors)
  auto rotate = [&](const uint4 (&rw)[4], float (&v)[4][8]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&rw[j]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(b[q]);
        v[j][2 * q] = f.x;
        v[j][2 * q + 1] = f.y;
      }
#pragma unroll
      for (int st = 1; st < 8; st <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (!(i & st)) {
            const float a = v[j][i], c = v[j][i + st];
            v[j][i] = __fadd_rn(a, c);
            v[j][i + st] = __fsub_rn(a, c);
          }
    }
#pragma unroll
    for (int m = 1; m < kLpr; m <<= 1) {
      const bool upper = (seg & m) != 0;
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float o = __shfl_xor_sync(0xffffffffu, v[j][i], m);
          v[j][i] = upper ? __fsub_rn(o, v[j][i]) : __fadd_rn(v[j][i], o);
        }
    }
#pragma unroll
    for (int st = 1; st < 4; st <<= 1)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (!(j & st)) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float a = v[j][i], c = v[j + st][i];
            v[j][i] = __fadd_rn(a, c);
            v[j + st][i] = __fsub_rn(a, c);
          }
        }
    constexpr float kNorm = D == 128 ? 0.0625f : 0.125f;    // 2^-k
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) v[j][i] *= kNorm;
  };
  auto absmax8 = [](const uint4& w) {
    const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&w);
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(v[j]);
      m = fmax3(m, fabsf(f.x), fabsf(f.y));
    }
    return m;
  };

  float mdo = 0.f;        // backward prep: max ||dO^_i|| over the block's rows
  // pass 1 (token blocks): amax over the whole block; the plain quantizer keeps the
  // block in registers for pass 2 (32 rows x 64 bytes per lane)
  int e_block = 0;
  if (!PER_TOKEN) {
    float a = 0.f;
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      if constexpr (ROT) {
        float v[4][8];
        uint4 rw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) rw[j] = load8(x, it * kRpi + sub, j);
        rotate(rw, v);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int i = 0; i < 8; i += 2) a = fmax3(a, fabsf(v[j][i]), fabsf(v[j][i + 1]));
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 x4 = kHold ? w[kHold ? it : 0][j] : load8(x, it * kRpi + sub, j);
          a = fmaxf(a, absmax8(x4));
        }
      }
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o2));
    e_block = roundup_exp(a);
  }
#pragma unroll(kHold ? kIters : 1)
  for (int it = 0; it < kIters; ++it) {
    const int r = it * kRpi + sub;
    const bool inrange = r < nrows;
    uint4 raw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) raw[j] = kHold ? w[kHold ? it : 0][j] : load8(x, r, j);
    int e = e_block;
    if (PER_TOKEN) {
      float m = fmaxf(fmaxf(absmax8(raw[0]), absmax8(raw[1])), fmaxf(absmax8(raw[2]), absmax8(raw[3])));
#pragma unroll
      for (int o2 = kLpr / 2; o2 > 0; o2 >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o2));
      e = roundup_exp(m);
    }
    const float s = exp2i(-e);
    const float back = ue8m0_to_f32((uint32_t)(e + 127));
    float2 ss2 = make_float2(0.f, 0.f), dd2 = make_float2(0.f, 0.f);
    uint32_t cmax4 = 0;
    float rv[ROT ? 4 : 1][ROT ? 8 : 1];
    if constexpr (ROT) rotate(raw, rv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162* v = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
      uint32_t packed[2];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = ROT ? make_float2(rv[ROT ? j : 0][ROT ? 2 * q : 0], rv[ROT ? j : 0][ROT ? 2 * q + 1 : 0])
                             : __bfloat1622float2(v[q]);
        const uint16_t c2 = e4m3x2(f.x * s, f.y * s);
        if (q & 1) packed[q >> 1] |= (uint32_t)c2 << 16; else packed[q >> 1] = c2;
      }
      // statistics of the reconstructed row x^ = 2^e c and D = dO^ . O, from the codes:
      // sums over the decoded codes, scaled by 2^e (2^2e) once at the end (exact)
      if (with_stats || WITH_D) {
        const uint4 oraw = WITH_D ? load8(o, r, j) : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162* ov = reinterpret_cast<const __nv_bfloat162*>(&oraw);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint16_t c2 = (uint16_t)(packed[q >> 1] >> (16 * (q & 1)));
          const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c2, __NV_E4M3);
          const float2 f = __half22float2(__half2(hr));
          if (STATS) ss2 = ffma2(f, f, ss2);
          if (WITH_D) dd2 = ffma2(f, __bfloat1622float2(ov[q]), dd2);
        }
        if (STATS) cmax4 = __vmaxu4(cmax4, __vmaxu4(packed[0] & 0x7F7F7F7Fu, packed[1] & 0x7F7F7F7Fu));
      }
      if (inrange) {
        const int64_t row = r0 + r;
        const int col = col_of(j);
        *reinterpret_cast<uint2*>(codes + (row * H + h) * D + col) = make_uint2(packed[0], packed[1]);
        if (WITH_D && D == 64 && !PER_TOKEN && !tail && dq_acc)      // zero the row's slice of its accumulator chunk
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(dq_acc + dq_chunk_elems(dq_tile0, h, col / 32, H, D)) +
                                    dq_chunk_byte(dq_row0 + r, (col % 32) * 2)) = make_uint4(0, 0, 0, 0);
      }
    }
    float ss = 0.f, mx = 0.f, dd = 0.f;
    if (with_stats || WITH_D) {
      ss = ss2.x + ss2.y;
      dd = dd2.x + dd2.y;
      uint32_t cmax = max(max(cmax4 & 0xFFu, (cmax4 >> 8) & 0xFFu), max((cmax4 >> 16) & 0xFFu, cmax4 >> 24));
#pragma unroll
      for (int o2 = kLpr / 2; o2 > 0; o2 >>= 1) {
        if (STATS) {
          ss += __shfl_xor_sync(0xffffffffu, ss, o2);
          cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o2));
        }
        if (WITH_D) dd += __shfl_xor_sync(0xffffffffu, dd, o2);
      }
      if (STATS) mx = e4m3_to_f32((uint8_t)cmax) * back;   // |code| orders like |value|
    }
    if (inrange && seg == 0) {
      const int64_t row = r0 + r;
      if (with_stats) stats[row * H + h] = make_float2(sqrtf(ss) * back, mx);
      if (WITH_D && !tail) mdo = fmaxf(mdo, sqrtf(ss) * back);
      if (WITH_D) dvec[(int64_t)h * T + row] = dd * back;
      if (PER_TOKEN) scales[row * H + h] = (uint8_t)(e + 127);
    }
  }
  if (!PER_TOKEN && lane < nrows) scales[(int64_t)(r0 + lane) * H + h] = (uint8_t)(tail ? 127 : e_block + 127);
  if (WITH_D && D == 128 && !PER_TOKEN && !tail && dq_acc) {
    // head-dim-major accumulator chunk of the block's tile and head: the block's 32 query
    // columns are the same 64 bytes (four 16-byte units, permuted by d mod 8) of each of the
    // 128 head-dim rows; the warp zeroes them with 16 stores of 16 bytes per lane
    uint8_t* chunk = reinterpret_cast<uint8_t*>(dq_acc + dqt_chunk_elems(dq_tile0, h, H));
    const int hf = dq_row0 >> 6, u0 = (dq_row0 & 63) >> 3;
#pragma unroll
    for (int k2 = 0; k2 < 16; ++k2) {
      const int idx = k2 * 32 + lane;
      *reinterpret_cast<uint4*>(chunk + dqt_chunk_byte(hf, idx >> 2, u0 + (idx & 3))) = make_uint4(0, 0, 0, 0);
    }
  }
  if (WITH_D && !PER_TOKEN && maxima && !tail) {
    // dQ boost inputs of (document, query head): max ||dO^_i||, max ||V^_j||, max |K^_jd|
    // over the block's rows, folded into the document maxima (non-negative floats
    // order like their bit patterns)
    const int hk = h / (H / hkv);
    float mv = 0.f, mk = 0.f;
    if (lane < nrows) {
      const int64_t row = r0 + lane;
      mv = v_stats[row * hkv + hk].x;
      mk = k_stats[row * hkv + hk].y;
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      mdo = fmaxf(mdo, __shfl_xor_sync(0xffffffffu, mdo, o2));
      mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o2));
      mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o2));
    }
    if (lane == 0) {
      int* mx3 = reinterpret_cast<int*>(maxima) + ((int64_t)doc * H + h) * 3;
      atomicMax(mx3 + 0, __float_as_int(mdo));
      atomicMax(mx3 + 1, __float_as_int(mv));
      atomicMax(mx3 + 2, __float_as_int(mk));
    }
  }
  if constexpr (!kHold) break;
  }  // work units
  if (kHold) asm volatile("cp.async.wait_group 0;" ::: "memory");   // no copy outlives the block
}

struct PrepExtra {          // backward prep only
  const float* k_stats;
  const float* v_stats;
  int hkv;
  float* maxima;            // [N, H, 3], zeroed by the caller
};

template <int D, bool PT, bool ST, bool WD, bool ROT = false>
cudaError_t launch_q_jobs(QJobs jobs, int njobs, int T, const int32_t* cu, int N, const void* plan, const void* o,
                          float* dvec, void* dq_acc, const PrepExtra& px, cudaStream_t s) {
  const int64_t units = PT ? (T + 31) / 32 : (int64_t)T / 32 + N + 1;
  int64_t warps = 0;
  for (int i = 0; i < 3; ++i) {
    if (i < njobs) warps += units * jobs.j[i].H;
    jobs.j[i].end = warps;
  }
  constexpr int kWarps = QShape<WD, ROT>::kWarps;
  int64_t blocks = (warps + kWarps - 1) / kWarps;
  // the register-held variant walks several units per warp (its next block prefetched);
  // the others keep one unit per warp
  if (!PT && !WD && !ROT) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorInvalidValue;
    const int64_t resident = (int64_t)sms * QShape<WD, ROT>::kMinBlocks;
    if (blocks > resident) blocks = resident;
  }
  if (blocks > 0x7FFFFFFF || blocks < 1) return cudaErrorInvalidValue;
  quantize_kernel<D, PT, ST, WD, ROT><<<(unsigned)blocks, kWarps * 32, 0, s>>>(
      jobs, T, cu, N, static_cast<const int*>(plan), static_cast<const __nv_bfloat16*>(o), dvec,
      static_cast<__half*>(dq_acc), reinterpret_cast<const float2*>(px.k_stats),
      reinterpret_cast<const float2*>(px.v_stats), px.hkv, px.maxima, warps);
  return cudaGetLastError();
}

QJob make_job(const void* x, int H, void* codes, void* scales, float* stats) {
  QJob j;
  j.x = static_cast<const __nv_bfloat16*>(x);
  j.codes = static_cast<uint8_t*>(codes);
  j.scales = static_cast<uint8_t*>(scales);
  j.stats = reinterpret_cast<float2*>(stats);
  j.H = H;
  j.end = 0;
  return j;
}

template <int D, bool PT, bool ST, bool WD, bool ROT = false>
cudaError_t launch_q(const void* x, int T, int H, const int32_t* cu, int N, const void* plan, void* codes,
                     void* scales, float* stats, const void* o, float* dvec, void* dq_acc, const PrepExtra& px,
                     cudaStream_t s) {
  QJobs jobs;
  jobs.j[0] = jobs.j[1] = jobs.j[2] = make_job(x, H, codes, scales, stats);
  return launch_q_jobs<D, PT, ST, WD, ROT>(jobs, 1, T, cu, N, plan, o, dvec, dq_acc, px, s);
}

template <int D>
cudaError_t dispatch(const void* x, int T, int H, const int32_t* cu, int N, const void* plan, int per_token,
                     void* codes, void* scales, float* stats, const void* o, float* dvec, void* dq_acc,
                     const PrepExtra& px, cudaStream_t s) {
  const bool st = stats != nullptr, wd = o != nullptr;
  if (wd) {
    if (per_token) return launch_q<D, true, true, true>(x, T, H, cu, N, plan, codes, scales, stats, o, dvec, dq_acc, px, s);
    return launch_q<D, false, true, true>(x, T, H, cu, N, plan, codes, scales, stats, o, dvec, dq_acc, px, s);
  }
  if (per_token) {
    if (st) return launch_q<D, true, true, false>(x, T, H, cu, N, plan, codes, scales, stats, o, dvec, dq_acc, px, s);
    return launch_q<D, true, false, false>(x, T, H, cu, N, plan, codes, scales, stats, o, dvec, dq_acc, px, s);
  }
  if (st) return launch_q<D, false, true, false>(x, T, H, cu, N, plan, codes, scales, stats, o, dvec, dq_acc, px, s);
  return launch_q<D, false, false, false>(x, T, H, cu, N, plan, codes, scales, stats, o, dvec, dq_acc, px, s);
}

// NVFP4 score operand (step a2, the mixed route; FLAMIA technical review section
// 2, "NVFP4 uses E2M1 codes, a local E4M3 scale for each 16-element group";
// Korean review section 3.2: the scales stay inside one token).  Reading C-7:
// no tensor-level scale; s = E4M3(amax / 6) (IEEE fp32 division, round to
// nearest even, saturating), raised to the smallest subnormal 2^-9 when a
// non-zero group would get a zero scale; code = E2M1(x / s) (IEEE fp32
// division, round to nearest even, saturating to +-6).
// One thread per 16-element group: 32 contiguous bytes in, 8 bytes of packed
// codes (element 2k in the low nibble of byte k) and one scale byte out.
__global__ void __launch_bounds__(256) nvfp4_kernel(const __nv_bfloat16* __restrict__ x, int64_t groups,
                                                    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < groups;
       gi += (int64_t)gridDim.x * blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + gi * 16);
    uint4 w[2] = {__ldg(src), __ldg(src + 1)};
    float f[16];
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&w[j]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 v = __bfloat1622float2(b[k]);
        f[8 * j + 2 * k] = v.x;
        f[8 * j + 2 * k + 1] = v.y;
        amax = fmax3(amax, fabsf(v.x), fabsf(v.y));
      }
    }
    uint8_t sc = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(amax, 6.0f), __NV_SATFINITE, __NV_E4M3);
    if (amax > 0.f && sc == 0) sc = 0x01;   // 2^-9
    const float s = e4m3_to_f32(sc);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float q0 = s > 0.f ? __fdiv_rn(f[2 * k], s) : 0.f;
      const float q1 = s > 0.f ? __fdiv_rn(f[2 * k + 1], s) : 0.f;
      const uint32_t b = (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(q0, q1), __NV_E2M1, cudaRoundNearest);
      packed[k >> 2] |= (b & 0xFFu) << (8 * (k & 3));
    }
    *reinterpret_cast<uint2*>(codes + gi * 8) = make_uint2(packed[0], packed[1]);
    scales[gi] = sc;
  }
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const void* x, int64_t elems, void* codes, void* scales, cudaStream_t s) {
  const int64_t groups = elems / 16;
  if (groups == 0) return cudaSuccess;
  int64_t blocks = (groups + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  nvfp4_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), groups,
                                                static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}

// o / dvec non-null selects the backward-prep variant (stats required); with the
// token-block rule it also zeroes dq_acc (if non-null) and folds the dQ boost
// inputs into maxima (if non-null; k_stats / v_stats of the hkv K/V heads).
// Q, K and V of one call in one launch (token-block or per-token rule; K and V
// with row stats).
cudaError_t launch_quantize_qkv(const void* q, const void* k, const void* v, int T, int hq, int hkv, int D,
                                const int32_t* cu, int N, const void* plan, int per_token, void* qc, void* qs,
                                void* kc, void* ks, float* kst, void* vc, void* vs, float* vst, cudaStream_t s) {
  QJobs jobs;
  jobs.j[0] = make_job(q, hq, qc, qs, nullptr);
  jobs.j[1] = make_job(k, hkv, kc, ks, kst);
  jobs.j[2] = make_job(v, hkv, vc, vs, vst);
  const PrepExtra px{nullptr, nullptr, 1, nullptr};
  if (D == 128 && per_token) return launch_q_jobs<128, true, true, false>(jobs, 3, T, cu, N, plan, nullptr, nullptr, nullptr, px, s);
  if (D == 128) return launch_q_jobs<128, false, true, false>(jobs, 3, T, cu, N, plan, nullptr, nullptr, nullptr, px, s);
  if (D == 64 && per_token) return launch_q_jobs<64, true, true, false>(jobs, 3, T, cu, N, plan, nullptr, nullptr, nullptr, px, s);
  if (D == 64) return launch_q_jobs<64, false, true, false>(jobs, 3, T, cu, N, plan, nullptr, nullptr, nullptr, px, s);
  return cudaErrorInvalidValue;
}

// Hadamard-rotated token-block quantization of Q or K (stats optional).
cudaError_t launch_quantize_rot(const void* x, int T, int H, int D, const int32_t* cu, int N, const void* plan,
                                void* codes, void* scales, float* stats, cudaStream_t s) {
  const PrepExtra px{nullptr, nullptr, 1, nullptr};
  if (D == 128 && stats)
    return launch_q<128, false, true, false, true>(x, T, H, cu, N, plan, codes, scales, stats, nullptr, nullptr,
                                                   nullptr, px, s);
  if (D == 128)
    return launch_q<128, false, false, false, true>(x, T, H, cu, N, plan, codes, scales, nullptr, nullptr, nullptr,
                                                    nullptr, px, s);
  if (D == 64 && stats)
    return launch_q<64, false, true, false, true>(x, T, H, cu, N, plan, codes, scales, stats, nullptr, nullptr,
                                                  nullptr, px, s);
  if (D == 64)
    return launch_q<64, false, false, false, true>(x, T, H, cu, N, plan, codes, scales, nullptr, nullptr, nullptr,
                                                   nullptr, px, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantize(const void* x, int T, int H, int D, const int32_t* cu, int N, const void* plan,
                            int per_token, void* codes, void* scales, float* stats, const void* o, float* dvec,
                            void* dq_acc, cudaStream_t s, const float* k_stats, const float* v_stats, int hkv,
                            float* maxima) {
  const PrepExtra px{k_stats, v_stats, hkv, maxima};
  if (D == 128) return dispatch<128>(x, T, H, cu, N, plan, per_token, codes, scales, stats, o, dvec, dq_acc, px, s);
  if (D == 64) return dispatch<64>(x, T, H, cu, N, plan, per_token, codes, scales, stats, o, dvec, dq_acc, px, s);
  return cudaErrorInvalidValue;
}

}  // namespace flamia
