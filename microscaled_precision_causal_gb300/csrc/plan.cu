// Work-list builder: Algorithm 2 of the FLAMIA technical review ("Document-
// local work list and launch", steps 01-06), run on the GPU once per
// microbatch with no host synchronisation (review section 6, "GPU list
// construction avoids host synchronization").
//
// One CTA of 1024 threads:
//   1. validate cu_seqlens (cu[0] = 0, non-decreasing, cu[N] <= T);
//   2. per-document counts of 32-token blocks, 128-token tiles and 256-query
//      items, exclusive prefix sums over documents;
//   3. forward items (cost = visible key tiles summed over the item's query
//      tiles) and backward key-tile items (cost = query tiles that see the
//      key tile), each sorted by decreasing cost with ties in document, then
//      tile order: a bitonic sort of 64-bit keys (cost descending, index).
// "Visible" follows the call's (left, right) window (causal: keys up to the
// query; noncausal: the whole document).  The costs only order the work; the
// item sets are the same for every window.
#include "common.cuh"

namespace flamia {

namespace {

constexpr int kThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the exclusive
// prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

// Bitonic sort of n <= blockDim.x keys (n a power of two): one key per thread in a
// register; partners closer than a warp are exchanged with shuffles, the others
// through shared memory.  Ascending.
__device__ void bitonic_sort_regs(unsigned long long* keys, int n) {
  const int i = threadIdx.x;
  // only the warps that hold keys sort (their rounds meet on named barrier 1, counted in
  // whole warps); the others wait at the block barrier at the end
  const int nlive = (n + 31) & ~31;
  if (i < nlive) {
    unsigned long long a = i < n ? keys[i] : ~0ull;
    for (int k = 2; k <= n; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        unsigned long long b;
        if (j >= 32) {
          asm volatile("bar.sync 1, %0;" ::"r"(nlive) : "memory");   // every read of the previous round done
          keys[i] = a;
          asm volatile("bar.sync 1, %0;" ::"r"(nlive) : "memory");
          b = keys[i ^ j];
        } else {
          b = __shfl_xor_sync(0xffffffffu, a, j);
        }
        const bool up = (i & k) == 0, lower = (i & j) == 0;
        a = (lower == up) ? (a < b ? a : b) : (a < b ? b : a);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(nlive) : "memory");
    if (i < n) keys[i] = a;
  }
  __syncthreads();
}

__device__ void bitonic_sort(unsigned long long* keys, int n) {  // n is a power of two
  if (n <= (int)blockDim.x) {
    bitonic_sort_regs(keys, n);
    return;
  }
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], b = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

constexpr int kSmemKeys = 4096;   // sorts of up to this many keys run in shared memory
constexpr int kMirror = 1024;     // up to this many documents, cu and the prefix arrays are read from
                                  // shared-memory copies (each item's document is a binary search)

__global__ void __launch_bounds__(kThreads) plan_kernel(const int32_t* __restrict__ cu, int N, int T, Window win,
                                                        int* __restrict__ plan_words) {
  __shared__ unsigned long long smem_keys[kSmemKeys];
  __shared__ int warp_sums[32];
  __shared__ int s_bad;
  __shared__ int s_carry[3];
  __shared__ int s_cu[kMirror + 1], s_tp[kMirror + 1], s_ip[kMirror + 1];
  const bool mirror = N <= kMirror;
  PlanView pv = plan_view(plan_words, T, N);
  int* blk_prefix = const_cast<int*>(pv.blk_prefix);
  int* tile_prefix = const_cast<int*>(pv.tile_prefix);
  int* item_prefix = const_cast<int*>(pv.item_prefix);
  int4* fwd = const_cast<int4*>(pv.fwd_items);
  int4* bwd = const_cast<int4*>(pv.bwd_items);
  int2* bwd_span = const_cast<int2*>(pv.bwd_span);
  int2* fwd_span = const_cast<int2*>(pv.fwd_span);
  const int cap = (int)plan_capacity(T, N);

  if (threadIdx.x == 0) {
    s_bad = 0;
    s_carry[0] = s_carry[1] = s_carry[2] = 0;
  }
  __syncthreads();
  // 1. validation
  for (int n = threadIdx.x; n < N; n += kThreads) {
    const int a = cu[n], b = cu[n + 1];
    if (b < a || (n == 0 && a != 0) || (n == N - 1 && b > T)) atomicOr(&s_bad, 1);
    if (mirror) {
      s_cu[n] = a;
      if (n == N - 1) s_cu[N] = b;
    }
  }
  __syncthreads();
  const int bad = s_bad;
  const int32_t* cuv = mirror ? s_cu : cu;   // cu, from shared memory when it fits
  // 2. prefix counts (chunks of kThreads documents)
  for (int base = 0; base < N; base += kThreads) {
    const int n = base + threadIdx.x;
    int L = 0;
    if (!bad && n < N) L = cuv[n + 1] - cuv[n];
    const int nb = (L + kBlock - 1) / kBlock, nt = (L + kTile - 1) / kTile,
              ni = (L + kTile * kItemTiles - 1) / (kTile * kItemTiles);
    int tot;
    const int pb = block_exclusive_scan(nb, warp_sums, &tot);
    const int cb = s_carry[0];
    __syncthreads();
    if (threadIdx.x == 0) s_carry[0] = cb + tot;
    const int pt = block_exclusive_scan(nt, warp_sums, &tot);
    const int ct = s_carry[1];
    __syncthreads();
    if (threadIdx.x == 0) s_carry[1] = ct + tot;
    const int pi = block_exclusive_scan(ni, warp_sums, &tot);
    const int ci = s_carry[2];
    __syncthreads();
    if (threadIdx.x == 0) s_carry[2] = ci + tot;
    if (n < N) {
      blk_prefix[n] = cb + pb;
      tile_prefix[n] = ct + pt;
      item_prefix[n] = ci + pi;
      if (mirror) {
        s_tp[n] = ct + pt;
        s_ip[n] = ci + pi;
      }
    }
    __syncthreads();
  }
  const int nblk = s_carry[0], ntile = s_carry[1], nitem = s_carry[2];
  if (threadIdx.x == 0) {
    blk_prefix[N] = nblk;
    tile_prefix[N] = ntile;
    item_prefix[N] = nitem;
    if (mirror) {
      s_tp[N] = ntile;
      s_ip[N] = nitem;
    }
  }
  __syncthreads();
  const int* tpv = mirror ? s_tp : tile_prefix;   // the prefix arrays, from shared memory when they fit
  const int* ipv = mirror ? s_ip : item_prefix;
  const bool over = ntile > cap || nitem > cap;
  if (threadIdx.x == 0) {
    plan_words[kPlanStatus] = (bad ? FLAMIA_DEV_BAD_CU_SEQLENS : 0) | (over ? FLAMIA_DEV_CAPACITY : 0);
    plan_words[kPlanNumSeqs] = N;
    plan_words[kPlanTotal] = T;
    plan_words[kPlanValid] = bad ? 0 : (N > 0 ? cuv[N] : 0);
    plan_words[kPlanBlocks] = bad ? 0 : nblk;
    plan_words[kPlanTiles] = (bad || over) ? 0 : ntile;
    plan_words[kPlanFwdItems] = (bad || over) ? 0 : nitem;
    plan_words[kPlanBwdItems] = (bad || over) ? 0 : ntile;
    plan_words[kPlanCapacity] = cap;
    plan_words[kPlanWindowLeft] = win.left;
    plan_words[kPlanWindowRight] = win.right;
    plan_words[kPlanFwdTicket] = 0;
  }
  if (bad || over) return;
  const unsigned long long kPad = ~0ull;
  const unsigned kCostMax = 0x7FFFFFFFu;

  // 3a. forward items
  {
    const int n2 = (int)pow2_ceil(nitem > 0 ? nitem : 1);
    unsigned long long* keys = n2 <= kSmemKeys ? smem_keys : pv.sort_keys;
    for (int i = threadIdx.x; i < n2; i += kThreads) {
      unsigned long long key = kPad;
      if (i < nitem) {
        const int doc = upper_doc(ipv, N, i);
        const int nt = tpv[doc + 1] - tpv[doc];
        const int t0 = (i - ipv[doc]) * kItemTiles;
        const int cnt = min(kItemTiles, nt - t0);
        int cost = 0;
        for (int t = t0; t < t0 + cnt; ++t) cost += win_khi(t, nt, win) - win_klo(t, win) + 1;
        key = ((unsigned long long)(kCostMax - (unsigned)cost) << 32) | (unsigned)i;
      }
      keys[i] = key;
    }
    __syncthreads();
    bitonic_sort(keys, n2);
    for (int r = threadIdx.x; r < nitem; r += kThreads) {
      const int i = (int)(keys[r] & 0xFFFFFFFFull);
      const int doc = upper_doc(ipv, N, i);
      const int nt = tpv[doc + 1] - tpv[doc];
      const int t0 = (i - ipv[doc]) * kItemTiles;
      const int cnt = min(kItemTiles, nt - t0);
      fwd[r] = make_int4(doc, t0, cnt, (int)(kCostMax - (unsigned)(keys[r] >> 32)));
      fwd_span[r] = make_int2(cuv[doc], cuv[doc + 1] - cuv[doc]);
    }
    __syncthreads();
  }
  // 3b. backward key-tile items
  {
    const int n2 = (int)pow2_ceil(ntile > 0 ? ntile : 1);
    unsigned long long* keys = n2 <= kSmemKeys ? smem_keys : pv.sort_keys;
    for (int i = threadIdx.x; i < n2; i += kThreads) {
      unsigned long long key = kPad;
      if (i < ntile) {
        const int doc = upper_doc(tpv, N, i);
        const int nt = tpv[doc + 1] - tpv[doc];
        const int u = i - tpv[doc];
        const int cost = win_thi(u, nt, win) - win_tlo(u, win) + 1;
        key = ((unsigned long long)(kCostMax - (unsigned)cost) << 32) | (unsigned)i;
      }
      keys[i] = key;
    }
    __syncthreads();
    bitonic_sort(keys, n2);
    for (int r = threadIdx.x; r < ntile; r += kThreads) {
      const int i = (int)(keys[r] & 0xFFFFFFFFull);
      const int doc = upper_doc(tpv, N, i);
      bwd[r] = make_int4(doc, i - tpv[doc], (int)(kCostMax - (unsigned)(keys[r] >> 32)), 0);
      bwd_span[r] = make_int2(cuv[doc], cuv[doc + 1] - cuv[doc]);
    }
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* cu, int N, int T, Window win, void* plan, cudaStream_t s) {
  plan_kernel<<<1, kThreads, 0, s>>>(cu, N, T, win, static_cast<int*>(plan));
  return cudaGetLastError();
}

}  // namespace flamia
