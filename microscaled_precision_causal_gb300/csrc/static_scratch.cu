// flamia_bwd_static_scratch: the backward pass for callers that cannot
// allocate device memory.
//
// Some callers own no allocator at the point where they run the backward: a
// plugin whose host framework hands it only its input and output buffers, or
// a latency-critical loop that must not pay cudaMalloc's device-wide
// synchronisation.  This entry point takes the same arguments as flamia_bwd
// except the workspace; its scratch (dO codes, scale bytes and row stats, D,
// the dQ boosts and the fp16 dQ accumulator) lives in the file-scope device
// array below, which every GPU that loads the library holds until the process
// exits.
//
// Set-up: the first call on each device (with that device current) resolves
// the array's device address with cudaGetSymbolAddress and caches it.  The cached address belongs to
// the device's current context: after cudaDeviceReset (or anything else that
// destroys and re-creates the primary context) the array may move, so a
// process that resets a device must not call this entry point on it again.  The call itself allocates
// nothing (no cudaMalloc / cudaFree, no allocating library routine).
//
// Sharing: every call uses the same array, which keeps the previous call's
// contents.  The parts that must start at zero (the fp16 dQ accumulator) are
// cleared by the call itself; the rest is overwritten before it is read.
// Calls whose GPU work overlaps (different streams, or different threads on
// one device without ordering) race on the array and produce wrong results.
#include <atomic>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = FLAMIA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_bwd_scratch[kScratchBytes];

std::atomic<void*> g_scratch_ptr[kMaxDevices];

}  // namespace

extern "C" int flamia_bwd_static_scratch(const flamia_qtensor* q, const flamia_qtensor* k, const flamia_qtensor* v,
                                         const void* out_bf16, const float* lse, const void* dout_bf16,
                                         const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens, int hq,
                                         int hkv, int head_dim, int causal, float softmax_scale,
                                         const flamia_options* opt, const void* plan, void* dq_bf16, void* dk_bf16,
                                         void* dv_bf16, void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLAMIA_ERR_CUDA;
  void* ptr = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || !ptr) return FLAMIA_ERR_CUDA;
    g_scratch_ptr[dev].store(ptr, std::memory_order_release);
  }
  // flamia_bwd checks every argument first and the workspace size last, so a bad
  // argument returns the same code as there, and only a problem larger than the
  // array returns FLAMIA_ERR_WORKSPACE (before anything is launched).
  return flamia_bwd(q, k, v, out_bf16, lse, dout_bf16, cu_seqlens, num_seqs, total_tokens, hq, hkv, head_dim, causal,
                    softmax_scale, opt, plan, dq_bf16, dk_bf16, dv_bf16, ptr, kScratchBytes, stream);
}
