// Host helper: TMA tensor-map encoding through the driver entry point (no
// link-time dependency on libcuda).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace flamia {

// Per-device one-time kernel set-up: the dynamic shared-memory limit and the
// register count the launch relies on are settled on the first call on each
// device, so that later calls -- including calls captured into a CUDA graph --
// only launch.
template <auto Kernel>
inline cudaError_t prepare_kernel(int smem_bytes, int* num_regs = nullptr) {
  static std::atomic<unsigned long long> ready{0};
  static int regs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(ready.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, Kernel);
    if (e != cudaSuccess) return e;
    regs[dev & 63] = fa.numRegs;
    ready.fetch_or(bit, std::memory_order_release);
  }
  if (num_regs) *num_regs = regs[dev & 63];
  return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

inline CUtensorMapSwizzle swizzle_for_row_bytes(uint32_t row_bytes) {
  return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// 8-bit tensor [dim2][dim1][dim0] (dim0 contiguous) with byte strides
// stride1 (between dim1 entries) and stride2; box (box0, 1, box2).
inline bool make_tmap_u8_3d(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                            uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box2) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {dim0, dim1, dim2};
  cuuint64_t gstr[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, 1, box2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), gdim, gstr, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for_row_bytes(box0), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor [dim2][dim1][dim0] (dim0 contiguous) with byte strides stride1 and stride2;
// box (box0, 1, box2), the swizzle of a box0 * 2-byte row.
inline bool make_tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t dim0, uint64_t dim1, uint64_t dim2,
                              uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box2) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t gdim[3] = {dim0, dim1, dim2};
  cuuint64_t gstr[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, 1, box2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstr, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for_row_bytes(box0 * 2), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace flamia
