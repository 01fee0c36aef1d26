// Shared device-side definitions: the 656-byte cache row format, the logical
// -> physical index translation, and the shared-memory operand layouts used by
// the tensor-core kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace smla {

// "FP8 with scale" row (vLLM flashmla_sparse.py, module docstring): bytes
// 0..511 hold 512 float8_e4m3 NoPE values, bytes 512..527 four float32 scales
// (one per 128 values), bytes 528..655 64 bfloat16 RoPE values.
constexpr int kRowBytes = 656;
constexpr int kNope = 512;
constexpr int kRope = 64;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kGroup = 128;
constexpr int kScaleOff = 512;
constexpr int kRopeOff = 528;
constexpr int kBlock = 64;  // paged block size (tokens per block)

// Status words written by kernels into the device status slot.
enum : int { kDevOk = 0, kDevWaitTimeout = 1 };

// Logical top-k index -> physical cache slot, following the Triton kernel
// triton_convert_req_index_to_global_index of flashmla_sparse.py:
//   slot = block_table[req, idx / 64] * 64 + idx % 64,
// -1 when idx < 0 or the block id is outside [0, MB).  In addition the slot
// is -1 when the request id is outside [0, R) or the physical block is
// outside [0, NB), so no later step can address memory outside the cache.
__device__ __forceinline__ int32_t translate_slot(int32_t idx, int32_t req, const int32_t* __restrict__ block_table,
                                                  int R, int MB, int64_t NB) {
  if (idx < 0 || req < 0 || req >= R) return -1;
  const int32_t b = idx >> 6;
  if (b >= MB) return -1;
  const int32_t p = __ldg(block_table + (int64_t)req * MB + b);
  if (p < 0 || (int64_t)p >= NB) return -1;
  return p * kBlock + (idx & 63);
}

// Byte offset of element (row r, column c) of a bf16 operand tile stored
// K-major with the 128-byte swizzle: 64-column panels of `rows` x 128 bytes,
// 8-row groups of 1024 bytes, 16-byte chunks XOR-permuted by (row % 8).
__host__ __device__ __forceinline__ uint32_t sw128_offset(int rows, int r, int c) {
  const int panel = c >> 6;
  const int chunk = (c & 63) >> 3;
  return (uint32_t)(panel * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ (r & 7)) << 4) + ((c & 7) << 1));
}
// Offset of 16-byte chunk `ch` (8 bf16 values, columns 8ch..8ch+7) of row r.
__host__ __device__ __forceinline__ uint32_t sw128_chunk(int rows, int r, int ch) {
  return (uint32_t)((ch >> 3) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// P^T operand (K = kv row j, N = head h), MN-major without swizzle: 8x8 core
// matrices (8 rows j of 16 bytes = 8 heads), head blocks 128 bytes apart,
// row blocks (HG/8)*128 bytes apart.
template <int HG>
__host__ __device__ __forceinline__ uint32_t pt_offset(int j, int h) {
  return (uint32_t)((j >> 3) * (HG / 8) * 128 + (h >> 3) * 128 + (j & 7) * 16 + (h & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  // first source operand goes to the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace smla
