// Quantize-and-store of new latent tokens into the 656-byte FP8 cache and
// the standalone logical -> physical index translation.
//
// Quantize-and-store follows the cache write of FlashMLASparseImpl.forward in
// vLLM flashmla_sparse.py (concat_and_cache_mla with kv_cache_dtype
// "fp8_ds_mla"): each token's 512 NoPE values are quantized per group of 128
// with scale = amax / 448 (IEEE float32 division), codes = float32(x / scale)
// rounded to nearest-even e4m3 with saturation; the 4 scales and the 64
// bfloat16 RoPE values are stored verbatim.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "smla_common.cuh"
#include "smla_kernels.h"

namespace smla {

namespace {

__device__ __forceinline__ uint16_t e4m3x2_rn_satfinite(float lo, float hi) {
  uint16_t r;
  // first source operand is placed in the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xFFFF0000u);
}

// One warp per token.  Lane l owns NoPE columns [16l, 16l+16), i.e. group
// l / 8; lanes 8g..8g+7 reduce the group's amax with shuffles.
__global__ void __launch_bounds__(256) quantize_store_kernel(const uint4* __restrict__ kv_new,
                                                             const int64_t* __restrict__ slot_mapping,
                                                             uint8_t* __restrict__ cache, int T, int64_t NB) {
  // a decode launched behind this grid as its programmatic dependent may start
  // its prologue now; it waits for this grid before it reads the cache
  grid_launch_dependents();
  const int token = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= T) return;
  const int64_t slot = slot_mapping[token];
  if (slot < 0 || slot >= NB * kBlock) return;  // skipped token
  const uint4* src = kv_new + (int64_t)token * (kDqk * 2 / 16);  // 72 chunks of 16 bytes per row
  const uint4 a = __ldg(src + 2 * lane);
  const uint4 b = __ldg(src + 2 * lane + 1);
  float x[16];
  bf16x2_to_f32(a.x, x[0], x[1]);
  bf16x2_to_f32(a.y, x[2], x[3]);
  bf16x2_to_f32(a.z, x[4], x[5]);
  bf16x2_to_f32(a.w, x[6], x[7]);
  bf16x2_to_f32(b.x, x[8], x[9]);
  bf16x2_to_f32(b.y, x[10], x[11]);
  bf16x2_to_f32(b.z, x[12], x[13]);
  bf16x2_to_f32(b.w, x[14], x[15]);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const float scale = __fdiv_rn(amax, 448.0f);
  uint32_t codes[4] = {0u, 0u, 0u, 0u};
  if (scale != 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = e4m3x2_rn_satfinite(__fdiv_rn(x[4 * i], scale), __fdiv_rn(x[4 * i + 1], scale));
      const uint16_t hi = e4m3x2_rn_satfinite(__fdiv_rn(x[4 * i + 2], scale), __fdiv_rn(x[4 * i + 3], scale));
      codes[i] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
  }
  uint8_t* row = cache + slot * kRowBytes;
  *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(row + kScaleOff + 4 * (lane >> 3)) = scale;
  if (lane < 8) *reinterpret_cast<uint4*>(row + kRopeOff + 16 * lane) = __ldg(src + 64 + lane);
}

__global__ void translate_kernel(const int32_t* __restrict__ indices, const int32_t* __restrict__ block_table,
                                 const int32_t* __restrict__ req_id, int32_t* __restrict__ slots, int64_t n, int K,
                                 int R, int MB, int64_t NB) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t t = i / K;
  slots[i] = translate_slot(__ldg(indices + i), __ldg(req_id + t), block_table, R, MB, NB);
}

}  // namespace

cudaError_t launch_quantize_store(const void* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T, int64_t NB,
                                  cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = ((int64_t)T * 32 + threads - 1) / threads;
  quantize_store_kernel<<<(unsigned)blocks, threads, 0, stream>>>(static_cast<const uint4*>(kv_new), slot_mapping,
                                                                  cache, T, NB);
  return cudaGetLastError();
}

cudaError_t launch_translate(const int32_t* indices, const int32_t* block_table, const int32_t* req_id,
                             int32_t* slots, int T, int K, int R, int MB, int64_t NB, cudaStream_t stream) {
  if (T <= 0 || K <= 0) return cudaSuccess;
  const int64_t n = (int64_t)T * K;
  translate_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(indices, block_table, req_id, slots, n, K, R, MB,
                                                                    NB);
  return cudaGetLastError();
}

}  // namespace smla
