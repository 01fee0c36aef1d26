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
#include <cuda_fp16.h>
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
  // Launched itself as a programmatic dependent of the preceding kernel (a
  // decode still reading the cache, say): the new rows and their slots, this
  // call's own inputs, are read and quantized at once; the cache is written
  // only after that grid has completed.
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
  const uint4 rope = lane < 8 ? __ldg(src + 64 + lane) : make_uint4(0u, 0u, 0u, 0u);
  grid_dependency_wait();
  uint8_t* row = cache + slot * kRowBytes;
  *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(row + kScaleOff + 4 * (lane >> 3)) = scale;
  if (lane < 8) *reinterpret_cast<uint4*>(row + kRopeOff + 16 * lane) = rope;
}

__global__ void translate_kernel(const int32_t* __restrict__ indices, const int32_t* __restrict__ block_table,
                                 const int32_t* __restrict__ req_id, int32_t* __restrict__ slots, int64_t n, int K,
                                 int R, int MB, int64_t NB) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t t = i / K;
  slots[i] = translate_slot(__ldg(indices + i), __ldg(req_id + t), block_table, R, MB, NB);
}

// Index translation with a prefill workspace (the HAS_PREFILL form of
// vLLM flashmla_sparse.py _convert_req_index_to_global_index_kernel): a token
// with prefill_req_id < 0 is a decode token (translate_slot); a prefill
// token's index becomes workspace_starts[prefill_req_id] + index, -1 when the
// index is negative, its block id is outside [0, MB), or prefill_req_id has
// no start (prefill_req_id >= P).
__global__ void translate_ws_kernel(const int32_t* __restrict__ indices, const int32_t* __restrict__ block_table,
                                    const int32_t* __restrict__ req_id, const int32_t* __restrict__ prefill_req_id,
                                    const int32_t* __restrict__ starts, int P, int32_t* __restrict__ out, int64_t n,
                                    int K, int R, int MB, int64_t NB) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t t = i / K;
  const int32_t idx = __ldg(indices + i);
  const int32_t pr = __ldg(prefill_req_id + t);
  int32_t v;
  if (pr < 0)
    v = translate_slot(idx, __ldg(req_id + t), block_table, R, MB, NB);
  else if (idx < 0 || (idx >> 6) >= MB || pr >= P)
    v = -1;
  else
    v = __ldg(starts + pr) + idx;
  out[i] = v;
}

// Gather and up-convert of the separate-mode FP8 prefill
// (cp_gather_and_upconvert_fp8_kv_cache in vLLM flashmla_sparse.py
// _forward_fp8_kv_separate_prefill_decode): position p < seq_lens[r] of
// request r (its slot through the block table) becomes bf16 row
// starts[r] + p of the workspace: NoPE value c = e4m3(code c) * scale[c / 128]
// as a float32 product rounded to bf16 (nearest, ties to even), RoPE copied
// as stored; an invalid slot gives a zero row, a destination outside [0, N)
// is skipped.  One warp per row, warps striding over each request's rows:
// lane l converts codes 16 l .. 16 l + 15 (scale group l / 8) and lanes
// 1..8 copy the RoPE chunks.
__global__ void __launch_bounds__(256) gather_upconvert_kernel(const uint8_t* __restrict__ cache, int64_t NB,
                                                               const int32_t* __restrict__ block_table, int R, int MB,
                                                               const int32_t* __restrict__ seq_lens,
                                                               const int32_t* __restrict__ starts,
                                                               uint4* __restrict__ ws, int64_t N) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int r = 0; r < R; ++r) {
    const int32_t len = __ldg(seq_lens + r), start = __ldg(starts + r);
    for (int64_t pos = warp0; pos < len; pos += n_warps) {
      const int64_t dst = (int64_t)start + pos;
      if (dst < 0 || dst >= N) continue;
      const int32_t slot = translate_slot((int32_t)pos, r, block_table, R, MB, NB);
      uint4* out = ws + dst * (kDqk * 2 / 16);  // 72 chunks of 16 bytes per bf16 row
      if (slot < 0) {
        out[2 * lane] = make_uint4(0, 0, 0, 0);
        out[2 * lane + 1] = make_uint4(0, 0, 0, 0);
        if (lane < 8) out[64 + lane] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint8_t* row = cache + (int64_t)slot * kRowBytes;
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(row) + lane);
      const uint4 tail = lane < 9 ? __ldg(reinterpret_cast<const uint4*>(row + kScaleOff) + lane) : make_uint4(0, 0, 0, 0);
      // lane 0's tail chunk holds the row's four scales; lane l uses scale l / 8
      const uint32_t s0 = __shfl_sync(0xffffffffu, tail.x, 0), s1 = __shfl_sync(0xffffffffu, tail.y, 0);
      const uint32_t s2 = __shfl_sync(0xffffffffu, tail.z, 0), s3 = __shfl_sync(0xffffffffu, tail.w, 0);
      const int g = lane >> 3;
      const float sc = __uint_as_float(g == 0 ? s0 : g == 1 ? s1 : g == 2 ? s2 : s3);
      const uint32_t w[4] = {c.x, c.y, c.z, c.w};
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t f16;
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16) : "h"((uint16_t)(w[k] >> (16 * h))));  // exact
          const float lo = __half2float(__ushort_as_half((uint16_t)(f16 & 0xFFFFu))) * sc;
          const float hi = __half2float(__ushort_as_half((uint16_t)(f16 >> 16))) * sc;
          o[2 * k + h] = pack_bf16x2(lo, hi);
        }
      }
      out[2 * lane] = make_uint4(o[0], o[1], o[2], o[3]);
      out[2 * lane + 1] = make_uint4(o[4], o[5], o[6], o[7]);
      if (lane >= 1 && lane < 9) out[64 + lane - 1] = tail;
    }
  }
}

}  // namespace

cudaError_t launch_translate_ws(const int32_t* indices, const int32_t* block_table, const int32_t* req_id,
                                const int32_t* prefill_req_id, const int32_t* starts, int P, int32_t* out, int T,
                                int K, int R, int MB, int64_t NB, cudaStream_t stream) {
  if (T <= 0 || K <= 0) return cudaSuccess;
  const int64_t n = (int64_t)T * K;
  translate_ws_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(indices, block_table, req_id, prefill_req_id,
                                                                       starts, P, out, n, K, R, MB, NB);
  return cudaGetLastError();
}

cudaError_t launch_gather_upconvert(const uint8_t* cache, int64_t NB, const int32_t* block_table, int R, int MB,
                                    const int32_t* seq_lens, const int32_t* starts, void* ws, int64_t N,
                                    int num_sms, cudaStream_t stream) {
  if (R <= 0 || N <= 0) return cudaSuccess;
  gather_upconvert_kernel<<<(unsigned)(num_sms * 8), 256, 0, stream>>>(cache, NB, block_table, R, MB, seq_lens,
                                                                       starts, static_cast<uint4*>(ws), N);
  return cudaGetLastError();
}

cudaError_t launch_quantize_store(const void* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T, int64_t NB,
                                  cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = ((int64_t)T * 32 + threads - 1) / threads;
  // a programmatic dependent of the preceding kernel on the stream: its launch
  // overlaps that kernel's tail, and the kernel waits for it before any access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_store_kernel, static_cast<const uint4*>(kv_new), slot_mapping,
                                     cache, T, NB);
  if (e != cudaSuccess) return e;
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
