// The NVFP4 cache: 352 bytes per token (vLLM PR #59342, "Purpose": the
// nvfp4_ds_mla cache holds 352 bytes per token against the FP8 one's 576).
// The pages give the size, not the layout; this library uses
//   bytes   0..255  the 512 NoPE values as E2M1 codes (OCP MX FP4), value 2i in
//                   the low nibble of byte i and 2i + 1 in the high nibble;
//   bytes 256..287  one E4M3 scale per block of 16 NoPE values;
//   bytes 288..351  the 64 RoPE values as E4M3.
// A row dequantizes alone: value c = e2m1(code c) * e4m3(scale c / 16), RoPE
// r = e4m3(byte 288 + r).  Every such value has at most 6 significant bits (2
// of the code times 4 of the scale) and lies in [2^-10, 2688] or is 0, so it
// is exact in f16 and in bf16.
//
// Quantize-and-store: per block, s = e4m3(amax / 6) and code = e2m1(x / s),
// float32 divisions, nearest-even with saturation on both grids (a block whose
// scale is 0 stores code 0); RoPE = e4m3(x).
//
// Decode reads the rows it attends to as stored and dequantizes them exactly.
// Below 128 heads the attention kernel's converter warps do it (smla_attn.cu).
// At 128 heads a staging kernel (here) writes each token's top-k rows as bf16
// rows of a workspace, translated through the block table as for the FP8
// cache, and the 128-head bf16 kernel runs over them.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "smla_common.cuh"
#include "smla_kernels.h"

namespace smla {

namespace {

constexpr int kNvRowBytes = 352;
constexpr int kNvScaleOff = 256;
constexpr int kNvRopeOff = 288;

// Eight floats -> eight E2M1 codes, value 2i in the low nibble of byte i
// (nearest-even, saturating to +-6).
__device__ __forceinline__ uint32_t e2m1x8_rn_satfinite(const float (&x)[8]) {
  uint32_t r;
  // the first source operand of each conversion goes to the high nibble
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return r;
}

// Two floats -> two E4M3 codes (lo in the low byte; nearest-even, saturating).
__device__ __forceinline__ uint16_t e4m3x2_rn_satfinite(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ void e4m3x2_to_f32(uint16_t codes, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  lo = __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((uint16_t)(h2 >> 16)));
}

// One byte of two E2M1 codes (low nibble first) -> two floats (exact).
__device__ __forceinline__ void e2m1x2_to_f32(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n .reg .b8 c, z;\n mov.b16 {c, z}, %1;\n cvt.rn.f16x2.e2m1x2 %0, c;\n}"
      : "=r"(h2)
      : "h"((uint16_t)(byte & 0xFFu)));
  lo = __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
  hi = __half2float(__ushort_as_half((uint16_t)(h2 >> 16)));
}

// One warp per token; lane l owns NoPE block l (values 16 l .. 16 l + 15) and
// RoPE values 2 l, 2 l + 1.
__global__ void __launch_bounds__(256) nvfp4_store_kernel(const uint4* __restrict__ kv_new,
                                                          const int64_t* __restrict__ slot_mapping,
                                                          uint8_t* __restrict__ cache, int T, int64_t NB) {
  const int token = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= T) return;
  const int64_t slot = slot_mapping[token];
  if (slot < 0 || slot >= NB * kBlock) return;  // skipped token
  const uint4* src = kv_new + (int64_t)token * (kDqk * 2 / 16);  // 72 chunks of 16 bytes per row
  const uint4 a = __ldg(src + 2 * lane), b = __ldg(src + 2 * lane + 1);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint8_t sb = (uint8_t)(e4m3x2_rn_satfinite(__fdiv_rn(amax, 6.0f), 0.f) & 0xFFu);
  float s, unused;
  e4m3x2_to_f32(sb, s, unused);
  uint32_t codes[2] = {0u, 0u};
  if (s != 0.f) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(x[8 * h + i], s);
      codes[h] = e2m1x8_rn_satfinite(y);
    }
  }
  uint8_t* row = cache + slot * kNvRowBytes;
  *reinterpret_cast<uint2*>(row + 8 * lane) = make_uint2(codes[0], codes[1]);
  row[kNvScaleOff + lane] = sb;
  const uint32_t rw = __ldg(reinterpret_cast<const uint32_t*>(src + 64) + lane);  // RoPE values 2 l, 2 l + 1
  *reinterpret_cast<uint16_t*>(row + kNvRopeOff + 2 * lane) =
      e4m3x2_rn_satfinite(__uint_as_float(rw << 16), __uint_as_float(rw & 0xFFFF0000u));
}

// Decode staging: one warp per (token, top-k position).  The slot comes from
// the block table as for the FP8 cache; a valid row becomes bf16 row
// t * K + k of `rows` and rows_idx[t * K + k] = t * K + k, an invalid one
// gets rows_idx = -1 and no row.  Lane l dequantizes NoPE block l and RoPE
// values 2 l, 2 l + 1.
__global__ void __launch_bounds__(256) nvfp4_stage_kernel(const uint8_t* __restrict__ cache, int64_t NB,
                                                          const int32_t* __restrict__ indices,
                                                          const int32_t* __restrict__ block_table,
                                                          const int32_t* __restrict__ req_id, int R, int MB, int K,
                                                          int64_t n, int32_t* __restrict__ rows_idx,
                                                          uint4* __restrict__ rows) {
  const int64_t i = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const int64_t t = i / K;
  const int32_t slot = translate_slot(__ldg(indices + i), __ldg(req_id + t), block_table, R, MB, NB);
  if (lane == 0) rows_idx[i] = slot < 0 ? -1 : (int32_t)i;
  if (slot < 0) return;
  const uint8_t* row = cache + (int64_t)slot * kNvRowBytes;
  const uint2 c = __ldg(reinterpret_cast<const uint2*>(row) + lane);
  float s, unused;
  e4m3x2_to_f32((uint16_t)__ldg(row + kNvScaleOff + lane), s, unused);
  const uint32_t cw[2] = {c.x, c.y};
  uint32_t o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float lo, hi;
    e2m1x2_to_f32(cw[k >> 2] >> (8 * (k & 3)), lo, hi);
    o[k] = pack_bf16x2(lo * s, hi * s);  // exact products, exact in bf16
  }
  uint4* out = rows + i * (kDqk * 2 / 16);  // 72 chunks of 16 bytes per bf16 row
  out[2 * lane] = make_uint4(o[0], o[1], o[2], o[3]);
  out[2 * lane + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  float r0, r1;
  e4m3x2_to_f32(__ldg(reinterpret_cast<const uint16_t*>(row + kNvRopeOff) + lane), r0, r1);
  reinterpret_cast<uint32_t*>(out + 64)[lane] = pack_bf16x2(r0, r1);
}

}  // namespace

cudaError_t launch_nvfp4_store(const void* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T, int64_t NB,
                               cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int64_t blocks = ((int64_t)T * 32 + 255) / 256;
  nvfp4_store_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint4*>(kv_new), slot_mapping, cache, T,
                                                           NB);
  return cudaGetLastError();
}

size_t nvfp4_stage_bytes(int T, int K) {
  const size_t n = (size_t)T * (size_t)K;
  return ((n * 4 + 255) / 256) * 256 + n * kDqk * 2;
}

cudaError_t launch_nvfp4_stage(const uint8_t* cache, int64_t NB, const int32_t* indices, const int32_t* block_table,
                               const int32_t* req_id, int T, int K, int R, int MB, void* stage,
                               cudaStream_t stream) {
  const int64_t n = (int64_t)T * K;
  if (n <= 0) return cudaSuccess;
  int32_t* rows_idx = static_cast<int32_t*>(stage);
  uint4* rows = reinterpret_cast<uint4*>(static_cast<uint8_t*>(stage) + ((n * 4 + 255) / 256) * 256);
  nvfp4_stage_kernel<<<(unsigned)((n * 32 + 255) / 256), 256, 0, stream>>>(cache, NB, indices, block_table, req_id, R,
                                                                          MB, K, n, rows_idx, rows);
  return cudaGetLastError();
}

}  // namespace smla
