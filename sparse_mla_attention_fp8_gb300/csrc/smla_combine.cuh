// LSE-weighted combine of partial attention results, shared by the decode
// and prefill kernels, and the balanced work split they both use.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "smla_common.cuh"

namespace smla {

// CTA c of G processes the unit-major tile range [tile_begin(c), tile_begin(c+1)).
__host__ __device__ __forceinline__ int64_t tile_begin(int64_t c, int64_t total, int G) { return (c * total) / G; }

// LSE-weighted merge of the partial results of units split across CTAs:
//   M = max_s lse_s,  w_s = exp(lse_s - M) / sum_s' exp(lse_s' - M),
//   out = sum_s w_s * O_s,  lse = M + log(sum_s exp(lse_s - M)).
// One block per unit; thread (h, c4) owns head h and float4 column chunks.
template <int HG>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                      int H, int n_hg, int nt, int64_t total, int G) {
  const int64_t u = blockIdx.x;
  auto owner = [&](int64_t x) -> int64_t {
    int64_t c = ((x + 1) * G - 1) / total;
    if (c >= G) c = G - 1;
    while (c + 1 < G && tile_begin(c + 1, total, G) <= x) ++c;
    while (c > 0 && tile_begin(c, total, G) > x) --c;
    return c;
  };
  const int64_t c_lo = owner(u * nt), c_hi = owner(u * nt + nt - 1);
  if (c_lo == c_hi) return;  // finished inside one CTA, already written
  const int t = (int)(u / n_hg), hg = (int)(u % n_hg);
  constexpr int kThreadsPerHead = 256 / HG;      // 16 (HG=16) or 8 (HG=32)
  const int h = threadIdx.x / kThreadsPerHead;
  const int sub = threadIdx.x % kThreadsPerHead;
  float m = -INFINITY;
  for (int64_t c = c_lo; c <= c_hi; ++c) m = fmaxf(m, __ldg(part_lse + (c + u) * HG + h));
  float wsum = 0.f;
  if (m != -INFINITY)
    for (int64_t c = c_lo; c <= c_hi; ++c) wsum += expf(__ldg(part_lse + (c + u) * HG + h) - m);
  if (sub == 0) lse[(int64_t)t * H + hg * HG + h] = (m == -INFINITY) ? -INFINITY : m + logf(wsum);
  const float inv = m == -INFINITY ? 0.f : 1.f / wsum;
  constexpr int kChunks = kDv / 4;                // 128 float4 per head row
  float4 acc[kChunks / kThreadsPerHead];
#pragma unroll
  for (int k = 0; k < kChunks / kThreadsPerHead; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (m != -INFINITY) {
    for (int64_t c = c_lo; c <= c_hi; ++c) {
      const float wgt = expf(__ldg(part_lse + (c + u) * HG + h) - m) * inv;
      const float4* src = reinterpret_cast<const float4*>(part_o + ((c + u) * HG + h) * kDv);
#pragma unroll
      for (int k = 0; k < kChunks / kThreadsPerHead; ++k) {
        const float4 v = __ldg(src + sub + k * kThreadsPerHead);
        acc[k].x += wgt * v.x;
        acc[k].y += wgt * v.y;
        acc[k].z += wgt * v.z;
        acc[k].w += wgt * v.w;
      }
    }
  }
  __nv_bfloat16* o = out + ((int64_t)t * H + hg * HG + h) * kDv;
#pragma unroll
  for (int k = 0; k < kChunks / kThreadsPerHead; ++k) {
    const int c4 = sub + k * kThreadsPerHead;
    __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(o + 4 * c4);
    d[0] = __floats2bfloat162_rn(acc[k].x, acc[k].y);
    d[1] = __floats2bfloat162_rn(acc[k].z, acc[k].w);
  }
}

}  // namespace smla
