// LSE-weighted combine of partial attention results, shared by the decode
// and prefill kernels, and the balanced work split they both use.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "smla_common.cuh"

namespace smla {

// CTA c of G processes the unit-major tile range [tile_begin(c), tile_begin(c+1)).
__host__ __device__ __forceinline__ int64_t tile_begin(int64_t c, int64_t total, int G) { return (c * total) / G; }

// The CTA whose tile range holds tile x.
__host__ __device__ __forceinline__ int64_t tile_owner(int64_t x, int64_t total, int G) {
  int64_t c = ((x + 1) * G - 1) / total;
  if (c >= G) c = G - 1;
  while (c + 1 < G && tile_begin(c + 1, total, G) <= x) ++c;
  while (c > 0 && tile_begin(c, total, G) > x) --c;
  return c;
}

// Blocks per unit of combine_kernel (one per 128-column quarter of the 512 value columns).
constexpr int kCombineSplit = 4;
constexpr int kCombineThreads = 256;
constexpr int kCombineChunk = 64;  // parts staged in shared memory at a time

// LSE-weighted merge of the partial results of units split across CTAs:
//   M = max_s lse_s,  w_s = exp(lse_s - M) / sum_s' exp(lse_s' - M),
//   out = sum_s w_s * O_s,  lse = M + log(sum_s exp(lse_s - M)).
// Grid: units x kCombineSplit blocks; block (u, quarter) merges the value
// columns [128 quarter, 128 quarter + 128) of every head of unit u.  The
// parts' LSEs are staged in shared memory kCombineChunk at a time, the
// per-head weights computed once per chunk (running max and sum across
// chunks), and each thread accumulates its (head, float4 column chunk) pairs
// over the chunk's parts with the loads of several parts in flight.
template <int HG>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ lse, int H, int n_hg, int nt,
                                                                  int64_t total, int G) {
  __shared__ float w_sh[kCombineChunk * HG];  // staged LSEs, then weights exp(lse - M_run)
  __shared__ float m_run[HG], s_run[HG], a_sh[HG];
  const int64_t u = blockIdx.x / kCombineSplit;
  const int quarter = blockIdx.x % kCombineSplit;
  const int64_t c_lo = tile_owner(u * nt, total, G), c_hi = tile_owner(u * nt + nt - 1, total, G);
  if (c_lo == c_hi) return;  // finished inside one CTA, already written
  const int t = (int)(u / n_hg), hg = (int)(u % n_hg);
  const int tid = threadIdx.x;
  constexpr int kPairs = HG * 32 / kCombineThreads;  // (head, float4 chunk) pairs per thread
  float4 acc[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < HG) {
    m_run[tid] = -INFINITY;
    s_run[tid] = 0.f;
  }
  const float4* po = reinterpret_cast<const float4*>(part_o);
  for (int64_t c0 = c_lo; c0 <= c_hi; c0 += kCombineChunk) {
    const int np = (int)((c_hi - c0 + 1) < kCombineChunk ? (c_hi - c0 + 1) : kCombineChunk);
    __syncthreads();  // previous chunk's weights consumed
    for (int i = tid; i < np * HG; i += kCombineThreads) w_sh[i] = __ldg(part_lse + (c0 + i / HG + u) * HG + i % HG);
    __syncthreads();
    if (tid < HG) {
      float m = m_run[tid];
      for (int p = 0; p < np; ++p) m = fmaxf(m, w_sh[p * HG + tid]);
      const float a = m == -INFINITY ? 1.f : expf(m_run[tid] - m);  // exp(-inf) = 0 when m_run was -inf
      float s = s_run[tid] * a;
      for (int p = 0; p < np; ++p) {
        const float wp = m == -INFINITY ? 0.f : expf(w_sh[p * HG + tid] - m);
        w_sh[p * HG + tid] = wp;
        s += wp;
      }
      a_sh[tid] = a;
      m_run[tid] = m;
      s_run[tid] = s;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const int idx = tid + kCombineThreads * i;
      const int h = idx >> 5, j = (idx & 31) + 32 * quarter;
      const float a = a_sh[h];
      float4 v = acc[i];
      v.x *= a;
      v.y *= a;
      v.z *= a;
      v.w *= a;
      int p = 0;
      for (; p + 4 <= np; p += 4) {
        float4 x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = __ldg(po + ((c0 + p + e + u) * HG + h) * (kDv / 4) + j);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float wgt = w_sh[(p + e) * HG + h];
          v.x += wgt * x[e].x;
          v.y += wgt * x[e].y;
          v.z += wgt * x[e].z;
          v.w += wgt * x[e].w;
        }
      }
      for (; p < np; ++p) {
        const float4 x = __ldg(po + ((c0 + p + u) * HG + h) * (kDv / 4) + j);
        const float wgt = w_sh[p * HG + h];
        v.x += wgt * x.x;
        v.y += wgt * x.y;
        v.z += wgt * x.z;
        v.w += wgt * x.w;
      }
      acc[i] = v;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const int idx = tid + kCombineThreads * i;
    const int h = idx >> 5, j = (idx & 31) + 32 * quarter;
    const float inv = s_run[h] > 0.f ? 1.f / s_run[h] : 0.f;
    __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(out + ((int64_t)t * H + hg * HG + h) * kDv + 4 * j);
    d[0] = __floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv);
    d[1] = __floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv);
  }
  if (quarter == 0 && tid < HG)
    lse[(int64_t)t * H + hg * HG + tid] = s_run[tid] > 0.f ? m_run[tid] + logf(s_run[tid]) : -INFINITY;
}

}  // namespace smla
