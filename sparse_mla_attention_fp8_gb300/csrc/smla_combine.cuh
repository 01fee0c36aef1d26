// LSE-weighted combine of partial attention results, shared by the decode
// and prefill kernels, and the balanced work split they both use.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#include "sm103_ptx.cuh"
#include "smla_common.cuh"

namespace smla {

// a / b for a >= 0, b > 0, in 32 bits whenever both fit: on the GPU a 64-bit
// division is a long out-of-line routine (run at every CTA's entry here).
__host__ __device__ __forceinline__ int64_t udiv_fast(int64_t a, int64_t b) {
  return (a <= 0xFFFFFFFFll && b <= 0xFFFFFFFFll) ? (int64_t)((uint32_t)a / (uint32_t)b) : a / b;
}

// CTA c of G processes the unit-major tile range [tile_begin(c), tile_begin(c+1)).
__host__ __device__ __forceinline__ int64_t tile_begin(int64_t c, int64_t total, int G) { return udiv_fast(c * total, G); }

// The CTA whose tile range holds tile x.
__host__ __device__ __forceinline__ int64_t tile_owner(int64_t x, int64_t total, int G) {
  int64_t c = udiv_fast((x + 1) * G - 1, total);
  if (c >= G) c = G - 1;
  while (c + 1 < G && tile_begin(c + 1, total, G) <= x) ++c;
  while (c > 0 && tile_begin(c, total, G) > x) --c;
  return c;
}

// Blocks per unit of combine_kernel: each merges 512 / combine_split value
// columns of every head of the unit, one (head, float4 column chunk) pair per
// thread.
template <int HG>
__host__ __device__ constexpr int combine_split() {
  return HG <= 32 ? 8 : 32;
}
template <int HG>
__host__ __device__ constexpr int combine_threads() {
  return HG * (128 / combine_split<HG>());
}
constexpr int kCombineChunk = 8;  // parts per round: their loads are in flight together

// LSE-weighted merge of the partial results of units split across CTAs:
//   M = max_s lse_s,  w_s = exp(lse_s - M) / sum_s' exp(lse_s' - M),
//   out = sum_s w_s * O_s,  lse = M + log(sum_s exp(lse_s - M)).
// Grid: combine_split<HG>() blocks of combine_threads<HG>() = HG x
// (128 / combine_split<HG>()) threads per unit (by_boundary = 0), or per
// boundary between consecutive CTA ranges (by_boundary = 1: the unit the
// boundary cuts, merged by the first boundary inside it; for many units over
// few CTAs).  combine_grid() picks the smaller.  Each thread first issues the loads of its
// partial-O chunk for kCombineChunk parts, then reads the parts' LSEs (from
// L2 or L1, shared by the block), so that one round trip covers both; parts
// beyond the first round are merged with a running max and sum.
template <int HG>
__global__ void __launch_bounds__(combine_threads<HG>()) combine_kernel(const float* __restrict__ part_o,
                                                                  const float* __restrict__ part_lse,
                                                                  __nv_bfloat16* __restrict__ out,
                                                                  float* __restrict__ lse, int H, int n_hg, int nt,
                                                                  int64_t total, int G, int by_boundary) {
  constexpr int kSplit = combine_split<HG>();
  constexpr int kChunks = 128 / kSplit;  // float4 column chunks per block and head
  grid_dependency_wait();  // the attention kernel's partials (launched as its programmatic dependent)
  int64_t u;
  if (by_boundary) {
    const int64_t c = blockIdx.x / kSplit + 1;  // boundary between CTA ranges c - 1 and c
    const int64_t b = tile_begin(c, total, G);
    u = udiv_fast(b, nt);
    if (b == u * nt) return;                                   // no unit is cut here
    if (tile_begin(c - 1, total, G) > u * nt) return;          // an earlier boundary cuts this unit
  } else {
    u = blockIdx.x / kSplit;
  }
  const int part = blockIdx.x % kSplit;
  const int64_t c_lo = tile_owner(u * nt, total, G), c_hi = tile_owner(u * nt + nt - 1, total, G);
  if (c_lo == c_hi) return;  // finished inside one CTA, already written
  const int tid = threadIdx.x;
  const int h = tid / kChunks, j = part * kChunks + tid % kChunks;  // head, float4 column chunk
  const int t = (int)udiv_fast(u, n_hg), hg = (int)(u - (int64_t)t * n_hg);
  const float4* po = reinterpret_cast<const float4*>(part_o);
  float m = -INFINITY, ssum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t c0 = c_lo; c0 <= c_hi; c0 += kCombineChunk) {
    const int np = (int)((c_hi - c0 + 1) < kCombineChunk ? (c_hi - c0 + 1) : kCombineChunk);
    float4 v[kCombineChunk];
    float l[kCombineChunk];
#pragma unroll
    for (int e = 0; e < kCombineChunk; ++e)
      if (e < np) v[e] = __ldg(po + ((c0 + e + u) * HG + h) * (kDv / 4) + j);
#pragma unroll
    for (int e = 0; e < kCombineChunk; ++e) l[e] = e < np ? __ldg(part_lse + (c0 + e + u) * HG + h) : -INFINITY;
    float mn = m;
#pragma unroll
    for (int e = 0; e < kCombineChunk; ++e) mn = fmaxf(mn, l[e]);
    if (mn == -INFINITY) continue;  // no valid row in any part so far
    const float a = __expf(m - mn);  // 0 when m was -inf
    ssum *= a;
    acc.x *= a;
    acc.y *= a;
    acc.z *= a;
    acc.w *= a;
#pragma unroll
    for (int e = 0; e < kCombineChunk; ++e) {
      if (e < np) {
        const float wgt = __expf(l[e] - mn);
        ssum += wgt;
        acc.x += wgt * v[e].x;
        acc.y += wgt * v[e].y;
        acc.z += wgt * v[e].z;
        acc.w += wgt * v[e].w;
      }
    }
    m = mn;
  }
  // approximate reciprocal and log (a few ulp; ssum >= 1 here)
  const float inv = ssum > 0.f ? __fdividef(1.f, ssum) : 0.f;
  __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(out + ((int64_t)t * H + hg * HG + h) * kDv + 4 * j);
  d[0] = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  d[1] = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  if (part == 0 && j == 0) lse[(int64_t)t * H + hg * HG + h] = ssum > 0.f ? m + __logf(ssum) : -INFINITY;
}

// Launches combine_kernel behind the attention kernel just issued on `stream`
// as its programmatic dependent: its launch overlaps the attention kernel's
// tail, and its first instruction waits for the partial results.
template <int HG>
inline cudaError_t launch_combine(const float* part_o, const float* part_lse, __nv_bfloat16* out, float* lse, int H,
                                  int n_hg, int nt, int64_t total, int G, int64_t units, cudaStream_t stream);

// Blocks and mode of combine_kernel for a split of `units` units over G CTA
// ranges.
template <int HG>
inline void combine_grid(int64_t units, int G, unsigned* blocks, int* by_boundary) {
  const int64_t boundaries = G > 1 ? G - 1 : 1;
  *by_boundary = boundaries < units ? 1 : 0;
  *blocks = (unsigned)((*by_boundary ? boundaries : units) * combine_split<HG>());
}

template <int HG>
inline cudaError_t launch_combine(const float* part_o, const float* part_lse, __nv_bfloat16* out, float* lse, int H,
                                  int n_hg, int nt, int64_t total, int G, int64_t units, cudaStream_t stream) {
  unsigned blocks;
  int by_boundary;
  combine_grid<HG>(units, G, &blocks, &by_boundary);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(combine_threads<HG>(), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<HG>, part_o, part_lse, out, lse, H, n_hg, nt, total, G, by_boundary);
}

}  // namespace smla
