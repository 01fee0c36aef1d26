// MLA weight absorption around the sparse attention (vLLM flashmla_sparse.py,
// FlashMLASparseImpl.forward and _v_up_proj), per head h as a batched GEMM on
// the tensor cores:
//   query side:  ql_nope[t, h, :] = q[t, h, 0:P] x W_UK_T[h]          (P -> 512)
//                q_out[t, h, :]   = ql_nope[t, h, :] ++ q[t, h, P:P+64]
//                (the page's bmm, transpose back and cat, in one kernel: the
//                epilogue writes the attention-ready [T, H, 576] query)
//   value side:  out[t, h, :]     = attn_out[t, h, :] x W_UV[h]        (512 -> V)
// bf16 operands, fp32 accumulation in tensor memory, bf16 results.
//
// One CTA per (N tile, 128-token tile, head), N tiles fastest so that the
// N tiles of one token tile share its A tile in L2, and one head's weights
// stay in L2 across its token tiles.  TMA loads of A (K-major, 128-byte
// swizzle: 128 tokens x 64 features per stage) and B (the weight rows,
// MN-major, 128-byte swizzle: 64 features x N columns) into a ring of stages;
// one thread issues tcgen05.mma kind::f16 (M = 128, N = BN, K = 16); four
// epilogue warps read the accumulator (one token row per thread), round to
// bf16, stage their 32 rows as 128-byte-swizzled 64-column panels in the
// (by then idle) stage memory and write each panel with a TMA store.  Two
// CTAs share an SM, so one's epilogue overlaps the other's loads.  Warp
// roles: 0 TMA producer, 1 MMA issuer, 2..5 epilogue (TMEM lane quarters 2,
// 3, 0, 1).
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "smla_common.cuh"
#include "smla_kernels.h"

namespace smla {

namespace {

constexpr int kBM = 128;     // tokens per tile (M)
constexpr int kBK = 64;      // features per stage (one 128-byte swizzle atom of bf16)
constexpr int kThreads = 6 * 32;
constexpr int kStoreRows = 32;  // rows of one TMA store box: one epilogue warp's TMEM lane quarter

template <int BN, int STAGES>
struct GemmLay {
  static constexpr int kATile = kBM * kBK * 2;          // 16 KB
  static constexpr int kBPanel = kBK * 128;             // 8 KB: 64 k rows x 64 n (128 bytes)
  static constexpr int kBTile = (BN / 64) * kBPanel;    // BN = 256: 32 KB
  static constexpr int kStage = kATile + kBTile;
  static constexpr int kOutPanel = kBM * 128;           // 16 KB: 128 rows x 64 bf16 columns
  static constexpr int kOffBar = STAGES * kStage;
  static constexpr int kNumBars = 2 * STAGES + 1;       // full[S], empty[S], done
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemAlloc = kOffMisc + 16 + 1024;
  static_assert(kStage % 1024 == 0, "stage alignment");
  static_assert((BN / 64) * kOutPanel <= STAGES * kStage, "output staging reuses the stage ring");
  static_assert(2 * (kSmemAlloc + 1024) <= 233472, "two CTAs per SM");
};

struct GemmParams {
  int T, K;                 // tokens, reduction length (a multiple of 64)
  int a_x0_stride;          // A column offset per head: the head's first feature in the 2-D view of A
  int b_y0_stride;          // B row offset per head: the head's first weight row in the 2-D view of B
  int c_x0_stride;          // C column offset per head in the 2-D view of C ([T, H * ldc])
  int H;
  const __nv_bfloat16* rope; // query side: q with its RoPE part at rope + (t * H + h) * rope_ld + rope_off, else null
  __nv_bfloat16* rope_dst;  // and its destination: rope_dst + (t * H + h) * rope_dst_ld
  int rope_ld, rope_off, rope_dst_ld;
  int* status;
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 2)
    head_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap a_map,
                     const __grid_constant__ CUtensorMap b_map, const __grid_constant__ CUtensorMap c_map) {
  using L = GemmLay<BN, STAGES>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kBM, h = blockIdx.z;
  const int nk = p.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars[s], 1);
      mbar_init(&bars[STAGES + s], 1);
    }
    mbar_init(&bars[2 * STAGES], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
#define GEMM_WAIT(idx, parity) mbar_wait(&bars[(idx)], (parity), abort_flag, p.status, kDevWaitTimeout)

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % STAGES, use = kt / STAGES;
        if (use >= 1 && !GEMM_WAIT(STAGES + s, (use + 1) & 1)) break;
        const uint32_t stage = smem_u32(smem + s * L::kStage);
        mbar_arrive_expect_tx(&bars[s], (uint32_t)L::kStage);
        tma_load_2d(stage, &a_map, h * p.a_x0_stride + kt * kBK, m0, &bars[s]);
        for (int j = 0; j < BN / 64; ++j)
          tma_load_2d(stage + L::kATile + j * L::kBPanel, &b_map, n0 + 64 * j, h * p.b_y0_stride + kt * kBK,
                      &bars[s]);
        ++issued;
      }
      // no copy may still be landing in shared memory when the CTA exits
      if (issued > 0) mbar_wait_drain(&bars[(issued - 1) % STAGES], ((issued - 1) / STAGES) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kBM, BN, 0, 1);
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % STAGES;
        if (!GEMM_WAIT(s, (kt / STAGES) & 1)) break;
        tc_fence_after();
        const uint32_t stage = smem_u32(smem + s * L::kStage);
        // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; B: MN-major,
        // 64-column panels kBPanel apart, 8-row (k) groups 1024 B apart
        const uint64_t da = make_sdesc(stage, 16, 1024, kLayoutSw128);
        const uint64_t db = make_sdesc(stage + L::kATile, L::kBPanel, 1024, kLayoutSw128);
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_ss(tmem, da + ((32 * k) >> 4), db + ((2048 * k) >> 4), idesc, (kt > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bars[STAGES + s]);
      }
      mma_commit(&bars[2 * STAGES]);  // the accumulator is complete (or, after an abort, nothing is in flight)
      mbar_wait_drain(&bars[2 * STAGES], 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int qd = warp & 3;
    const int r = 32 * qd + lane;  // the tile row (token m0 + r) this thread's TMEM lane holds
    // query side: the RoPE part goes after the absorbed NoPE part (once, with the first N tile), copied
    // while the MMAs run: 8 lanes per 128-byte row, 4 rows per pass
    if (p.rope != nullptr && blockIdx.x == 0) {
#pragma unroll
      for (int it = 0; it < kStoreRows / 4; ++it) {
        const int t = m0 + 32 * qd + 4 * it + (lane >> 3);
        if (t < p.T) {
          const int64_t th = (int64_t)t * p.H + h;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.rope + th * p.rope_ld + p.rope_off) + (lane & 7));
          reinterpret_cast<uint4*>(p.rope_dst + th * p.rope_dst_ld)[lane & 7] = v;
        }
      }
    }
    bool dead = !GEMM_WAIT(2 * STAGES, 0);
    dead = __any_sync(0xffffffffu, dead);
    tc_fence_after();
    if (!dead) {
      const uint32_t row_addr = tmem + ((uint32_t)(32 * qd) << 16);
#pragma unroll 1
      for (int j = 0; j < BN / 64; ++j) {
        // the accumulator is complete, so every stage (operand tiles and loads) is idle: panel j of the
        // output is staged at j * kOutPanel, rows 128 bytes apart, 16-byte chunks swizzled by row & 7
        const uint32_t panel = smem_u32(smem + j * L::kOutPanel);
        const uint32_t row_base = panel + (uint32_t)r * 128u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16_sync(row_addr + 64 * j + 16 * c, v);
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          st_shared_v4(row_base + ((uint32_t)((2 * c) ^ (r & 7)) << 4), o[0], o[1], o[2], o[3]);
          st_shared_v4(row_base + ((uint32_t)((2 * c + 1) ^ (r & 7)) << 4), o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        // rows at or beyond T lie outside the tensor map and are not written; a box with no row below T
        // is not issued at all
        if (lane == 0 && m0 + 32 * qd < p.T) {
          tma_store_2d(&c_map, panel + (uint32_t)(32 * qd) * 128u, h * p.c_x0_stride + n0 + 64 * j, m0 + 32 * qd);
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait_read_all();  // shared memory stays valid until the stores have read it
      __syncwarp();
    }
  }
#undef GEMM_WAIT
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor map over a [rows, cols] row-major matrix, box [box_cols, box_rows], 128-byte swizzle;
// rows or columns outside the matrix read as zeros.
cudaError_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                     uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows}, es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::once_flag g_gemm_attr_once[2][64];
cudaError_t g_gemm_attr_err[2][64];

template <int BN, int STAGES>
cudaError_t launch_head_gemm(const GemmParams& p, const CUtensorMap& a_map, const CUtensorMap& b_map,
                             const CUtensorMap& c_map, int n_tiles, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int bi = BN == 256 ? 0 : 1;
  std::call_once(g_gemm_attr_once[bi][dev], [bi, dev] {
    g_gemm_attr_err[bi][dev] = cudaFuncSetAttribute(
        head_gemm_kernel<BN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, GemmLay<BN, STAGES>::kSmemAlloc);
  });
  if (g_gemm_attr_err[bi][dev] != cudaSuccess) return g_gemm_attr_err[bi][dev];
  if ((p.T + kBM - 1) / kBM > 65535 || p.H > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)n_tiles, (unsigned)((p.T + kBM - 1) / kBM), (unsigned)p.H);
  head_gemm_kernel<BN, STAGES>
      <<<grid, kThreads, GemmLay<BN, STAGES>::kSmemAlloc, stream>>>(p, a_map, b_map, c_map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_absorb_q(const void* q, const void* w_uk_t, void* q_out, int T, int H, int P, int* status,
                            cudaStream_t stream) {
  const int ld = P + kRope;
  CUtensorMap a_map, b_map, c_map;
  cudaError_t e = make_map(&a_map, q, (uint64_t)T, (uint64_t)H * ld, kBK, kBM);
  if (e != cudaSuccess) return e;
  e = make_map(&b_map, w_uk_t, (uint64_t)H * P, kDv, 64, kBK);
  if (e != cudaSuccess) return e;
  e = make_map(&c_map, q_out, (uint64_t)T, (uint64_t)H * kDqk, 64, kStoreRows);
  if (e != cudaSuccess) return e;
  GemmParams p{};
  p.T = T;
  p.K = P;
  p.a_x0_stride = ld;
  p.b_y0_stride = P;
  p.c_x0_stride = kDqk;
  p.H = H;
  p.rope = static_cast<const __nv_bfloat16*>(q);
  p.rope_ld = ld;
  p.rope_off = P;
  p.rope_dst = static_cast<__nv_bfloat16*>(q_out) + kDv;
  p.rope_dst_ld = kDqk;
  p.status = status;
  return launch_head_gemm<256, 2>(p, a_map, b_map, c_map, kDv / 256, stream);
}

cudaError_t launch_v_up_proj(const void* attn_out, const void* w_uv, void* out, int T, int H, int V, int* status,
                             cudaStream_t stream) {
  if (V % 128 != 0) return cudaErrorInvalidValue;
  CUtensorMap a_map, b_map, c_map;
  cudaError_t e = make_map(&a_map, attn_out, (uint64_t)T, (uint64_t)H * kDv, kBK, kBM);
  if (e != cudaSuccess) return e;
  e = make_map(&b_map, w_uv, (uint64_t)H * kDv, (uint64_t)V, 64, kBK);
  if (e != cudaSuccess) return e;
  e = make_map(&c_map, out, (uint64_t)T, (uint64_t)H * V, 64, kStoreRows);
  if (e != cudaSuccess) return e;
  GemmParams p{};
  p.T = T;
  p.K = kDv;
  p.a_x0_stride = kDv;
  p.b_y0_stride = kDv;
  p.c_x0_stride = V;
  p.H = H;
  p.rope = nullptr;
  p.status = status;
  return launch_head_gemm<128, 3>(p, a_map, b_map, c_map, V / 128, stream);
}

}  // namespace smla
