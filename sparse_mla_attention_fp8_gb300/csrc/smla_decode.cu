// FP8 sparse MLA decode on sm_103a, reading the 656-byte cache rows as stored.
//
// What is computed (vLLM flashmla_sparse.py: the "FP8 with scale" row format
// in the module docstring, FlashMLASparseImpl.forward and its FP8 decode
// kernel call): for each query token t and each of its H heads,
//   s_j = softmax_scale * <q[t,h,:], K_j>, K_j = [e4m3(c) * scale_j[c/128] for
//         c < 512] ++ RoPE_j (64 bf16),
//   out = sum_j softmax(s)_j * K_j[0:512],  lse = log sum_j exp(s_j),
// over the token's top-k rows (translated through the paged block table);
// invalid rows are masked, a token without valid rows gets out = 0, lse = -inf.
//
// Design: the tensor cores read the cache bytes as stored, with no
// dequantization pass.
//  * Tiles of 128 top-k rows are gathered by TMA (tile::gather4, 128-byte
//    swizzle) straight into shared memory: the 512 e4m3 codes as four
//    K-major operand panels, the 64 bf16 RoPE values as a fifth panel and the
//    four float32 scales beside them.  Two tiles are double-buffered.
//  * Q is split once per (token, 16-head group) into two e4m3 terms,
//    q * 2^s_h = hi + lo (s_h a per-head power of two putting max |q| near
//    448), exact for all but negligibly small components; hi and lo are the
//    two halves of an N = 32 operand.  QK^T for each 128-column scale group g
//    is one kind::f8f6f4 product E_g [Q_hi Q_lo]^T (M = 128 rows, N = 32,
//    K = 128 codes), the RoPE part a bf16 product; the softmax combines
//    s = 2^-s_h sum_g scale_g (S_g,hi + S_g,lo) + S_rope in fp32.
//  * P.V for value chunk q (= scale group q) is one kind::f8f6f4 product
//    O_q^T += E_q^T P'_q with the same code panel read MN-major and
//    P'_q = 2^7 p * scale_q / R_q split into e4m3 hi + lo (R_q a running
//    power-of-two bound of the group's scales).  The running max is refreshed
//    whenever a tile's maximum exceeds it by more than a factor 2 (so p <= 2),
//    which keeps P' <= 256: the top of the e4m3 range, where hi + lo carries
//    8 significant bits down to ~2^-10 of the largest weight.  O is rescaled
//    in tensor memory when R_q or the running max changes.
//  * Warp roles: index translation (1 warp), TMA producer (1), tensor-core
//    issuer (1 thread), Q preparation (4 warps), softmax / epilogue (4 warps,
//    one thread per tile row / output column).
#include <cuda.h>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "smla_combine.cuh"
#include "smla_common.cuh"
#include "smla_kernels.h"

namespace smla {

namespace {

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr int HG = 16;       // heads per CTA work unit
constexpr float kMaxSlack = 1.0f;      // log2 growth of a head's max tolerated before rescaling O (p <= 2)
constexpr float kPScale = 128.0f;      // P' = kPScale * p * scale / R  <=  256
constexpr float kPScaleInv = 1.0f / 128.0f;
constexpr int kRows = 128;   // top-k rows per tile

// ---- shared memory layout (offsets from a 1024-byte aligned base)
constexpr int kPanel = kRows * 128;                   // 16 KB: 128 rows x 128 bytes
constexpr int kKvRope = 4 * kPanel;                   // RoPE panel after the 4 code panels
// Scale rows: each TMA destination must be 128-byte aligned, so the 4 rows of
// one gather (64 bytes) get a 128-byte slot: row r at (r / 4) * 128 + (r % 4) * 16.
constexpr int kKvScale = 5 * kPanel;
constexpr int kKvBuf = 5 * kPanel + (kRows / 4) * 128;  // 86016
constexpr int kQPanel = 32 * 128;                     // 32 operand rows (hi, lo) x 128 codes
constexpr int kQRope = 4 * kQPanel;                   // 16 rows x 64 bf16
constexpr int kQBuf = 4 * kQPanel + HG * 128;         // 18432
constexpr int kPGroup = kRows * 32;                   // P'_q: 128 rows x 32 codes
constexpr int kOffKv = 0;
constexpr int kOffQ = kOffKv + 2 * kKvBuf;
constexpr int kOffP = kOffQ + 2 * kQBuf;
constexpr int kOffSlots = kOffP + 4 * kPGroup;        // int32 [4][128]
constexpr int kOffValid = kOffSlots + 4 * kRows * 4;  // uint8 [2][128]
constexpr int kOffPre = kOffValid + 2 * kRows;        // float [4][16] inverse Q prescales
constexpr int kOffRedMax = kOffPre + 4 * HG * 4;      // float [2][4 warps][16]
constexpr int kOffRedSc = kOffRedMax + 2 * 4 * HG * 4;  // float [2][4 warps][4]
constexpr int kOffRedSum = kOffRedSc + 2 * 4 * 4 * 4;   // float [4 warps][16]
constexpr int kOffBar = kOffRedSum + 4 * HG * 4;
enum {
  kBarKvFull = 0, kBarKvEmpty = 2, kBarSFull = 4, kBarPFull = 6, kBarPvDone = 7, kBarIdxFull = 8,
  kBarIdxEmpty = 12, kBarQFull = 16, kBarQEmpty = 18, kBarOFree = 20, kNumBars = 21
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kKvBuf % 1024 == 0, "operand alignment");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// ---- tensor memory columns
constexpr int kSCols = 4 * 32 + HG;   // per S buffer: 4 groups x (hi, lo) x 16 heads + RoPE
constexpr int kOCol = 2 * kSCols;     // O^T: 4 chunks x (hi, lo) x 16 heads
constexpr int kTmemCols = 512;
static_assert(kOCol + 4 * 32 <= kTmemCols, "tensor memory budget");

// ---- warp roles
constexpr int kMmaWarp = 4, kIndexWarp = 5, kTmaWarp = 6, kQWarp0 = 7;
constexpr int kThreads = 32 * 11;

__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

struct Params {
  const __nv_bfloat16* q;
  const int32_t* indices;
  const int32_t* block_table;
  const int32_t* req_id;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int* status;
  float scale_log2;
  int T, H, K, R, MB;
  int64_t NB;
  int n_hg, nt;
  int64_t total;
  int G;
};

struct TileInfo {
  int u, kt, t, hg;
  bool seg_start, seg_end;
};

__device__ __forceinline__ TileInfo tile_info(const Params& p, int64_t x, int64_t xbeg, int64_t xend) {
  TileInfo ti;
  ti.u = (int)(x / p.nt);
  ti.kt = (int)(x - (int64_t)ti.u * p.nt);
  ti.t = ti.u / p.n_hg;
  ti.hg = ti.u - ti.t * p.n_hg;
  ti.seg_start = (x == xbeg) || (ti.kt == 0);
  ti.seg_end = (x == xend - 1) || (ti.kt == p.nt - 1);
  return ti;
}

__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
      "%4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// e4m3 pair (round to nearest even, saturating) of two floats: lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// decode an e4m3 pair (low byte first) to two floats (exact)
__device__ __forceinline__ float2 e4m3x2_decode(uint32_t pair16) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)pair16));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
// x -> (hi, lo) e4m3 codes with x = hi + lo wherever both are representable.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = e4m3x2(x0, x1);
  const float2 d = e4m3x2_decode(hi);
  lo = e4m3x2(x0 - d.x, x1 - d.y);
}

// 16 values per lane reduced across the warp; lane l ends with value index l >> 1.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int w = 16, n = 8; n >= 1; w >>= 1, n >>= 1) {
    const bool up = lane & w;
#pragma unroll
    for (int j = 0; j < n; ++j) {
      const float send = up ? v[j] : v[j + n];
      const float keep = up ? v[j + n] : v[j];
      v[j] = op(keep, __shfl_xor_sync(kFullMask, send, w));
    }
  }
  v[0] = op(v[0], __shfl_xor_sync(kFullMask, v[0], 1));
  return v[0];
}

__device__ __forceinline__ float pow2_ceil(float x) {  // smallest power of two >= x (x > 0, normal)
  const uint32_t u = __float_as_uint(x);
  const uint32_t e = u & 0x7F800000u;
  return __uint_as_float((u & 0x007FFFFFu) ? e + 0x00800000u : e);
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_decode_fp8_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap map_row,
                                 const __grid_constant__ CUtensorMap map_scale) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + kOffSlots);
  uint8_t* valid = smem + kOffValid;
  float* pre_ring = reinterpret_cast<float*>(smem + kOffPre);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t xbeg = tile_begin(blockIdx.x, p.total, p.G);
  const int64_t xend = tile_begin(blockIdx.x + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarKvFull + i], 1);
      mbar_init(&bars[kBarKvEmpty + i], 1);
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarQFull + i], 4);
      mbar_init(&bars[kBarQEmpty + i], 1);
    }
    mbar_init(&bars[kBarPFull], 4);
    mbar_init(&bars[kBarPvDone], 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarIdxFull + i], 32);
      mbar_init(&bars[kBarIdxEmpty + i], 1);
    }
    mbar_init(&bars[kBarOFree], 4);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

#define SMLA_WAIT(bar_idx, parity) mbar_wait(&bars[(bar_idx)], (parity), abort_flag, p.status, kDevWaitTimeout)

  if (warp == kIndexWarp) {
    // ------------------------------------------------------------ index translation
    // The next tile's indices are loaded before this tile's block-table reads,
    // so each tile costs about one memory round trip.
    int32_t cur[4], nxt[4], req_cur = 0, req_nxt = 0;
    auto load_idx = [&](int tl, int32_t (&v)[4], int32_t& rq) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      rq = __ldg(p.req_id + ti.t);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = ti.kt * kRows + lane + 32 * i;
        v[i] = k < p.K ? __ldg(p.indices + (int64_t)ti.t * p.K + k) : -1;
      }
    };
    if (n_local > 0) load_idx(0, cur, req_cur);
    for (int tl = 0; tl < n_local; ++tl) {
      if (tl + 1 < n_local) load_idx(tl + 1, nxt, req_nxt);
      const int b4 = tl & 3;
      if (tl >= 4 && !SMLA_WAIT(kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        slots_ring[b4 * kRows + lane + 32 * i] = translate_slot(cur[i], req_cur, p.block_table, p.R, p.MB, p.NB);
      mbar_arrive(&bars[kBarIdxFull + b4]);
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
      req_cur = req_nxt;
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    // Lane l gathers rows 4l..4l+3 of each tile: the four 128-code panels, the
    // RoPE values and the scales.  Invalid rows use row coordinate -1, which
    // the tensor map fills with zeros.
    const uint32_t kv0 = smem_u32(smem + kOffKv);
    const int r = 4 * lane;
    const uint32_t roff = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128);
    for (int tl = 0; tl < n_local; ++tl) {
      const int b = tl & 1, b4 = tl & 3;
      if (!SMLA_WAIT(kBarIdxFull + b4, (tl >> 2) & 1)) break;
      if (tl >= 2 && !SMLA_WAIT(kBarKvEmpty + b, ((tl >> 1) + 1) & 1)) break;
      const int4 s = *reinterpret_cast<const int4*>(slots_ring + b4 * kRows + r);
      *reinterpret_cast<uint32_t*>(valid + b * kRows + r) =
          (s.x >= 0 ? 1u : 0u) | (s.y >= 0 ? 1u << 8 : 0u) | (s.z >= 0 ? 1u << 16 : 0u) | (s.w >= 0 ? 1u << 24 : 0u);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kBarKvFull + b], kRows * (512 + 128 + 16));
        mbar_arrive(&bars[kBarIdxEmpty + b4]);  // slots copied to registers
      }
      __syncwarp();
      const uint32_t kv = kv0 + b * kKvBuf;
#pragma unroll
      for (int pn = 0; pn < 4; ++pn)
        tma_gather4(kv + pn * kPanel + roff, &map_row, 128 * pn, s.x, s.y, s.z, s.w, &bars[kBarKvFull + b]);
      tma_gather4(kv + kKvRope + roff, &map_row, kRopeOff, s.x, s.y, s.z, s.w, &bars[kBarKvFull + b]);
      tma_gather4(kv + kKvScale + lane * 128, &map_scale, kScaleOff, s.x, s.y, s.z, s.w, &bars[kBarKvFull + b]);
    }
  } else if (warp >= kQWarp0) {
    // ------------------------------------------------------------ Q preparation
    // 8 threads per head: thread part owns NoPE columns [64 part, 64 part + 64)
    // and RoPE chunk `part`.  q * 2^s_h = hi + lo in e4m3 with s_h chosen so
    // that max |q * 2^s_h| <= 448.
    const int qt = tid - 32 * kQWarp0;  // 0..127
    const int h = qt >> 3, part = qt & 7;
    int seg = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      if (!ti.seg_start) continue;
      const int qb = seg & 1;
      if (seg >= 2 && !SMLA_WAIT(kBarQEmpty + qb, ((seg >> 1) + 1) & 1)) break;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)ti.t * p.H + ti.hg * HG + h) * kDqk);
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __ldg(src + 8 * part + i);
      const uint4 rope = __ldg(src + 64 + part);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
      amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
      int sh = 0;
      if (amax > 0.f) {
        int e;
        frexpf(448.f / amax, &e);  // 448 / amax = m * 2^e, m in [0.5, 1)
        sh = e - 1;
      }
      const float pre = ldexpf(1.f, sh);
      const uint32_t qs = smem_u32(smem + kOffQ + qb * kQBuf);
      // codes for columns 64 part .. 64 part + 63: panel part / 2, chunks 4 (part % 2) .. +3
      const int pn = part >> 1;
#pragma unroll
      for (int i = 0; i < 8; i += 2) {  // 16 columns per chunk = two uint4 of bf16
        uint32_t hi[4], lo[4];
        const uint32_t w8[8] = {v[i].x, v[i].y, v[i].z, v[i].w, v[i + 1].x, v[i + 1].y, v[i + 1].z, v[i + 1].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t h0, l0, h1, l1;
          split2(__uint_as_float(w8[2 * k] << 16) * pre, __uint_as_float(w8[2 * k] & 0xFFFF0000u) * pre, h0, l0);
          split2(__uint_as_float(w8[2 * k + 1] << 16) * pre, __uint_as_float(w8[2 * k + 1] & 0xFFFF0000u) * pre, h1, l1);
          hi[k] = h0 | (h1 << 16);
          lo[k] = l0 | (l1 << 16);
        }
        const int ch = 4 * (part & 1) + (i >> 1);
        sts128(qs + pn * kQPanel + sw128_chunk(32, h, ch) - (ch >> 3) * 32 * 128,
               make_uint4(hi[0], hi[1], hi[2], hi[3]));
        sts128(qs + pn * kQPanel + sw128_chunk(32, 16 + h, ch) - (ch >> 3) * 32 * 128,
               make_uint4(lo[0], lo[1], lo[2], lo[3]));
      }
      sts128(qs + kQRope + sw128_chunk(HG, h, part), rope);
      if (part == 0) pre_ring[(seg & 3) * HG + h] = ldexpf(1.f, -sh);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarQFull + qb]);
      ++seg;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor-core issuer
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_qk8 = idesc_e4m3(128, 32, 0, 0);
      constexpr uint32_t id_qkr = make_idesc_bf16(128, HG, 0, 0);
      constexpr uint32_t id_pv = idesc_e4m3(128, 32, 1, 1);
      const uint32_t kv0 = smem_u32(smem + kOffKv), q0 = smem_u32(smem + kOffQ), p0 = smem_u32(smem + kOffP);
      int seg_q = 0, seg_o = 0, next_qk = 0, next_pv = 0;
      uint64_t t_idle = 0;
      while (next_pv < n_local) {
        bool progressed = false;
        if (next_qk < n_local && next_qk < next_pv + 2) {
          const int tl = next_qk;
          const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
          const int b = tl & 1;
          const int seg = ti.seg_start ? seg_q : seg_q - 1;
          const int qb = seg & 1;
          const bool q_ok = !ti.seg_start || mbar_test_wait(&bars[kBarQFull + qb], (seg >> 1) & 1);
          if (q_ok && mbar_test_wait(&bars[kBarKvFull + b], (tl >> 1) & 1)) {
            if (ti.seg_start) ++seg_q;
            tc_fence_after();
            const uint32_t kv = kv0 + b * kKvBuf, qs = q0 + qb * kQBuf;
            const uint32_t sb = tmem + b * kSCols;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint64_t da = make_sdesc(kv + g * kPanel + 32 * k, 16, 1024, kLayoutSw128);
                const uint64_t db = make_sdesc(qs + g * kQPanel + 32 * k, 16, 1024, kLayoutSw128);
                mma_f8(sb + 32 * g, da, db, id_qk8, k > 0 ? 1u : 0u);
              }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t da = make_sdesc(kv + kKvRope + 32 * k, 16, 1024, kLayoutSw128);
              const uint64_t db = make_sdesc(qs + kQRope + 32 * k, 16, 1024, kLayoutSw128);
              mma_ss(sb + 128, da, db, id_qkr, k > 0 ? 1u : 0u);
            }
            mma_commit(&bars[kBarSFull + b]);
            if (ti.seg_end) mma_commit(&bars[kBarQEmpty + qb]);
            ++next_qk;
            progressed = true;
          }
        }
        if (next_pv < next_qk) {
          const int tl = next_pv;
          const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
          const int b = tl & 1;
          const bool o_ok = !ti.seg_start || seg_o == 0 || mbar_test_wait(&bars[kBarOFree], (seg_o - 1) & 1);
          if (o_ok && mbar_test_wait(&bars[kBarPFull], tl & 1)) {
            if (ti.seg_start) ++seg_o;
            tc_fence_after();
            const uint32_t kv = kv0 + b * kKvBuf;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                // A = codes^T (value column c x row j), MN-major; B = P'_q (row j x 32), MN-major
                const uint64_t da = make_sdesc(kv + q * kPanel + 4096 * k, kPanel, 1024, kLayoutSw128);
                const uint64_t db = make_sdesc(p0 + q * kPGroup + 1024 * k, 256, 128, kLayoutNone);
                mma_f8(tmem + kOCol + 32 * q, da, db, id_pv, (ti.seg_start && k == 0) ? 0u : 1u);
              }
            }
            mma_commit(&bars[kBarKvEmpty + b]);
            mma_commit(&bars[kBarPvDone]);
            ++next_pv;
            progressed = true;
          }
        }
        if (progressed) {
          t_idle = 0;
        } else {
          if (*abort_flag) break;
          const uint64_t now = globaltimer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > kWaitLimitNs) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, kDevWaitTimeout);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue (warps 0..3)
    const int w = warp;
    const int j = tid;  // tile row of this thread's TMEM lane; also the value column within a chunk
    const uint32_t lane_base = (uint32_t)(32 * w) << 16;
    const uint32_t p0 = smem_u32(smem + kOffP);
    float* red_max = reinterpret_cast<float*>(smem + kOffRedMax);
    float* red_sc = reinterpret_cast<float*>(smem + kOffRedSc);
    float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
    float m_used[HG], l_part[HG], ip[HG], Rq[4];
    int seg = -1, seg_first_kt = 0, n_seg_tiles = 0;
    bool dead = false;
    for (int tl = 0; tl < n_local; ++tl) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      const int b = tl & 1;
      if (ti.seg_start) {
        ++seg;
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          m_used[h] = -INFINITY;
          l_part[h] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) Rq[g] = 0.f;
        seg_first_kt = ti.kt;
        n_seg_tiles = 0;
      }
      if (!dead) dead = !SMLA_WAIT(kBarSFull + b, (tl >> 1) & 1);
      if (!dead) dead = !SMLA_WAIT(kBarKvFull + b, (tl >> 1) & 1);  // row flags and scales
      tc_fence_after();
      if (ti.seg_start) {
#pragma unroll
        for (int h = 0; h < HG; ++h) ip[h] = pre_ring[(seg & 3) * HG + h];
      }
      const bool row_ok = !dead && valid[b * kRows + j] != 0;
      float sc[4];
      {
        const float4 v4 =
            *reinterpret_cast<const float4*>(smem + kOffKv + b * kKvBuf + kKvScale + (j >> 2) * 128 + (j & 3) * 16);
        sc[0] = row_ok ? v4.x : 0.f;
        sc[1] = row_ok ? v4.y : 0.f;
        sc[2] = row_ok ? v4.z : 0.f;
        sc[3] = row_ok ? v4.w : 0.f;
      }
      // logits (log2 units): 2^-s_h sum_g scale_g (S_g,hi + S_g,lo) + S_rope
      float sl[HG];
      {
        const uint32_t sa = tmem + lane_base + b * kSCols;
        float acc[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) acc[h] = 0.f;
        if (!dead) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t hi[16], lo[16];
            tmem_ld16(sa + 32 * g, hi);
            tmem_ld16(sa + 32 * g + 16, lo);
            tmem_ld_wait();
            reg_fence16(hi);
            reg_fence16(lo);
#pragma unroll
            for (int h = 0; h < HG; ++h) acc[h] = fmaf(sc[g], __uint_as_float(hi[h]) + __uint_as_float(lo[h]), acc[h]);
          }
          uint32_t rp[16];
          tmem_ld16_sync(sa + 128, rp);
#pragma unroll
          for (int h = 0; h < HG; ++h) acc[h] = fmaf(acc[h], ip[h], __uint_as_float(rp[h]));
        }
#pragma unroll
        for (int h = 0; h < HG; ++h) sl[h] = row_ok ? acc[h] * p.scale_log2 : -INFINITY;
      }
      // tile maxima: per head (logits) and per scale group (scales), across the 128 rows
      float* redm = red_max + (tl & 1) * 4 * HG;
      float* reds = red_sc + (tl & 1) * 4 * 4;
      {
        float v[16];
#pragma unroll
        for (int h = 0; h < HG; ++h) v[h] = sl[h];
        const float mx = warp_reduce16<true>(v, lane);
        if ((lane & 1) == 0) redm[w * HG + (lane >> 1)] = mx;
        float s4[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
          for (int g = 0; g < 4; ++g) s4[g] = fmaxf(s4[g], __shfl_xor_sync(kFullMask, s4[g], off));
        if (lane == 0)
#pragma unroll
          for (int g = 0; g < 4; ++g) reds[w * 4 + g] = s4[g];
      }
      named_bar_sync(1, 128);
      bool rescale = false;
      float alpha[HG], beta[4];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float tmax = fmaxf(fmaxf(redm[h], redm[HG + h]), fmaxf(redm[2 * HG + h], redm[3 * HG + h]));
        const float nm = fmaxf(m_used[h], tmax);
        alpha[h] = 1.f;
        if (nm > m_used[h] + kMaxSlack) {
          alpha[h] = exp2f(m_used[h] - nm);
          m_used[h] = nm;
          rescale = true;
        }
        l_part[h] *= alpha[h];
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float smax = fmaxf(fmaxf(reds[g], reds[4 + g]), fmaxf(reds[8 + g], reds[12 + g]));
        beta[g] = 1.f;
        if (smax > Rq[g]) {
          const float rn = pow2_ceil(smax);
          if (Rq[g] > 0.f) {
            beta[g] = Rq[g] / rn;
            rescale = true;
          }
          Rq[g] = rn;
        }
      }
      if (rescale && n_seg_tiles > 0 && !dead) {
        // O^T holds this segment's earlier P.V: wait for the latest and rescale in place
        dead = !SMLA_WAIT(kBarPvDone, (tl - 1) & 1);
        if (!dead) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              uint32_t o[16];
              const uint32_t addr = tmem + lane_base + kOCol + 32 * q + 16 * half;
              tmem_ld16_sync(addr, o);
#pragma unroll
              for (int h = 0; h < HG; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h] * beta[q]);
              tmem_st16(addr, o);
            }
          }
          tmem_st_wait();
        }
      }
      // probabilities, running sums, P'_q = p * scale_q / R_q as e4m3 hi + lo
      float pr[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        pr[h] = row_ok ? exp2f(sl[h] - m_used[h]) : 0.f;
        l_part[h] += pr[h];
      }
      if (tl >= 1 && !dead) dead = !SMLA_WAIT(kBarPvDone, (tl - 1) & 1);  // P buffer free
      if (!dead) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float f = Rq[g] > 0.f ? kPScale * sc[g] / Rq[g] : 0.f;
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t h0, l0, h1, l1;
            split2(pr[4 * k] * f, pr[4 * k + 1] * f, h0, l0);
            split2(pr[4 * k + 2] * f, pr[4 * k + 3] * f, h1, l1);
            hi[k] = h0 | (h1 << 16);
            lo[k] = l0 | (l1 << 16);
          }
          // MN-major core matrices: 8 rows x 16 codes; code blocks 128 B apart, row blocks 256 B apart
          const uint32_t base = p0 + g * kPGroup + (j >> 3) * 256 + (j & 7) * 16;
          sts128(base, make_uint4(hi[0], hi[1], hi[2], hi[3]));
          sts128(base + 128, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(&bars[kBarPFull]);
      ++n_seg_tiles;

      if (ti.seg_end) {
        {
          float v[16];
#pragma unroll
          for (int h = 0; h < HG; ++h) v[h] = l_part[h];
          const float sm = warp_reduce16<false>(v, lane);
          if ((lane & 1) == 0) red_sum[w * HG + (lane >> 1)] = sm;
        }
        named_bar_sync(1, 128);
        if (!dead) dead = !SMLA_WAIT(kBarPvDone, tl & 1);  // last P.V of the segment
        tc_fence_after();
        const bool full = (seg_first_kt == 0) && (ti.kt == p.nt - 1);
        const int64_t slot = (int64_t)blockIdx.x + ti.u;
        float inv[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float lt = red_sum[h] + red_sum[HG + h] + red_sum[2 * HG + h] + red_sum[3 * HG + h];
          inv[h] = lt > 0.f ? 1.f / lt : 0.f;
          if (tid == h) {
            const float lse_v = lt > 0.f ? (m_used[h] + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
            if (full)
              p.lse[(int64_t)ti.t * p.H + ti.hg * HG + h] = lse_v;
            else
              p.part_lse[slot * HG + h] = lse_v;
          }
        }
        if (!dead) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t ohi[16], olo[16];
            tmem_ld16(tmem + lane_base + kOCol + 32 * q, ohi);
            tmem_ld16(tmem + lane_base + kOCol + 32 * q + 16, olo);
            tmem_ld_wait();
            reg_fence16(ohi);
            reg_fence16(olo);
            const int c = 128 * q + j;
#pragma unroll
            for (int h = 0; h < HG; ++h) {
              const float val = (__uint_as_float(ohi[h]) + __uint_as_float(olo[h])) * (Rq[q] * kPScaleInv) * inv[h];
              if (full)
                p.out[((int64_t)ti.t * p.H + ti.hg * HG + h) * kDv + c] = __float2bfloat16_rn(val);
              else
                p.part_o[(slot * HG + h) * kDv + c] = val;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !dead) mbar_arrive(&bars[kBarOFree]);
      }
    }
  }
#undef SMLA_WAIT

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

}  // namespace

// Tensor maps of the cache viewed as a 2-D byte array [NB*64 rows, 656 bytes]:
// 128-byte boxes with the 128-byte swizzle (codes, RoPE) and 16-byte boxes
// without swizzle (scales).
cudaError_t make_cache_maps(const uint8_t* cache, int64_t NB, CUtensorMap* row_map, CUtensorMap* scale_map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gdim[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)(NB * kBlock)};
  const cuuint64_t gstride[1] = {(cuuint64_t)kRowBytes};
  const cuuint32_t box_row[2] = {128, 1}, box_scale[2] = {16, 1}, es[2] = {1, 1};
  CUresult r = enc(row_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(cache), gdim, gstride, box_row, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  r = enc(scale_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(cache), gdim, gstride, box_scale, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

AttnPlan plan_decode_fp8(int T, int H, int K, int num_splits, int num_sms) {
  AttnPlan pl;
  pl.HG = HG;
  pl.n_hg = H / HG;
  pl.nt = K > 0 ? (K + kRows - 1) / kRows : 1;
  pl.units = (int64_t)T * pl.n_hg;
  pl.total = pl.units * pl.nt;
  int64_t G = num_splits > 0 ? pl.units * (int64_t)num_splits : (int64_t)num_sms;
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  const size_t lse_bytes = (size_t)(((n_slots * HG * 4) + 255) / 256) * 256;
  pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * HG * kDv * 4;
  return pl;
}

cudaError_t launch_decode_fp8(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap row_map, scale_map;
  cudaError_t e = make_cache_maps(a.cache, a.NB, &row_map, &scale_map);
  if (e != cudaSuccess) return e;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int64_t n_slots = (int64_t)plan.G + plan.units - 1;
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.indices = a.indices;
  p.block_table = a.block_table;
  p.req_id = a.req_id;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = reinterpret_cast<int*>(ws);
  p.part_lse = reinterpret_cast<float*>(ws + kWsStatusBytes);
  p.part_o = reinterpret_cast<float*>(ws + kWsStatusBytes + ((n_slots * HG * 4 + 255) / 256) * 256);
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.T = a.T;
  p.H = a.H;
  p.K = a.K;
  p.R = a.R;
  p.MB = a.MB;
  p.NB = a.NB;
  p.n_hg = plan.n_hg;
  p.nt = plan.nt;
  p.total = plan.total;
  p.G = plan.G;
  sparse_mla_decode_fp8_kernel<<<plan.G, kThreads, kSmemAlloc, stream>>>(p, row_map, scale_map);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  combine_kernel<HG><<<(unsigned)plan.units, 256, 0, stream>>>(p.part_o, p.part_lse, p.out, p.lse, p.H, p.n_hg, p.nt,
                                                               p.total, p.G);
  return cudaGetLastError();
}

}  // namespace smla
