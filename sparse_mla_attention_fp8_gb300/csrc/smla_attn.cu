// BF16 sparse MLA prefill on sm_103a for head counts other than 128 (heads in
// groups of 16 or 32), over a dense [N, 576] bf16 latent buffer; the same
// kernel decodes over the NVFP4 paged cache (kNv: rows dequantized exactly
// into the bf16 operand tiles by the converter warps).
//
// What is computed (vLLM flashmla_sparse.py, FlashMLASparseImpl.forward on
// the prefill path, flash_mla_sparse_prefill): every query token t attends
// with each of its H heads to its own K top-k latent rows (MQA 576/512: all
// heads share the rows; V is the 512-wide NoPE part of each row).  Per head h:
//   s_j   = softmax_scale * <q[t,h,:], row_j>        (576-wide)
//   out   = sum_j softmax(s)_j * row_j[0:512]         (bf16 [T, H, 512])
//   lse   = log(sum_j exp(s_j))                       (fp32 [T, H])
// Indices outside [0, N) are masked; a token with no valid row gets out = 0
// and lse = -inf.
//
// Design (one persistent CTA per SM, warp-specialised, tcgen05 tensor cores):
//  * Work units are (token, head group of HG heads); each unit is K/64 tiles
//    of 64 top-k rows.  The CTAs split the unit-major tile sequence into equal
//    contiguous ranges, so a unit may be split across CTAs ("segments"); a
//    unit finished inside one CTA is written directly, the others go through
//    an LSE-weighted combine kernel.
//  * Index warp: checks tile row indices into a 4-deep shared ring and
//    (re)loads the unit's Q block into shared memory.
//  * Converter warps: stream rows from memory with 16-byte coalesced loads (a
//    warp reads one 1152-byte row per step, 4 rows in flight) and write the
//    K-major, 128-byte-swizzled bf16 operand tile (two tiles are
//    double-buffered).
//  * MMA warp (one thread): S^T = K Q^T with tcgen05.mma (M = 64 rows, N = HG
//    heads, K = 576); O^T += V^T P^T per 128-column value chunk (M = 128,
//    N = HG, K = 64 rows), reading V straight from the same tile as an
//    MN-major operand.  Accumulators live in tensor memory.
//  * Softmax warpgroup (4 warps): online softmax with lazy rescaling of O
//    (only when a running max grows by more than 2^8), P written to shared
//    memory as the B operand of P.V, epilogue.
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "sm103_ptx.cuh"
#include "smla_common.cuh"
#include "smla_combine.cuh"
#include "smla_kernels.h"

namespace smla {

namespace {

constexpr uint32_t kFull = 0xffffffffu;

template <int HG, bool kNv>
struct Cfg {
  static constexpr int kRows = 64;                       // top-k rows per tile
  static constexpr int kPanel = kRows * 128;             // one 64-column panel of the row tile
  static constexpr int kKvTile = 9 * kPanel;             // 576 columns
  static constexpr int kQPanel = HG * 128;
  static constexpr int kQBytes = 9 * kQPanel;
  // Q blocks in flight (next unit prefetched); NVFP4 rows give the room to
  // their staging instead
  static constexpr int kQBufs = (HG == 16 && !kNv) ? 2 : 1;
  static constexpr int kPBytes = kRows * HG * 2;
  static constexpr int kMmaWarp = 4;
  static constexpr int kIndexWarp = 5;
  static constexpr int kConvWarp0 = 6;
  static constexpr int kConvWarps = 10;
  static constexpr int kThreads = 32 * (kConvWarp0 + kConvWarps);
  static constexpr int kDepth = 4;                       // rows in flight per converter warp
  static constexpr int kSCol = 0;                        // S^T buffers: columns [0, 2 * HG)
  static constexpr int kOCol = 2 * HG;                   // O^T: 4 chunks of HG columns
  static constexpr int kColsUsed = kOCol + 4 * HG;
  static constexpr int kTmemCols = kColsUsed <= 128 ? 128 : (kColsUsed <= 256 ? 256 : 512);
  // shared memory layout, offsets from a 1024-byte aligned base
  static constexpr int kOffKv = 0;
  static constexpr int kOffQ = kOffKv + 2 * kKvTile;
  static constexpr int kOffP = kOffQ + kQBufs * kQBytes;
  static constexpr int kOffSlots = kOffP + 2 * kPBytes;  // int32 [4][64]
  static constexpr int kOffValid = kOffSlots + 4 * kRows * 4;  // uint8 [2][64]
  static constexpr int kOffRedMax = kOffValid + 2 * kRows;     // float [2][4][HG]
  static constexpr int kOffRedSum = kOffRedMax + 2 * 4 * HG * 4;  // float [4][HG]
  static constexpr int kOffBar = kOffRedSum + 4 * HG * 4;
  // barriers
  static constexpr int kBarKvFull = 0, kBarKvEmpty = 2, kBarSFull = 4, kBarPFull = 6, kBarPvDone = 8,
                       kBarIdxFull = 10, kBarIdxEmpty = 14, kBarQFull = 18, kBarQEmpty = 20, kBarOFree = 22;
  static constexpr int kNumBars = 23;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  // NVFP4 rows: each converter warp stages its rows of two tiles (up to
  // 2 x kNvRows rows of 352 bytes, then their slots) by cp.async, after the
  // rest of the layout
  static constexpr int kNvRows = (kRows + kConvWarps - 1) / kConvWarps;  // rows of a tile per converter warp, at most
  static constexpr int kOffStage = (kSmemBytes + 127) / 128 * 128;
  static constexpr int kOffStageSlots = kOffStage + kConvWarps * 2 * kNvRows * 352;
  static constexpr int kSmemAllocNv = kOffStageSlots + kConvWarps * 2 * kNvRows * 4 + 1024;
  static_assert(!kNv || (HG == 16 && kSmemAllocNv <= 232448), "NVFP4 rows: 16-head groups, shared memory budget");
  static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "operand tiles must be 1024-byte aligned");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
  static_assert(kColsUsed <= 512, "tensor memory budget");
};

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  const int32_t* indices;
  // NVFP4 rows (kNv): the [NB, 64, 352] cache and its paging; N = NB
  const uint8_t* cache;
  const int32_t* block_table;
  const int32_t* req_id;
  int R, MB;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;
  float* part_lse;
  int* status;
  float scale_log2;
  int T, H, K;
  int64_t N;
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

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}


// Reduce 16 values per lane across the 32 lanes of a warp.  On return every
// lane holds the full reduction of value index (lane >> 1).
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  {
    const bool up = lane & 16;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float send = up ? v[j] : v[j + 8];
      const float keep = up ? v[j + 8] : v[j];
      v[j] = op(keep, __shfl_xor_sync(kFull, send, 16));
    }
  }
  {
    const bool up = lane & 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = up ? v[j] : v[j + 4];
      const float keep = up ? v[j + 4] : v[j];
      v[j] = op(keep, __shfl_xor_sync(kFull, send, 8));
    }
  }
  {
    const bool up = lane & 4;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = up ? v[j] : v[j + 2];
      const float keep = up ? v[j + 2] : v[j];
      v[j] = op(keep, __shfl_xor_sync(kFull, send, 4));
    }
  }
  {
    const bool up = lane & 2;
    const float send = up ? v[0] : v[1];
    const float keep = up ? v[1] : v[0];
    v[0] = op(keep, __shfl_xor_sync(kFull, send, 2));
  }
  v[0] = op(v[0], __shfl_xor_sync(kFull, v[0], 1));
  return v[0];
}

// Optional per-tile timeline for performance work: with SMLA_TRACE defined,
// roles record clock64() at their hand-off points into g_smla_trace_attn (set
// by the host through smla_trace_set_attn).  Compiled out otherwise.
#ifdef SMLA_TRACE
__device__ long long* g_smla_trace_attn = nullptr;
constexpr int kTraceTiles = 64, kTraceEvents = 15;
#define ATTN_TRACE(tl, ev)                                                                                   \
  do {                                                                                                       \
    if (g_smla_trace_attn && (tl) < kTraceTiles)                                                           \
      g_smla_trace_attn[((size_t)blockIdx.x * kTraceTiles + (tl)) * kTraceEvents + (ev)] = clock64();      \
  } while (0)
#else
#define ATTN_TRACE(tl, ev) ((void)0)
#endif
enum { kAEvIdx = 0, kAEvConvIssue, kAEvConvFull, kAEvQk, kAEvSoftStart, kAEvSoftBar, kAEvPFull, kAEvPv, kAEvEpiEnd,
       kAEvEnter, kAEvExit, kAEvPvWait, kAEvConvStart, kAEvConvHalf, kAEvConvLanded };

// An f16 pair -> a bf16 pair (exact for the values used here: at most 6
// significant bits, normal in both formats or zero).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h2) {
  return pack_bf16x2(__half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half((uint16_t)(h2 >> 16))));
}
// Four E2M1 codes (16 bits, value i in nibble i) -> two bf16 pairs, exactly.
// The bf16 bits of the eight magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 are looked
// up with byte permutes (high bytes 00 3F 3F 3F 40 40 40 40, low bytes
// 00 00 80 C0 00 40 80 C0), and each code's sign bit is moved to bit 15 of its
// half.
__device__ __forceinline__ void e2m1x4_to_bf16x2(uint32_t c16, uint32_t& w01, uint32_t& w23) {
  const uint32_t sel = c16 & 0x7777u;
  const uint32_t hi = __byte_perm(0x3F3F3F00u, 0x40404040u, sel);
  const uint32_t lo = __byte_perm(0xC0800000u, 0xC0804000u, sel);
  w01 = __byte_perm(lo, hi, 0x5140) | ((c16 << 12) & 0x8000u) | ((c16 << 24) & 0x80000000u);
  w23 = __byte_perm(lo, hi, 0x7362) | ((c16 << 4) & 0x8000u) | ((c16 << 16) & 0x80000000u);
}
__device__ __forceinline__ uint32_t mul_bf16x2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Eight NVFP4 NoPE values (four code bytes) times their block scale (an E4M3
// byte) -> one 16-byte chunk of bf16 values, exactly: code * scale has at most
// 6 significant bits and lies in [2^-10, 2688] or is 0, so the bf16 product is
// exact.
__device__ __forceinline__ uint4 nvfp4_chunk(uint32_t codes, uint32_t scale_byte) {
  uint32_t sc2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(sc2) : "h"((uint16_t)(scale_byte * 0x0101u)));
  const uint32_t s2 = f16x2_to_bf16x2(sc2);  // the scale in both halves, exact
  uint32_t o[4];
  e2m1x4_to_bf16x2(codes & 0xFFFFu, o[0], o[1]);
  e2m1x4_to_bf16x2(codes >> 16, o[2], o[3]);
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = mul_bf16x2_rn(o[k], s2);
  return make_uint4(o[0], o[1], o[2], o[3]);
}
// Eight E4M3 RoPE values (two words) -> one 16-byte chunk of bf16 values (exact).
__device__ __forceinline__ uint4 e4m3x8_chunk(uint32_t w0, uint32_t w1) {
  const uint32_t w[2] = {w0, w1};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(w[k >> 1] >> (16 * (k & 1)))));
    o[k] = f16x2_to_bf16x2(h2);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// kNv: the rows are NVFP4 cache rows (352 bytes, paged through the block
// table) instead of bf16 latent rows; they are dequantized exactly into the
// same bf16 operand tiles.
template <int HG, bool kNv>
__global__ void __launch_bounds__(Cfg<HG, kNv>::kThreads, 1) sparse_mla_attn_kernel(const __grid_constant__ Params p) {
  using C = Cfg<HG, kNv>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  grid_launch_dependents();  // the combine may be launched behind this grid right away
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + C::kOffSlots);
  uint8_t* valid = smem + C::kOffValid;
  float* red_max = reinterpret_cast<float*>(smem + C::kOffRedMax);
  float* red_sum = reinterpret_cast<float*>(smem + C::kOffRedSum);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t xbeg = tile_begin(blockIdx.x, p.total, p.G);
  const int64_t xend = tile_begin(blockIdx.x + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);
  if (tid == 0) ATTN_TRACE(0, kAEvEnter);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[C::kBarKvFull + i], C::kConvWarps);
      mbar_init(&bars[C::kBarKvEmpty + i], 1);
      mbar_init(&bars[C::kBarSFull + i], 1);
      mbar_init(&bars[C::kBarPFull + i], 4);
      mbar_init(&bars[C::kBarPvDone + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[C::kBarIdxFull + i], 32);
      mbar_init(&bars[C::kBarIdxEmpty + i], C::kConvWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[C::kBarQFull + i], 32);
      mbar_init(&bars[C::kBarQEmpty + i], 1);
    }
    mbar_init(&bars[C::kBarOFree], 4);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

#define SMLA_WAIT(bar_idx, parity) mbar_wait(&bars[(bar_idx)], (parity), abort_flag, p.status, kDevWaitTimeout)

  if (warp == C::kIndexWarp) {
    // ------------------------------------------------------------ index warp
    int seg = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      const int b4 = tl & 3;
      if (tl >= 4 && !SMLA_WAIT(C::kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
      int32_t* slots = slots_ring + b4 * C::kRows;
      for (int r = lane; r < C::kRows; r += 32) {
        const int k = ti.kt * C::kRows + r;
        int32_t s = -1;
        if (k < p.K) {
          const int32_t idx = __ldg(p.indices + (int64_t)ti.t * p.K + k);
          if constexpr (kNv)
            s = translate_slot(idx, __ldg(p.req_id + ti.t), p.block_table, p.R, p.MB, p.N);
          else
            s = (idx >= 0 && (int64_t)idx < p.N) ? idx : -1;
        }
        slots[r] = s;
      }
      mbar_arrive(&bars[C::kBarIdxFull + b4]);
      if (lane == 0) ATTN_TRACE(tl, kAEvIdx);
      if (ti.seg_start) {
        const int qb = seg % C::kQBufs;
        if (seg >= C::kQBufs && !SMLA_WAIT(C::kBarQEmpty + qb, ((seg / C::kQBufs) - 1) & 1)) break;
        const __nv_bfloat16* qsrc = p.q + ((int64_t)ti.t * p.H + (int64_t)ti.hg * HG) * kDqk;
        const uint32_t qbase = smem_u32(smem + C::kOffQ + qb * C::kQBytes);
        // all 16-byte chunks in flight at once (asynchronous copies), then one wait
        for (int i = lane; i < HG * 72; i += 32) {
          const int h = i / 72, ch = i - h * 72;
          cp_async16(qbase + sw128_chunk(HG, h, ch), qsrc + (int64_t)h * kDqk + ch * 8);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&bars[C::kBarQFull + qb]);
        ++seg;
      }
    }
  } else if (kNv && warp >= C::kConvWarp0) {
    // ------------------------------------------------------------ NVFP4 converters
    // Converter warp cw handles rows cw, cw + 10, ... of every tile (RW rows).
    // Two tiles ahead, it copies them as stored (22 chunks of 16 bytes each)
    // by cp.async into its staging half for that tile (one commit group per
    // tile); once a tile's rows have landed and its operand buffer is free,
    // lane l dequantizes output chunks l and l + 32 (and RoPE chunk l for
    // l < 8) of every row into the bf16 tile.
    const int cw = warp - C::kConvWarp0;
    const int RW = (C::kRows - cw + C::kConvWarps - 1) / C::kConvWarps;
    uint8_t* stage = smem + C::kOffStage + cw * 2 * C::kNvRows * 352;
    int32_t* stage_slot = reinterpret_cast<int32_t*>(smem + C::kOffStageSlots) + cw * 2 * C::kNvRows;
    bool ok = true;
    auto issue_tile = [&](int tl) {
      if (tl < n_local && ok) {
        const int b4 = tl & 3, half = tl & 1;
        ok = SMLA_WAIT(C::kBarIdxFull + b4, (tl >> 2) & 1);
        if (ok) {
          if (cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvIssue);
          for (int k = 0; k < RW; ++k) {
            const int32_t slot = slots_ring[b4 * C::kRows + cw + k * C::kConvWarps];
            if (lane == 0) stage_slot[half * C::kNvRows + k] = slot;
            if (slot >= 0 && lane < 22)
              cp_async16(smem_u32(stage + (half * C::kNvRows + k) * 352 + 16 * lane),
                         p.cache + (int64_t)slot * 352 + 16 * lane);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[C::kBarIdxEmpty + b4]);
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    issue_tile(0);
    issue_tile(1);
    for (int tl = 0; tl < n_local && ok; ++tl) {
      const int b = tl & 1, half = tl & 1;
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      __syncwarp();  // the tile's rows have landed for every lane of the warp
      if (cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvLanded);
      if (tl >= 2 && !(ok = SMLA_WAIT(C::kBarKvEmpty + b, ((tl >> 1) + 1) & 1))) break;
      if (cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvStart);
      const uint32_t tile = smem_u32(smem + C::kOffKv + b * C::kKvTile);
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int k = 0; k < C::kNvRows; ++k) {
        if (k < RW) {
          const int r = cw + k * C::kConvWarps;
          const uint8_t* row = stage + (half * C::kNvRows + k) * 352;
          const bool v = stage_slot[half * C::kNvRows + k] >= 0;
          uint4 c0 = z, c1 = z, c2 = z;
          if (v) {
            c0 = nvfp4_chunk(*reinterpret_cast<const uint32_t*>(row + 4 * lane), row[256 + (lane >> 1)]);
            c1 = nvfp4_chunk(*reinterpret_cast<const uint32_t*>(row + 128 + 4 * lane), row[272 + (lane >> 1)]);
            if (lane < 8) {
              const uint2 rr = *reinterpret_cast<const uint2*>(row + 288 + 8 * lane);
              c2 = e4m3x8_chunk(rr.x, rr.y);
            }
          }
          sts128(tile + sw128_chunk(C::kRows, r, lane), c0);
          sts128(tile + sw128_chunk(C::kRows, r, lane + 32), c1);
          if (lane < 8) sts128(tile + sw128_chunk(C::kRows, r, lane + 64), c2);
          if (lane == 0) valid[b * C::kRows + r] = v ? 1 : 0;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();  // every lane has written its chunks and read the staging half
      if (lane == 0) mbar_arrive(&bars[C::kBarKvFull + b]);
      if (cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvFull);
      issue_tile(tl + 2);
    }
    // no copy may still be landing in shared memory when the CTA exits
    cp_async_wait_all();
  } else if (warp >= C::kConvWarp0) {
    // ------------------------------------------------------------ converters
    const int cw = warp - C::kConvWarp0;
    const int RW = (C::kRows - cw + C::kConvWarps - 1) / C::kConvWarps;  // rows of each tile handled here
    const int n_items = n_local * RW;
    struct Raw {
      uint4 a, b, c;  // three 16-byte chunks of the row
      int32_t slot;
    };
    Raw buf[C::kDepth];
    bool ok = true;

    auto issue = [&](int m, Raw& rb) {
      const int tl = m / RW, k = m - tl * RW;
      const int r = cw + k * C::kConvWarps;
      const int b4 = tl & 3;
      if (k == 0) ok = ok && SMLA_WAIT(C::kBarIdxFull + b4, (tl >> 2) & 1);
      if (!ok) return;
      if (k == 0 && cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvIssue);
      const int32_t slot = slots_ring[b4 * C::kRows + r];
      if (k == RW - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::kBarIdxEmpty + b4]);
      }
      rb.slot = slot;
      if (slot >= 0) {
        const uint8_t* row = reinterpret_cast<const uint8_t*>(p.kv + (int64_t)slot * kDqk);
        rb.a = ld_stream(row + 16 * lane);
        rb.b = ld_stream(row + 16 * (lane + 32));
        if (lane < 8) rb.c = ld_stream(row + 16 * (lane + 64));
      }
    };

    auto convert = [&](int m, Raw& rb) {
      const int tl = m / RW, k = m - tl * RW;
      const int r = cw + k * C::kConvWarps;
      const int b = tl & 1;
      if (k == 0 && tl >= 2) ok = ok && SMLA_WAIT(C::kBarKvEmpty + b, ((tl >> 1) + 1) & 1);
      if (!ok) return;
      if (k == 0 && cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvStart);
      if (k == 3 && cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvHalf);
      const uint32_t tile = smem_u32(smem + C::kOffKv + b * C::kKvTile);
      const bool v = rb.slot >= 0;
      const uint4 z = make_uint4(0, 0, 0, 0);
      sts128(tile + sw128_chunk(C::kRows, r, lane), v ? rb.a : z);
      sts128(tile + sw128_chunk(C::kRows, r, lane + 32), v ? rb.b : z);
      if (lane < 8) sts128(tile + sw128_chunk(C::kRows, r, lane + 64), v ? rb.c : z);
      if (lane == 0) valid[b * C::kRows + r] = v ? 1 : 0;
      if (k == RW - 1) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::kBarKvFull + b]);
        if (cw == 0 && lane == 0) ATTN_TRACE(tl, kAEvConvFull);
      }
    };

#pragma unroll
    for (int j = 0; j < C::kDepth; ++j)
      if (j < n_items) issue(j, buf[j]);
    for (int base = 0; base < n_items && ok; base += C::kDepth) {
#pragma unroll
      for (int j = 0; j < C::kDepth; ++j) {
        const int m = base + j;
        if (m < n_items) {
          convert(m, buf[j]);
          if (m + C::kDepth < n_items) issue(m + C::kDepth, buf[j]);
        }
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues every tensor-core op.  It polls (never blocks on) the
    // two inputs it can consume: the next P operand for P.V, checked first
    // because its completion frees an operand tile, and the next converted
    // tile for QK^T (which may run up to two tiles ahead of P.V, one per S
    // buffer).
    if (lane == 0 && n_local > 0) {
      int seg_q = 0, seg_o = 0;  // segments whose first QK^T / first P.V was issued
      constexpr uint32_t idesc_qk = make_idesc_bf16(64, HG, 0, 0);
      constexpr uint32_t idesc_pv = make_idesc_bf16(128, HG, 1, 1);
      constexpr uint32_t pkb = HG * 16;  // bytes per 8-row block of P^T
      const uint32_t kv_base = smem_u32(smem + C::kOffKv);
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      const uint32_t p_base = smem_u32(smem + C::kOffP);
      int next_qk = 0, next_pv = 0;
      uint64_t t_idle = 0;
      while (next_pv < n_local) {
        bool progressed = false;
        // ---- P.V of tile next_pv: needs its P operands (and, for a segment's
        // first tile, the previous segment's epilogue to have read O)
        if (next_pv < next_qk) {
          const int tl = next_pv;
          const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
          const int b = tl & 1;
          const bool o_ok = !ti.seg_start || seg_o == 0 || mbar_test_wait(&bars[C::kBarOFree], (seg_o - 1) & 1);
          if (o_ok && mbar_test_wait(&bars[C::kBarPFull + b], (tl >> 1) & 1)) {
            if (ti.seg_start) ++seg_o;
            tc_fence_after();
            const uint32_t kv = kv_base + b * C::kKvTile;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t pb = p_base + b * C::kPBytes;
#pragma unroll
              for (int s = 0; s < 4; ++s) {
                const uint64_t da = make_sdesc(kv + 2 * q * C::kPanel + s * 2048, C::kPanel, 1024, kLayoutSw128);
                const uint64_t db = make_sdesc(pb + 2 * s * pkb, pkb, 128, kLayoutNone);
                mma_ss(tmem + C::kOCol + q * HG, da, db, idesc_pv, (ti.seg_start && s == 0) ? 0u : 1u);
              }
            }
            mma_commit(&bars[C::kBarKvEmpty + b]);
            mma_commit(&bars[C::kBarPvDone + b]);
            ATTN_TRACE(tl, kAEvPv);
            ++next_pv;
            progressed = true;
          }
        }
        // ---- QK^T of tile next_qk: needs its tile, its Q block and a free S buffer
        if (next_qk < n_local && next_qk < next_pv + 2) {
          const int tl = next_qk;
          const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
          const int b = tl & 1;
          const int seg = ti.seg_start ? seg_q : seg_q - 1;
          const int qb = seg % C::kQBufs;
          const bool q_ok = !ti.seg_start || mbar_test_wait(&bars[C::kBarQFull + qb], (seg / C::kQBufs) & 1);
          if (q_ok && mbar_test_wait(&bars[C::kBarKvFull + b], (tl >> 1) & 1)) {
            if (ti.seg_start) ++seg_q;
            tc_fence_after();
            const uint32_t kv = kv_base + b * C::kKvTile;
            const uint32_t qs = q_base + qb * C::kQBytes;
            const uint32_t sbuf = tmem + C::kSCol + b * HG;
#pragma unroll
            for (int s = 0; s < 36; ++s) {
              const uint32_t off = (s & 3) * 32;
              const uint64_t da = make_sdesc(kv + (s >> 2) * C::kPanel + off, 16, 1024, kLayoutSw128);
              const uint64_t db = make_sdesc(qs + (s >> 2) * C::kQPanel + off, 16, 1024, kLayoutSw128);
              mma_ss(sbuf, da, db, idesc_qk, s == 0 ? 0u : 1u);
            }
            mma_commit(&bars[C::kBarSFull + b]);
            ATTN_TRACE(tl, kAEvQk);
            if (ti.seg_end) mma_commit(&bars[C::kBarQEmpty + qb]);
            ++next_qk;
            progressed = true;
          }
        }
        if (progressed) {
          t_idle = 0;
        } else {
          // bounded idle: give up (and unwind the CTA) if nothing became ready
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
    // ------------------------------------------------------------ softmax warpgroup (warps 0..3)
    const int w = warp;
    const int r = 16 * w + lane;  // tile row held in this thread's TMEM lane (lanes 0..15 only)
    const uint32_t lane_base = (uint32_t)(32 * w) << 16;
    const uint32_t p_base = smem_u32(smem + C::kOffP);
    constexpr int NB16 = HG / 16;
    float m_used[HG], l_part[HG];
    int seg_first_kt = 0, n_seg_tiles = 0;
    bool dead = false;
    for (int tl = 0; tl < n_local; ++tl) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      const int b = tl & 1;
      if (ti.seg_start) {
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          m_used[h] = -INFINITY;
          l_part[h] = 0.f;
        }
        seg_first_kt = ti.kt;
        n_seg_tiles = 0;
      }
      if (!dead) dead = !SMLA_WAIT(C::kBarSFull + b, (tl >> 1) & 1);
      if (!dead) dead = !SMLA_WAIT(C::kBarKvFull + b, (tl >> 1) & 1);  // orders the row-valid flags
      if (tid == 0) ATTN_TRACE(tl, kAEvSoftStart);
      tc_fence_after();
      const bool row_ok = !dead && lane < 16 && valid[b * C::kRows + r] != 0;
      const uint32_t s_addr = tmem + lane_base + C::kSCol + b * HG;
      // scaled logits (log2 units) of head block hb
      auto logits = [&](int hb, float (&sv)[16]) {
        uint32_t a0[16];
        tmem_ld16_sync(s_addr + hb * 16, a0);
#pragma unroll
        for (int j = 0; j < 16; ++j) sv[j] = row_ok ? __uint_as_float(a0[j]) * p.scale_log2 : -INFINITY;
      };
      // pass 1: logits (kept for pass 2) and the per-head maximum of this tile
      float* redm = red_max + (tl & 1) * 4 * HG;
      float sl[NB16][16];
#pragma unroll
      for (int hb = 0; hb < NB16; ++hb) {
        if (!dead) {
          logits(hb, sl[hb]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) sl[hb][j] = -INFINITY;
        }
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = sl[hb][j];
        const float mx = warp_reduce16<true>(v, lane);
        if ((lane & 1) == 0) redm[w * HG + hb * 16 + (lane >> 1)] = mx;
      }
      named_bar_sync(1, 128);
      if (tid == 0) ATTN_TRACE(tl, kAEvSoftBar);
      bool any_rescale = false;
      float alpha[HG];
#pragma unroll
      for (int h = 0; h < HG; ++h) {
        const float tmax = fmaxf(fmaxf(redm[h], redm[HG + h]), fmaxf(redm[2 * HG + h], redm[3 * HG + h]));
        const float nm = fmaxf(m_used[h], tmax);
        alpha[h] = 1.f;
        if (nm > m_used[h] + 8.0f) {
          alpha[h] = exp2f(m_used[h] - nm);
          m_used[h] = nm;
          any_rescale = true;
        }
        l_part[h] *= alpha[h];
      }
      if (any_rescale && n_seg_tiles > 0 && !dead) {
        // O^T holds the P.V of this segment's earlier tiles: wait for the latest, rescale in place.
        dead = !SMLA_WAIT(C::kBarPvDone + ((tl - 1) & 1), ((tl - 1) >> 1) & 1);
        if (!dead) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int hb = 0; hb < NB16; ++hb) {
              uint32_t o[16];
              const uint32_t addr = tmem + lane_base + C::kOCol + q * HG + hb * 16;
              tmem_ld16_sync(addr, o);
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[hb * 16 + j]);
              tmem_st16(addr, o);
            }
          }
          tmem_st_wait();
        }
      }
      // pass 2: probabilities, running sums, P^T rows
      if (tl >= 2 && !dead) dead = !SMLA_WAIT(C::kBarPvDone + b, ((tl >> 1) + 1) & 1);  // P buffers free
      if (tid == 0) ATTN_TRACE(tl, kAEvPvWait);
#pragma unroll
      for (int hb = 0; hb < NB16; ++hb) {
        float pr[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          pr[j] = row_ok ? exp2f(sl[hb][j] - m_used[hb * 16 + j]) : 0.f;
          l_part[hb * 16 + j] += pr[j];
        }
        if (!dead && lane < 16) {
          const uint32_t pbuf = p_base + b * C::kPBytes;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint4 v = make_uint4(pack_bf16x2(pr[8 * e + 0], pr[8 * e + 1]), pack_bf16x2(pr[8 * e + 2], pr[8 * e + 3]),
                                       pack_bf16x2(pr[8 * e + 4], pr[8 * e + 5]), pack_bf16x2(pr[8 * e + 6], pr[8 * e + 7]));
            sts128(pbuf + pt_offset<HG>(r, hb * 16 + 8 * e), v);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(&bars[C::kBarPFull + b]);
      if (tid == 0) ATTN_TRACE(tl, kAEvPFull);
      ++n_seg_tiles;

      if (ti.seg_end) {
        // final sums across the 64 rows
#pragma unroll
        for (int hb = 0; hb < NB16; ++hb) {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = l_part[hb * 16 + j];
          const float sm = warp_reduce16<false>(v, lane);
          if ((lane & 1) == 0) red_sum[w * HG + hb * 16 + (lane >> 1)] = sm;
        }
        named_bar_sync(1, 128);
        if (!dead) dead = !SMLA_WAIT(C::kBarPvDone + b, (tl >> 1) & 1);  // all P.V of the segment done
        tc_fence_after();
        const bool full = (seg_first_kt == 0) && (ti.kt == p.nt - 1);
        const int64_t slot = (int64_t)blockIdx.x + ti.u;  // partial-result slot of this segment
        float inv[HG];
#pragma unroll
        for (int h = 0; h < HG; ++h) {
          const float lt = red_sum[h] + red_sum[HG + h] + red_sum[2 * HG + h] + red_sum[3 * HG + h];
          inv[h] = lt > 0.f ? __fdividef(1.f, lt) : 0.f;  // approximate (a few ulp)
          if (tid == h) {
            const float lse2 = lt > 0.f ? (m_used[h] + __log2f(lt)) : -INFINITY;
            const float lse_v = lse2 * 0.69314718055994530942f;
            if (full) {
              p.lse[(int64_t)ti.t * p.H + ti.hg * HG + h] = lse_v;
            } else {
              p.part_lse[slot * HG + h] = lse_v;
            }
          }
        }
        if (!dead) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = 128 * q + 32 * w + lane;
#pragma unroll
            for (int hb = 0; hb < NB16; ++hb) {
              uint32_t o[16];
              tmem_ld16_sync(tmem + lane_base + C::kOCol + q * HG + hb * 16, o);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int h = hb * 16 + j;
                const float val = __uint_as_float(o[j]) * inv[h];
                if (full) {
                  p.out[((int64_t)ti.t * p.H + ti.hg * HG + h) * kDv + c] = __float2bfloat16_rn(val);
                } else {
                  p.part_o[(slot * HG + h) * kDv + c] = val;
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !dead) mbar_arrive(&bars[C::kBarOFree]);
        if (tid == 0) ATTN_TRACE(tl, kAEvEpiEnd);
      }
    }
  }
#undef SMLA_WAIT

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0) ATTN_TRACE(0, kAEvExit);
}

// Per device, head-group size and row format: the kernel's dynamic shared
// memory limit has been raised (once, thread-safely).
std::once_flag g_attr_once[4][64];
cudaError_t g_attr_err[4][64];

template <int HG, bool kNv>
cudaError_t launch_impl(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  using C = Cfg<HG, kNv>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int hi = (HG == 16 ? 0 : 1) + (kNv ? 2 : 0);
  std::call_once(g_attr_once[hi][dev], [hi, dev] {
    g_attr_err[hi][dev] = cudaFuncSetAttribute(sparse_mla_attn_kernel<HG, kNv>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               kNv ? C::kSmemAllocNv : C::kSmemAlloc);
  });
  if (g_attr_err[hi][dev] != cudaSuccess) return g_attr_err[hi][dev];
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int64_t n_slots = (int64_t)plan.G + plan.units - 1;
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.kv = static_cast<const __nv_bfloat16*>(a.kv);
  p.indices = a.indices;
  p.cache = a.cache;
  p.block_table = a.block_table;
  p.req_id = a.req_id;
  p.R = a.R;
  p.MB = a.MB;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.status = reinterpret_cast<int*>(ws);
  p.part_lse = reinterpret_cast<float*>(ws + kWsStatusBytes);
  p.part_o = reinterpret_cast<float*>(ws + kWsStatusBytes + ((n_slots * HG * 4 + 255) / 256) * 256);
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.T = a.T;
  p.H = a.H;
  p.K = a.K;
  p.N = a.NB;
  p.n_hg = plan.n_hg;
  p.nt = plan.nt;
  p.total = plan.total;
  p.G = plan.G;
  sparse_mla_attn_kernel<HG, kNv><<<plan.G, C::kThreads, kNv ? C::kSmemAllocNv : C::kSmemAlloc, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  e = launch_combine<HG>(p.part_o, p.part_lse, p.out, p.lse, p.H, p.n_hg, p.nt, p.total, p.G, plan.units, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_set_attn(long long* buf) {
  return (int)cudaMemcpyToSymbol(g_smla_trace_attn, &buf, sizeof(buf));
}
#endif

AttnPlan plan_prefill_bf16(int T, int H, int K, int num_splits, int num_sms) {
  if (wide_supported(H)) return plan_prefill_wide(T, K, num_splits, num_sms);
  AttnPlan pl;
  pl.HG = (H % 32 == 0) ? 32 : 16;
  pl.n_hg = H / pl.HG;
  pl.nt = K > 0 ? (K + 63) / 64 : 1;
  pl.units = (int64_t)T * pl.n_hg;
  pl.total = pl.units * pl.nt;
  int64_t G = num_splits > 0 ? pl.units * (int64_t)num_splits : (int64_t)num_sms;
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  const size_t lse_bytes = (size_t)(((n_slots * pl.HG * 4) + 255) / 256) * 256;
  pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * pl.HG * kDv * 4;
  return pl;
}

cudaError_t launch_prefill_bf16(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (plan.HG == 128) return launch_prefill_wide(a, plan, stream);
  return plan.HG == 16 ? launch_impl<16, false>(a, plan, stream) : launch_impl<32, false>(a, plan, stream);
}

bool nvfp4_native_supported(int H) { return !wide_supported(H); }

// The NVFP4 decode runs 16-head groups at every head count below 128 (its row
// staging leaves no room for a 32-head group's Q and P buffers).
AttnPlan plan_decode_nvfp4(int T, int H, int K, int num_splits, int num_sms) {
  AttnPlan pl = plan_prefill_bf16(T, 16, K, num_splits, num_sms);
  pl.n_hg = H / 16;
  pl.units = (int64_t)T * pl.n_hg;
  pl.total = pl.units * pl.nt;
  int64_t G = num_splits > 0 ? pl.units * (int64_t)num_splits : (int64_t)num_sms;
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  const size_t lse_bytes = (size_t)(((n_slots * pl.HG * 4) + 255) / 256) * 256;
  pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * pl.HG * kDv * 4;
  return pl;
}

cudaError_t launch_decode_nvfp4(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (plan.HG != 16) return cudaErrorInvalidValue;
  return launch_impl<16, true>(a, plan, stream);
}

AttnPlan plan_attention(bool fp8, int T, int H, int K, int num_splits, int num_sms) {
  return fp8 ? plan_decode_fp8(T, H, K, num_splits, num_sms) : plan_prefill_bf16(T, H, K, num_splits, num_sms);
}

cudaError_t launch_attention(bool fp8, const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  return fp8 ? launch_decode_fp8(a, plan, stream) : launch_prefill_bf16(a, plan, stream);
}

}  // namespace smla
