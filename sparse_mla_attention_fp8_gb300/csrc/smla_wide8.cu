// FP8 sparse MLA decode with 128 heads on the tensor cores' FP8 path: the
// cache rows' codes feed kind::f8f6f4 MMAs as stored, with no conversion
// (vLLM flashmla_sparse.py: the "FP8 with scale" row format and the FP8
// decode of FlashMLASparseImpl.forward; the query quantized to FP8, as the
// backend of [vLLM PR #59342] does for every quantized cache).
//
// What is computed: for each query token t and each of its 128 heads h,
//   s_j = softmax_scale * <q[t,h,:], K_j>, K_j = [e4m3(c) * scale_j[c/128] for
//         c < 512] ++ RoPE_j (64 bf16),
//   out = sum_j softmax(s)_j * K_j[0:512],  lse = log sum_j exp(s_j),
// over the token's top-k rows (translated through the paged block table).
//
// One cluster of two CTAs per work range (as in the bf16 prefill's kernel):
// CTA c owns the value columns 256 c .. 256 c + 255, i.e. scale groups 2c and
// 2c + 1, and half c of the RoPE part, and computes the part of the logits
// over those features; the two partials are exchanged through distributed
// shared memory (16-bit fixed point).
//  * Q (prepared by a small kernel): per (token, head, scale group) a power of
//    two 2^s_hg puts the group's largest |q| in (224, 448]; q * 2^s_hg =
//    hi + lo in e4m3; RoPE stays bf16.  Per CTA: 4 panels (group x hi/lo) of
//    128 heads x 128 codes, 128-byte swizzle, and a bf16 RoPE half.
//  * Rows: TMA tile::gather4 puts each row's two 128-code runs (one per
//    scale group) straight into two 128-byte-swizzled panels, and its RoPE
//    half into a 64-byte-swizzled panel; the scales come by 16-byte cp.async.
//    Four operand tiles of 64 rows (22 KB each).
//  * QK^T: S_g = Q_g,hi E_g^T + Q_g,lo E_g^T (kind::f8f6f4, M = 128 heads,
//    N = 64 rows, K = 32 per step: 16 MMAs) and the RoPE part in bf16 (2
//    MMAs), into one S buffer of 3 x 64 tensor-memory columns.
//  * Exchange warps combine s = sum_g scale_g 2^-s_hg S_g + S_rope in fp32,
//    trade the partial with the peer CTA, and write the full logits to a
//    64-column logit buffer.
//  * Softmax: lazy running max per head (p <= 2^1.75); P'_g = p * scale_g /
//    R_g * 2^7 with R_g a running power-of-two bound of group g's scales, so
//    P' < 430 sits at the top of e4m3's range, stored as e4m3 hi + lo (A
//    operand, 64-byte swizzle); P.V: O_g += P'_g,hi V_g + P'_g,lo V_g
//    (kind::f8f6f4, M = 128, N = 128, K = 32 per step: 8 MMAs).  O is rescaled
//    in tensor memory when a max or an R_g changes.
//  * Tensor memory: O 256 + S 192 + logits 64 = 512 columns.
// On GB300 this kernel is slower than the f16 kernel of smla_wide.cu: its
// exchange warps, which read and scale three S accumulators per tile, set a
// cadence of about 8.5 K cycles per tile against 6.2 K.
#include <cstdint>
#include <mutex>
#include <cuda.h>
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
constexpr int kHeads = 128;                   // heads per pair = M of every MMA
constexpr int kRows = 64;                     // top-k rows per tile
constexpr int kCodePanel = kRows * 128;       // 8 KB: 64 rows x 128 codes of one scale group
constexpr int kRopePanel = kRows * 64;        // 4 KB: 64 rows x 32 bf16 (this CTA's RoPE half)
constexpr int kTileRope = 2 * kCodePanel;     // offsets inside an operand tile
constexpr int kTileScale = kTileRope + kRopePanel;
constexpr int kKBuf = 22 * 1024;              // 2 code panels, RoPE half, 64 x 16 bytes of scales
constexpr int kKBufs = 4;
constexpr int kQPanel = kHeads * 128;         // 16 KB: 128 heads x 128 e4m3 (one group, hi or lo)
constexpr int kQRope = 4 * kQPanel;           // 128 heads x 32 bf16, 64-byte swizzle
constexpr int kQBuf = kQRope + kHeads * 64;   // 72 KB
constexpr int kPMat = kHeads * kRows;         // 8 KB: one P' matrix, 128 heads x 64 rows e4m3
constexpr int kPBuf = 4 * kPMat;              // (group, hi / lo)
constexpr int kXData = kHeads * 64;           // exchange slot: 16-bit partials, then one fp32 step per head
constexpr int kXSlot = kXData + kHeads * 4;
constexpr int kLoaders = 4;                   // loader lw gathers rows 16 lw .. 16 lw + 15
// Running max of a head: refreshed to kMaxHead above the tile's maximum when
// that maximum exceeds it by more than kMaxSlack (log2 units), so p <= 2^1.75.
constexpr float kMaxSlack = 1.75f, kMaxHead = 0.75f;
// P'_g = p * sc_g / R_g * kPLift: with p <= 2^1.75 and sc_g <= R_g, P' < 430
// stays at the top of e4m3's range (448), as far as it goes from the
// subnormal floor (2^-9) that would otherwise swallow the small weights of a
// group whose bound is set by a few large scales.
constexpr float kPLift = 128.0f;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBuf;
constexpr int kOffP = kOffK + kKBufs * kKBuf;
constexpr int kOffX = kOffP + kPBuf;
constexpr int kOffSlots = kOffX + 2 * kXSlot;                  // int32 [4][64]
constexpr int kOffValid = kOffSlots + 4 * kRows * 4;           // uint8 [kKBufs][64]
// Per tile (two buffers, by tile parity): the halves' logit maxima (float
// [2][128]), the rows' P' factors sc_g kPLift / R_g as f16 pairs (uint32
// [2 groups][32 row pairs]) and the groups' bounds R_g (float [2]).
constexpr int kOffRed = kOffValid + kKBufs * kRows;
constexpr int kRedBytes = 2 * kHeads * 4;
constexpr int kOffRatio = kOffRed + 2 * kRedBytes;
constexpr int kRatioBytes = 2 * 32 * 4;
constexpr int kOffRs = kOffRatio + 2 * kRatioBytes;
constexpr int kOffBar = kOffRs + 2 * 8;
enum {
  kBarKFull = 0, kBarKEmpty = kBarKFull + kKBufs, kBarSFull = kBarKEmpty + kKBufs, kBarSFree = kBarSFull + 1,
  kBarLReady = kBarSFree + 1, kBarLFree = kBarLReady + 1, kBarPFull = kBarLFree + 1, kBarPDone = kBarPFull + 1,
  kBarXFull = kBarPDone + 1, kBarXFree = kBarXFull + 2, kBarIdxFull = kBarXFree + 2, kBarIdxEmpty = kBarIdxFull + 4,
  kBarQFull = kBarIdxEmpty + 4, kBarQEmpty = kBarQFull + 1, kBarOFree = kBarQEmpty + 1, kBarDrain = kBarOFree + 1,
  kBarDrainPv = kBarDrain + 1, kNumBars = kBarDrainPv + 1
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag, merge decision
constexpr int kSmemAlloc = kOffMisc + 16 + 1024;
static_assert(kOffK % 1024 == 0 && kKBuf % 1024 == 0 && kOffP % 1024 == 0 && kQRope % 1024 == 0, "alignment");
static_assert(kTileScale + kRows * 16 <= kKBuf, "operand tile");
static_assert(kOffBar % 8 == 0 && kOffRed % 16 == 0 && kOffRatio % 16 == 0 && kOffX % 16 == 0, "alignment");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// tensor memory columns
constexpr int kOCol = 0;    // O_c: 2 groups x 128 fp32 columns
constexpr int kSCol = 256;  // S: group 0, group 1, RoPE, 64 columns each
constexpr int kLCol = 448;  // the tile's full logits (log2 domain), 64 columns
constexpr int kTmemCols = 512;

constexpr int kSoftWarps = 4, kXchgWarp0 = 4, kXchgWarps = 8, kMmaWarp = 12, kIndexWarp = 13, kLoadWarp0 = 14;
constexpr int kPvWarp = kLoadWarp0 + kLoaders;
constexpr int kNumWarps = kPvWarp + 1;
constexpr int kThreads = 32 * kNumWarps;

struct Params {
  const uint8_t* cache;        // [NB, 64, 656] rows (scales read by cp.async)
  const float* qinv;           // [T, 128, 4]: 2^-s of each (head, group) prescale
  const int32_t* indices;      // [T, K] logical token indices
  const int32_t* block_table;  // [R, MB]
  const int32_t* req_id;       // [T]
  int R, MB;
  __nv_bfloat16* out;          // [T, 128, 512]
  int out_v8;                  // out is 32-byte aligned
  float* lse;                  // [T, 128]
  float* part_o;               // [slots, 128, 512]
  float* part_lse;             // [slots, 128]
  int* merge_flag;             // [T, 2, 2]: in-kernel merge of split tokens (zeroed by the Q preparation)
  float* merge_lse;            // [T, 2, 2, 128]
  int fused;
  int* status;
  float scale_log2;            // softmax_scale * log2(e)
  int T, K;
  int64_t NB;                  // physical 64-row blocks
  int nt;                      // tiles per token
  int64_t total;               // T * nt
  int G;                       // pairs
};

// st.async of 32-bit words into the peer CTA's shared memory, completing `bar`
// (cluster addresses) by the bytes written.
__device__ __forceinline__ void st_async_v4_b32(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(a),
               "r"(bar)
               : "memory");
}
__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// kind::f8f6f4 instruction descriptor, e4m3 A and B, fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// Two floats -> e4m3 hi and lo pairs (low byte from x0), x ~ hi + lo (split in f16x2).
__device__ __forceinline__ void split2_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  uint32_t a, d, r;
  uint16_t t;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(a) : "f"(x1), "f"(x0));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(t) : "r"(a));
  hi = t;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(t));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(d));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(t) : "r"(r));
  lo = t;
}
// An f16 pair -> e4m3 hi and lo pairs (low byte from the low half), x ~ hi + lo.
__device__ __forceinline__ void split_h2(uint32_t a, uint32_t& hi, uint32_t& lo) {
  uint32_t d, r;
  uint16_t t;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(t) : "r"(a));
  hi = t;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(t));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(d));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(t) : "r"(r));
  lo = t;
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float pow2_ceil(float x) {  // smallest power of two >= x (x > 0)
  const uint32_t u = __float_as_uint(x);
  const uint32_t e = u & 0x7F800000u;
  return __uint_as_float((u & 0x007FFFFFu) ? e + 0x00800000u : e);
}
__device__ __forceinline__ float rcp_pow2(float x) { return __uint_as_float(0x7F000000u - __float_as_uint(x)); }
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// the mbarrier counts one arrival once every earlier cp.async of this thread has landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Byte offset of 16-byte chunk `ch` (0..3) of row `r` in a 64-byte-swizzled
// panel of 64-byte rows (the layout a TMA load with 64-byte swizzle writes).
__device__ __forceinline__ uint32_t sw64_chunk(int r, int ch) {
  return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void tile_pos(const Params& p, int64_t x, int& u, int& kt) {
  u = (int)(x / p.nt);
  kt = (int)(x - (int64_t)u * p.nt);
}

// Optional per-tile timeline for performance work: with SMLA_TRACE defined,
// roles record clock64() at their hand-off points into g_smla_trace_wide8
// (set by the host through smla_trace_set_wide8).  Compiled out otherwise.
#ifdef SMLA_TRACE
__device__ long long* g_smla_trace_wide8 = nullptr;
constexpr int kTraceTiles = 64, kTraceEvents = 18;
#define W8_TRACE(tl, ev)                                                                                     \
  do {                                                                                                       \
    if (g_smla_trace_wide8 && (tl) < kTraceTiles)                                                          \
      g_smla_trace_wide8[((size_t)blockIdx.x * kTraceTiles + (tl)) * kTraceEvents + (ev)] = clock64();     \
  } while (0)
#else
#define W8_TRACE(tl, ev) ((void)0)
#endif
enum { kEvIdx = 0, kEvKFull, kEvQk, kEvXS, kEvXSent, kEvXRecv, kEvLReady, kEvSoftL, kEvSoftPDone, kEvPFull, kEvPv,
       kEvLoadIssue, kEvKEmpty, kEvEpiStart, kEvEpiEnd, kEvEnter, kEvExit, kEvQFull };

// Maps: m_code = the cache rows' bytes with 128-byte boxes (128-byte swizzle);
// m_rope = 64-byte boxes (64-byte swizzle); q_map = the prepared Q codes,
// [T x 128 rows, 4 groups x (hi, lo) x 128 bytes], 128-byte boxes of 128
// heads; q_rope_map = the input q's bytes, 64-byte boxes (one RoPE half) of
// 128 heads (64-byte swizzle).
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(96)
    sparse_mla_wide8_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap m_code,
                            const __grid_constant__ CUtensorMap m_rope, const __grid_constant__ CUtensorMap q_map,
                            const __grid_constant__ CUtensorMap q_rope_map) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + kOffSlots);
  uint8_t* valid = smem + kOffValid;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c = (int)cluster_ctarank();  // value half owned by this CTA
  const int pair = blockIdx.x >> 1;
  const int64_t xbeg = tile_begin(pair, p.total, p.G);
  const int64_t xend = tile_begin(pair + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);
  if (threadIdx.x == 0) W8_TRACE(0, kEvEnter);

  if (tid == 0) {
    for (int i = 0; i < kKBufs; ++i) {
      // per loader: one arrival with the bytes of its TMA copies and 16 for its rows' scale copies
      mbar_init(&bars[kBarKFull + i], kLoaders * 17);
      mbar_init(&bars[kBarKEmpty + i], 1);
    }
    mbar_init(&bars[kBarSFull], 1);
    mbar_init(&bars[kBarSFree], kXchgWarps);
    mbar_init(&bars[kBarLReady], kXchgWarps);
    mbar_init(&bars[kBarLFree], kSoftWarps);
    mbar_init(&bars[kBarPFull], kSoftWarps);
    mbar_init(&bars[kBarPDone], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarXFull + i], 1);           // this CTA's expect-tx; the peer's bytes complete it
      mbar_init(&bars[kBarXFree + i], kXchgWarps / 2);  // one arrival per peer exchange warp of the half
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarIdxFull + i], 32);
      mbar_init(&bars[kBarIdxEmpty + i], kLoaders);
    }
    mbar_init(&bars[kBarQFull], 1);
    mbar_init(&bars[kBarQEmpty], 1);
    mbar_init(&bars[kBarOFree], kSoftWarps * 32);
    mbar_init(&bars[kBarDrain], 1);
    mbar_init(&bars[kBarDrainPv], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  // the peer's barriers must be initialised before anything arrives on them
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

#define SMLA_WAIT(bar_idx, parity) mbar_wait(&bars[(bar_idx)], (parity), abort_flag, p.status, kDevWaitTimeout)
#define SMLA_WAIT_X(bar_idx, parity) \
  mbar_wait_cluster(&bars[(bar_idx)], (parity), abort_flag, p.status, kDevWaitTimeout)

  if (warp == kIndexWarp) {
    // ------------------------------------------------------------ index translation + Q
    int seg = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      int u, kt;
      tile_pos(p, xbeg + tl, u, kt);
      const bool seg_start = tl == 0 || kt == 0;
      const int b4 = tl & 3;
      if (tl >= 4 && !SMLA_WAIT(kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
      const int32_t req = __ldg(p.req_id + u);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = lane + 32 * i;
        const int k = kt * kRows + r;
        int32_t sl = -1;
        if (k < p.K) sl = translate_slot(__ldg(p.indices + (int64_t)u * p.K + k), req, p.block_table, p.R, p.MB, p.NB);
        slots_ring[b4 * kRows + r] = sl;
      }
      mbar_arrive(&bars[kBarIdxFull + b4]);
      if (lane == 0) W8_TRACE(tl, kEvIdx);
      if (seg_start) {
        // the segment's Q block, once the previous segment's last QK^T is done
        if (seg >= 1 && !SMLA_WAIT(kBarQEmpty, (seg - 1) & 1)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[kBarQFull], (uint32_t)kQBuf);
          for (int b = 0; b < 4; ++b)  // panel b: group b / 2 of this CTA, hi (b even) or lo
            tma_load_2d(smem_u32(smem + kOffQ + b * kQPanel), &q_map, ((2 * c + (b >> 1)) * 2 + (b & 1)) * 128,
                        u * kHeads, &bars[kBarQFull]);
          tma_load_2d(smem_u32(smem + kOffQ + kQRope), &q_rope_map, 2 * kDv + 64 * c, u * kHeads, &bars[kBarQFull]);
        }
        __syncwarp();
        ++seg;
      }
    }
    // no Q copy may still be landing in shared memory when the CTA exits
    if (seg > 0 && lane == 0) mbar_wait_drain(&bars[kBarQFull], (seg - 1) & 1);
    __syncwarp();
  } else if (warp >= kLoadWarp0 && warp < kPvWarp) {
    // ------------------------------------------------------------ row loaders
    // Loader lw gathers rows 16 lw .. 16 lw + 15 of every tile: 4 groups of 4
    // rows x 3 boxes (the CTA's two 128-code runs, its RoPE half), lane 3 g + b
    // issuing box b of group g, and lanes 0..15 copy their row's 16 bytes of
    // scales.  Invalid rows (slot -1) read as zeros.  Its arrivals on the
    // tile's full barrier: one with the bytes of its TMA copies (after its
    // writes of the rows' valid flags), and one per scale copy as it lands.
    const int lw = warp - kLoadWarp0;
    const int grp = lane / 3, box = lane - grp * 3;
    const int r_g = 16 * lw + 4 * grp;  // tile row of the lane's group
    int last_b = -1, last_use = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      const int b4 = tl & 3, kb = tl % kKBufs, use = tl / kKBufs;
      if (!SMLA_WAIT(kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = lane < 16 ? slots_ring[b4 * kRows + 16 * lw + lane] : -1;
      const int g0 = __shfl_sync(kFullMask, slot, (4 * grp) & 31), g1 = __shfl_sync(kFullMask, slot, (4 * grp + 1) & 31);
      const int g2 = __shfl_sync(kFullMask, slot, (4 * grp + 2) & 31), g3 = __shfl_sync(kFullMask, slot, (4 * grp + 3) & 31);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarIdxEmpty + b4]);
      if (use >= 1 && !SMLA_WAIT(kBarKEmpty + kb, (use + 1) & 1)) break;
      if (lane == 0 && lw == 0) W8_TRACE(tl, kEvKEmpty);
      if (lane < 16) valid[kb * kRows + 16 * lw + lane] = slot >= 0 ? 1 : 0;
      __syncwarp();
      const uint32_t tile = smem_u32(smem + kOffK + kb * kKBuf);
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarKFull + kb], (uint32_t)(16 * (2 * 128 + 64)));
      __syncwarp();
      if (lane < 12) {
        if (box < 2)
          tma_gather4_2d(tile + box * kCodePanel + (uint32_t)((r_g >> 3) * 1024 + (r_g & 7) * 128), &m_code,
                         128 * (2 * c + box), g0, g1, g2, g3, &bars[kBarKFull + kb]);
        else
          tma_gather4_2d(tile + kTileRope + (uint32_t)((r_g >> 3) * 512 + (r_g & 7) * 64), &m_rope,
                         kRopeOff + 64 * c, g0, g1, g2, g3, &bars[kBarKFull + kb]);
      }
      if (lane == 0 && lw == 0) W8_TRACE(tl, kEvLoadIssue);
      if (lane < 16) {
        const int r = 16 * lw + lane;
        const uint8_t* src = slot >= 0 ? p.cache + (int64_t)slot * kRowBytes + kScaleOff : p.cache;
        cp_async_16(tile + kTileScale + 16 * r, src, slot >= 0 ? 16u : 0u);
        cp_async_arrive(&bars[kBarKFull + kb]);
      }
      last_b = kb;
      last_use = use;
    }
    // no copy may still be landing in shared memory when the CTA exits
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (last_b >= 0 && lane == 0) mbar_wait_drain(&bars[kBarKFull + last_b], last_use & 1);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ QK^T issuer
    // One thread: per tile, S_g = Q_g,hi E_g^T + Q_g,lo E_g^T for the CTA's two
    // groups (e4m3 x e4m3, 4 steps of 32 codes each) and S_rope (bf16, 2 steps
    // of 16 values), once the rows, the segment's Q and the S buffer (read by
    // the exchange warps) are there.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_qk = idesc_e4m3(128, kRows, 0, 0);
      constexpr uint32_t id_qkr = make_idesc_bf16(128, kRows, 0, 0);
      // shared-memory descriptors: constant high words, low words = base + offset / 16
      constexpr uint32_t kHi128 = sdesc_hi(1024, kLayoutSw128), kHi64 = sdesc_hi(512, kLayoutSw64);
      const uint32_t dq = sdesc_lo(smem_u32(smem + kOffQ), 16), dk0 = sdesc_lo(smem_u32(smem + kOffK), 16);
      int seg = 0, kt = (int)(xbeg % p.nt), issued = 0;
      for (int tl = 0; tl < n_local; ++tl) {
        const int kb = tl % kKBufs;
        const bool seg_start = tl == 0 || kt == 0;
        const bool seg_end = tl == n_local - 1 || kt == p.nt - 1;
        if (tl >= 1 && !SMLA_WAIT(kBarSFree, (tl - 1) & 1)) break;
        if (seg_start && !SMLA_WAIT(kBarQFull, seg & 1)) break;
        W8_TRACE(tl, kEvQFull);
        if (!SMLA_WAIT(kBarKFull + kb, (tl / kKBufs) & 1)) break;
        W8_TRACE(tl, kEvKFull);
        tc_fence_after();
        const uint32_t dk = dk0 + ((kb * kKBuf) >> 4);
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int s = 0; s < 4; ++s)
              mma_f8(tmem + kSCol + 64 * g, sdesc_join<kHi128>(dq + (((2 * g + hl) * kQPanel + 32 * s) >> 4)),
                     sdesc_join<kHi128>(dk + ((g * kCodePanel + 32 * s) >> 4)), id_qk, (hl | s) != 0 ? 1u : 0u);
#pragma unroll
        for (int s = 0; s < 2; ++s)  // RoPE half: 8-row atoms of 64 bytes
          mma_ss(tmem + kSCol + 128, sdesc_join<kHi64>(dq + ((kQRope + 32 * s) >> 4)),
                 sdesc_join<kHi64>(dk + ((kTileRope + 32 * s) >> 4)), id_qkr, s != 0 ? 1u : 0u);
        mma_commit(&bars[kBarSFull]);
        W8_TRACE(tl, kEvQk);
        if (seg_end) {
          mma_commit(&bars[kBarQEmpty]);
          ++seg;
        }
        ++issued;
        kt = kt + 1 == p.nt ? 0 : kt + 1;
      }
      // every issued tensor-core operation completes before tensor memory is released
      if (issued > 0) {
        mma_commit(&bars[kBarDrain]);
        mbar_wait_drain(&bars[kBarDrain], 0);
      }
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P.V issuer
    // One thread: O_g += P'_g,hi V_g + P'_g,lo V_g once P' is written (and,
    // first in a segment, the previous segment's epilogue has read O).  A =
    // P' (128 heads x 64 rows, K-major, 64-byte swizzle), B = the group's
    // code panel read MN-major (one 128-byte atom wide, 8-row groups 1024
    // bytes apart, 32 rows per step).  Its completion frees the row tile and P'.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_pv = idesc_e4m3(128, 128, 0, 1);
      constexpr uint32_t kHi128 = sdesc_hi(1024, kLayoutSw128), kHi64 = sdesc_hi(512, kLayoutSw64);
      const uint32_t dp = sdesc_lo(smem_u32(smem + kOffP), 16);
      const uint32_t dv0 = sdesc_lo(smem_u32(smem + kOffK), kCodePanel);
      int seg_o = 0, kt = (int)(xbeg % p.nt), issued = 0;
      for (int tl = 0; tl < n_local; ++tl) {
        const int kb = tl % kKBufs;
        const bool seg_start = tl == 0 || kt == 0;
        if (seg_start && seg_o > 0 && !SMLA_WAIT(kBarOFree, (seg_o - 1) & 1)) break;
        if (!SMLA_WAIT(kBarPFull, tl & 1)) break;
        if (seg_start) ++seg_o;
        tc_fence_after();
        const uint32_t dv = dv0 + ((kb * kKBuf) >> 4);
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int s = 0; s < 2; ++s)
              mma_f8(tmem + kOCol + 128 * g, sdesc_join<kHi64>(dp + (((2 * g + hl) * kPMat + 32 * s) >> 4)),
                     sdesc_join<kHi128>(dv + ((g * kCodePanel + 4096 * s) >> 4)), id_pv,
                     (seg_start && hl == 0 && s == 0) ? 0u : 1u);
        mma_commit(&bars[kBarKEmpty + kb]);
        mma_commit(&bars[kBarPDone]);
        W8_TRACE(tl, kEvPv);
        ++issued;
        kt = kt + 1 == p.nt ? 0 : kt + 1;
      }
      if (issued > 0) {
        mma_commit(&bars[kBarDrainPv]);
        mbar_wait_drain(&bars[kBarDrainPv], 0);
      }
    }
    __syncwarp();
  } else {
    const int qd = warp & 3;
    const int h = 32 * qd + lane;  // head = TMEM lane of S, L and O
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    uint32_t* ratio = reinterpret_cast<uint32_t*>(smem + kOffRatio);
    float* rs = reinterpret_cast<float*>(smem + kOffRs);
    if (warp >= kXchgWarp0) {
      // ---------------------------------------------------------- exchange (warps 4..11)
      // Warp group e handles rows 32 e .. 32 e + 31 of every tile: the partial
      // logit over the CTA's features, s_c = 2^-s_h,2c sc_2c S_0 +
      // 2^-s_h,2c+1 sc_2c+1 S_1 + S_rope, goes to the peer as 16-bit fixed
      // point (st.async into its exchange slot e, the bytes completing its
      // barrier: each head's 32 values as q = round(x 32767 / a), a the
      // largest magnitude among them, plus the step a / 32767, so a received
      // value is off by at most 2^-16 a), the peer's partial is added, rows
      // are masked and scaled to the log2 domain and written to the logit
      // buffer with the half's maximum per head.  Every warp also derives the
      // tile's scale bounds R_g (a power of two >= every scale of group g seen
      // in the segment so far, the same in every warp), and one warp per half
      // writes its rows' P' factors sc_g kPLift / R_g.
      const uint32_t peer = (uint32_t)(c ^ 1);
      const uint32_t x_chunk = (uint32_t)(h * 64);
      const uint32_t x_remote = mapa_shared(smem_u32(smem + kOffX), peer);
      const uint32_t xfull_remote = mapa_shared(smem_u32(&bars[kBarXFull]), peer);
      const uint32_t xfree_remote = mapa_shared(smem_u32(&bars[kBarXFree]), peer);
      const int e = (warp - kXchgWarp0) >> 2;
      const bool lead = lane == 0 && qd == 0;  // registers the slot's expected bytes
      bool dead = false;
      float R0 = 0.f, R1 = 0.f;
      int u = (int)(xbeg / p.nt), kt = (int)(xbeg - (int64_t)u * p.nt);
      for (int tl = 0; tl < n_local; ++tl) {
        const bool seg_start = tl == 0 || kt == 0;
        const float2 qa = __ldg(reinterpret_cast<const float2*>(p.qinv + ((int64_t)u * kHeads + h) * 4 + 2 * c));
        if (++kt == p.nt) {
          kt = 0;
          ++u;
        }
        const int kb = tl % kKBufs, rb = tl & 1;
        // row validity and scales (in the tile once its full barrier has completed)
        if (!dead) dead = !SMLA_WAIT(kBarKFull + kb, (tl / kKBufs) & 1);
        uint32_t vb = 0u;
        {
          const uint4* vf = reinterpret_cast<const uint4*>(valid + kb * kRows + 32 * e);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint4 w4 = vf[i];
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              // bytes are 0 or 1: gather bit 0 of each byte
              uint32_t b = w[k] & 0x01010101u;
              b = (b | (b >> 7)) & 0x00030003u;
              b = (b | (b >> 14)) & 0xFu;
              vb |= b << (4 * (4 * i + k));
            }
          }
        }
        const uint8_t* tsc = smem + kOffK + kb * kKBuf + kTileScale + 8 * c;
        const float2 sc_a = *reinterpret_cast<const float2*>(tsc + 16 * lane);
        const float2 sc_b = *reinterpret_cast<const float2*>(tsc + 16 * (32 + lane));
        float m0 = fmaxf(sc_a.x, sc_b.x), m1 = fmaxf(sc_a.y, sc_b.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          m0 = fmaxf(m0, __shfl_xor_sync(kFullMask, m0, o));
          m1 = fmaxf(m1, __shfl_xor_sync(kFullMask, m1, o));
        }
        if (seg_start) R0 = R1 = 0.f;
        R0 = fmaxf(R0, pow2_ceil(m0));
        R1 = fmaxf(R1, pow2_ceil(m1));
        const float2 sc = e ? sc_b : sc_a;  // row 32 e + lane
        if (lead) mbar_arrive_expect_tx(&bars[kBarXFull + e], (uint32_t)kXSlot);
        if (!dead) dead = !SMLA_WAIT(kBarSFull, tl & 1);
        tc_fence_after();
        float s[32];
        {
          const uint32_t scol = tmem + lane_base + kSCol + 32 * e;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            uint32_t r0[8], r1[8], r2[8];
            tmem_ld8(scol + 8 * jj, r0);
            tmem_ld8(scol + 64 + 8 * jj, r1);
            tmem_ld8(scol + 128 + 8 * jj, r2);
            tmem_ld_wait();
            reg_fence8(r0);
            reg_fence8(r1);
            reg_fence8(r2);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int jr = 8 * jj + j;
              const float f0 = qa.x * __shfl_sync(kFullMask, sc.x, jr);
              const float f1 = qa.y * __shfl_sync(kFullMask, sc.y, jr);
              s[jr] = fmaf(f0, __uint_as_float(r0[j]), fmaf(f1, __uint_as_float(r1[j]), __uint_as_float(r2[j])));
            }
          }
        }
        // S is in registers: the next QK^T may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarSFree]);
        if (tid == 32 * kXchgWarp0) W8_TRACE(tl, kEvXS);
        // 16-bit fixed point relative to the largest magnitude (offset binary;
        // fma(x, 32767 / a, 1.5 * 2^23 + 32768) rounds to the nearest integer
        // and leaves the code in its low 16 bits; a code u placed under the
        // exponent of 2^23 reads as 2^23 + u).  Chunk i of head h sits at
        // position (i + h / 2) % 4 of the head's 64 bytes.
        {
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(s[j]));
          const float inv = amax > 0x1p-100f ? __fdividef(32767.f, amax) : 0.f;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = __byte_perm(__float_as_uint(fmaf(s[2 * j], inv, 12615680.f)),
                                __float_as_uint(fmaf(s[2 * j + 1], inv, 12615680.f)), 0x5410);
          if (tl >= 1 && !dead) dead = !SMLA_WAIT_X(kBarXFree + e, (tl - 1) & 1);
          if (!dead) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              st_async_v4_b32(x_remote + e * kXSlot + x_chunk + 16 * ((i + (h >> 1)) & 3), pk[4 * i], pk[4 * i + 1],
                              pk[4 * i + 2], pk[4 * i + 3], xfull_remote + 8 * e);
            st_async_b32(x_remote + e * kXSlot + kXData + 4 * h, __float_as_uint(amax * (1.f / 32767.f)),
                         xfull_remote + 8 * e);
          }
          if (tid == 32 * kXchgWarp0) W8_TRACE(tl, kEvXSent);
        }
        if (!dead) dead = !SMLA_WAIT_X(kBarXFull + e, tl & 1);
        if (tid == 32 * kXchgWarp0) W8_TRACE(tl, kEvXRecv);
        if (!dead) {
          const uint8_t* src = smem + kOffX + e * kXSlot;
          const float step = *reinterpret_cast<const float*>(src + kXData + 4 * h);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + x_chunk + 16 * ((i + (h >> 1)) & 3));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float lo = __uint_as_float(__byte_perm(w[k], 0x4B00u, 0x5410)) - 8421376.f;  // 2^23 + 32768
              const float hi = __uint_as_float(__byte_perm(w[k], 0x4B00u, 0x5432)) - 8421376.f;
              s[8 * i + 2 * k] = fmaf(lo, step, s[8 * i + 2 * k]);
              s[8 * i + 2 * k + 1] = fmaf(hi, step, s[8 * i + 2 * k + 1]);
            }
          }
        }
        // the slot's values are in registers: the peer may overwrite it
        __syncwarp();
        if (!dead && lane == 0) mbar_arrive_cluster_relaxed(xfree_remote + 8 * e);
        float mt = -INFINITY;
        uint32_t r[2][16];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float x = (vb >> j) & 1u ? s[j] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, x);
          r[j >> 4][j & 15] = __float_as_uint(x);
        }
        // the softmax has read the previous tile's logits
        if (tl >= 1 && !dead) dead = !SMLA_WAIT(kBarLFree, (tl - 1) & 1);
        tc_fence_after();
        tmem_st16(tmem + lane_base + kLCol + 32 * e, r[0]);
        tmem_st16(tmem + lane_base + kLCol + 32 * e + 16, r[1]);
        tmem_st_wait();
        red[rb * (2 * kHeads) + e * kHeads + h] = mt;
        if (qd == 0) {
          const float i0 = R0 > 0.f ? rcp_pow2(R0) * kPLift : 0.f, i1 = R1 > 0.f ? rcp_pow2(R1) * kPLift : 0.f;
          const float f0 = sc.x * i0, f1 = sc.y * i1;
          const float f0n = __shfl_down_sync(kFullMask, f0, 1), f1n = __shfl_down_sync(kFullMask, f1, 1);
          if ((lane & 1) == 0) {
            ratio[rb * 64 + 16 * e + (lane >> 1)] = pack_f16x2(f0, f0n);
            ratio[rb * 64 + 32 + 16 * e + (lane >> 1)] = pack_f16x2(f1, f1n);
          }
          if (e == 0 && lane == 0) {
            rs[2 * rb] = R0;
            rs[2 * rb + 1] = R1;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarLReady]);
        if (tid == 32 * kXchgWarp0) W8_TRACE(tl, kEvLReady);
      }
    } else {
      // ---------------------------------------------------------- softmax + epilogue (warps 0..3)
      // Lazy running max per head (O rescaled only when the tile's max exceeds
      // it by more than kMaxSlack), p = 2^(x - m) <= 2^1.75 in f16, P'_g = p * (sc_g
      // kPLift / R_g) split into e4m3 hi + lo.  O_g holds sum_j P'_g,j V_g,j,
      // i.e. kPLift / R_g times the weighted values; a tile that raises R_g
      // takes O_g along by R_old / R_new (a power of two).
      float m_used = -INFINITY, l_sum = 0.f, rp0 = 0.f, rp1 = 0.f;
      int n_seg_tiles = 0;
      bool dead = false;
      int u = (int)(xbeg / p.nt), kt = (int)(xbeg - (int64_t)u * p.nt);
      for (int tl = 0; tl < n_local; ++tl) {
        const bool seg_start = tl == 0 || kt == 0;
        const bool seg_end = tl == n_local - 1 || kt == p.nt - 1;
        const int rb = tl & 1;
        if (seg_start) {
          m_used = -INFINITY;
          l_sum = 0.f;
          rp0 = rp1 = 0.f;
          n_seg_tiles = 0;
        }
        if (!dead) dead = !SMLA_WAIT(kBarLReady, tl & 1);
        tc_fence_after();
        const float mt = fmaxf(red[rb * (2 * kHeads) + h], red[rb * (2 * kHeads) + kHeads + h]);
        const float R0 = rs[2 * rb], R1 = rs[2 * rb + 1];
        const bool need = mt > m_used + kMaxSlack || (m_used == -INFINITY && mt > -INFINITY);
        const bool scale_m = need && n_seg_tiles > 0 && m_used > -INFINITY;
        const float m_new = mt + kMaxHead;
        const float dm = scale_m ? m_used - m_new : 0.f;
        if (need) m_used = m_new;
        const float a_l = scale_m ? ex2_approx(dm) : 1.f;
        // R only grows within a segment (R_new > R_old >= 0 when they differ)
        const float a0 = n_seg_tiles > 0 && R0 != rp0 ? a_l * rp0 * rcp_pow2(R0) : a_l;
        const float a1 = n_seg_tiles > 0 && R1 != rp1 ? a_l * rp1 * rcp_pow2(R1) : a_l;
        rp0 = R0;
        rp1 = R1;
        // p of the tile's 64 rows as f16 pairs (row pair i in p2[i]) and their sum
        const bool none = m_used == -INFINITY;
        uint32_t p2[32];
        float lt = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tmem + lane_base + kLCol + 32 * e, r0);
          tmem_ld16(tmem + lane_base + kLCol + 32 * e + 16, r1);
          tmem_ld_wait();
          reg_fence16(r0);
          reg_fence16(r1);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float x0 = none ? 0.f : ex2_approx(__uint_as_float(r0[2 * j]) - m_used);
            const float x1 = none ? 0.f : ex2_approx(__uint_as_float(r0[2 * j + 1]) - m_used);
            const float x2 = none ? 0.f : ex2_approx(__uint_as_float(r1[2 * j]) - m_used);
            const float x3 = none ? 0.f : ex2_approx(__uint_as_float(r1[2 * j + 1]) - m_used);
            lt += (x0 + x1) + (x2 + x3);
            p2[16 * e + j] = pack_f16x2(x0, x1);
            p2[16 * e + 8 + j] = pack_f16x2(x2, x3);
          }
        }
        // the logits are in registers: the exchange warps may write the next tile's
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarLFree]);
        if (tid == 0) W8_TRACE(tl, kEvSoftL);
        l_sum = l_sum * a_l + lt;
        // P.V(tl - 1) has read P' and added to O
        if (tl >= 1 && !dead) dead = !SMLA_WAIT(kBarPDone, (tl - 1) & 1);
        if (tid == 0) W8_TRACE(tl, kEvSoftPDone);
        tc_fence_after();
        // TMEM access is warp-wide: a warp with any head to rescale runs the pass
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
          const float a = g ? a1 : a0;
          if (!__any_sync(kFullMask, a != 1.f)) continue;
#pragma unroll 1
          for (int q = 0; q < 128 / 16; ++q) {
            uint32_t r[16];
            const uint32_t col = tmem + lane_base + kOCol + 128 * g + 16 * q;
            tmem_ld16_sync(col, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a);
            tmem_st16(col, r);
          }
        }
        // P'_g hi and lo: head h's 64 bytes per matrix, chunk ch = rows 16 ch .. 16 ch + 15
        {
          const uint32_t* rt = ratio + rb * 64;
          const uint32_t pw = smem_u32(smem + kOffP);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              const uint4 fa = *reinterpret_cast<const uint4*>(rt + 32 * g + 8 * ch);
              const uint4 fb = *reinterpret_cast<const uint4*>(rt + 32 * g + 8 * ch + 4);
              const uint32_t f[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
              uint32_t hi[4], lo[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                uint32_t h0, l0, h1, l1;
                split_h2(mul_f16x2(p2[8 * ch + 2 * k], f[2 * k]), h0, l0);
                split_h2(mul_f16x2(p2[8 * ch + 2 * k + 1], f[2 * k + 1]), h1, l1);
                hi[k] = h0 | (h1 << 16);
                lo[k] = l0 | (l1 << 16);
              }
              const uint32_t off = sw64_chunk(h, ch);
              st_shared_v4(pw + (2 * g) * kPMat + off, hi[0], hi[1], hi[2], hi[3]);
              st_shared_v4(pw + (2 * g + 1) * kPMat + off, lo[0], lo[1], lo[2], lo[3]);
            }
          }
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarPFull]);
        if (tid == 0) W8_TRACE(tl, kEvPFull);
        ++n_seg_tiles;
        // epilogue at the end of a segment
        if (seg_end) {
          if (!dead) dead = !SMLA_WAIT(kBarPDone, tl & 1);
          tc_fence_after();
          if (tid == 0) W8_TRACE(tl, kEvEpiStart);
          const bool full_unit = n_seg_tiles == p.nt;  // the whole token ran in this pair
          // out = O_g R_g / (kPLift l)
          // approximate reciprocal and logarithms (a few ulp)
          const float rl = l_sum > 0.f ? __fdividef(1.f, l_sum) : 0.f;
          const float inv0 = rp0 * (1.f / kPLift) * rl;
          const float inv1 = rp1 * (1.f / kPLift) * rl;
          const float lse_v = l_sum > 0.f ? (m_used + __log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
          const int64_t slot = (int64_t)pair + u;
          // A fused part's normalized output in the slot's block for CTA c,
          // lane-major so that a warp's accesses are contiguous: columns
          // 256 c + 16 q + 4 j .. + 3 of head h at float4 (4 q + j) * 128 + h.
          auto fused_block = [&](int64_t sl) {
            return reinterpret_cast<float4*>(p.part_o + (sl * kHeads + 64 * c) * kDv);
          };
          // 16 bf16 output values (8 packed words) of head h at column 256 c + 16 q
          auto store_out16 = [&](int q, const uint32_t (&ow)[8]) {
            __nv_bfloat16* d = p.out + ((int64_t)u * kHeads + h) * kDv + 256 * c + 16 * q;
            if (p.out_v8) {
              st_global_v8(d, ow);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(d);
              dst[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
              dst[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
            }
          };
          if (p.fused && !full_unit) {
            // The token's two parts: part 0 from its first tile (the end of
            // this pair's range), part 1 to its last (the start of the next
            // pair's).  A part whose partner has published merges at once;
            // otherwise it publishes its normalized output and LSEs, then
            // checks the partner again (sequentially consistent fences on
            // both sides: at least one of the two sees the other, and two
            // merges write the same values).  Nothing waits on another CTA.
            const int part = kt + 1 > n_seg_tiles ? 1 : 0;  // the segment's first tile is not the token's first
            const int64_t fi = ((int64_t)u * 2 + c) * 2;
            int* flag_own = p.merge_flag + fi + part;
            const int* flag_oth = p.merge_flag + fi + (1 - part);
            const int64_t slot_oth = part == 1 ? slot - 1 : slot + 1;  // the partner's pair is the previous / next one
            volatile int* bc = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
            int merge = 0;
            if (!dead) {
              if (tid == 0) *bc = ld_acquire_gpu(flag_oth);
              named_bar_sync(1, 32 * kSoftWarps);
              merge = *bc;
              named_bar_sync(1, 32 * kSoftWarps);
              if (!merge) {
                float4* base = fused_block(slot);
#pragma unroll 1
                for (int q = 0; q < 256 / 16; ++q) {
                  uint32_t r[16];
                  tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
                  const float inv = q < 8 ? inv0 : inv1;
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    base[(4 * q + j) * kHeads + h] =
                        make_float4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                                    __uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv);
                }
                p.merge_lse[(fi + part) * kHeads + h] = lse_v;
                __threadfence();
                named_bar_sync(1, 32 * kSoftWarps);
                if (tid == 0) {
                  st_release_gpu(flag_own, 1);
                  __threadfence();
                  *bc = ld_acquire_gpu(flag_oth);
                }
                named_bar_sync(1, 32 * kSoftWarps);
                merge = *bc;
              }
            }
            if (merge) {
              // out = (w0 O_0 + w1 O_1) / (w0 + w1), w_i = exp(lse_i - M), in the same order on either side
              const float lse_o = __ldcg(p.merge_lse + (fi + 1 - part) * kHeads + h);
              const float l0 = part == 0 ? lse_v : lse_o, l1 = part == 0 ? lse_o : lse_v;
              const float M = fmaxf(l0, l1);
              const float w0 = M == -INFINITY ? 0.f : __expf(l0 - M), w1 = M == -INFINITY ? 0.f : __expf(l1 - M);
              const float ws = w0 + w1, iw = ws > 0.f ? __fdividef(1.f, ws) : 0.f;
              const float4* oth = fused_block(slot_oth);
              // two 16-column chunks per step, the partner's eight loads issued first
#pragma unroll 1
              for (int q = 0; q < 256 / 16; q += 2) {
                float4 o[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = __ldcg(oth + (4 * q + j) * kHeads + h);
                uint32_t r[2][16];
                tmem_ld16(tmem + lane_base + kOCol + 16 * q, r[0]);
                tmem_ld16(tmem + lane_base + kOCol + 16 * q + 16, r[1]);
                tmem_ld_wait();
                const float inv = q < 8 ? inv0 : inv1;  // q and q + 1 lie in one group
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  reg_fence16(r[e]);
                  uint32_t ow[8];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const float ov[4] = {o[4 * e + j].x, o[4 * e + j].y, o[4 * e + j].z, o[4 * e + j].w};
                    float v[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                      const float mine = __uint_as_float(r[e][4 * j + k]) * inv;
                      const float x0 = part == 0 ? mine : ov[k], x1 = part == 0 ? ov[k] : mine;
                      v[k] = fmaf(w1, x1, w0 * x0) * iw;
                    }
                    ow[2 * j] = pack_bf16x2(v[0], v[1]);
                    ow[2 * j + 1] = pack_bf16x2(v[2], v[3]);
                  }
                  store_out16(q + e, ow);
                }
              }
              if (c == 0) p.lse[(int64_t)u * kHeads + h] = ws > 0.f ? M + __logf(ws) : -INFINITY;
            }
          } else {
            for (int q = 0; q < 256 / 16; ++q) {
              uint32_t r[16];
              tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
              if (dead) continue;
              const float inv = q < 8 ? inv0 : inv1;
              if (full_unit) {
                uint32_t ow[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  ow[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
                store_out16(q, ow);
              } else {
                // the workspace is 256-byte aligned: two 32-byte stores
                float* dst = p.part_o + (slot * kHeads + h) * kDv + 256 * c + 16 * q;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  uint32_t w[8];
#pragma unroll
                  for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(__uint_as_float(r[8 * j + k]) * inv);
                  st_global_v8(dst + 8 * j, w);
                }
              }
            }
            if (!dead && c == 0) {
              if (full_unit)
                p.lse[(int64_t)u * kHeads + h] = lse_v;
              else
                p.part_lse[slot * kHeads + h] = lse_v;
            }
          }
          tc_fence_before();
          mbar_arrive(&bars[kBarOFree]);
          if (tid == 0) W8_TRACE(tl, kEvEpiEnd);
        }
        if (++kt == p.nt) {
          kt = 0;
          ++u;
        }
      }
    }
  }
#undef SMLA_WAIT
#undef SMLA_WAIT_X
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // no CTA leaves while its peer may still write into its shared memory
  cluster_sync_all();
  if (threadIdx.x == 0) W8_TRACE(0, kEvExit);
}

// Q preparation: per (token, head) row and scale group g (128 values) a
// power of two 2^s puts the group's largest |q| in (224, 448]; q 2^s (exact in
// f16 for bf16 inputs in range) is split into e4m3 hi + lo, and qinv = 2^-s.
// q8 rows: [group][hi, lo][128 codes].  One warp per row (lane l: values
// 8 l .. 8 l + 7 and 256 + 8 l .. 256 + 8 l + 7); it also zeroes the
// attention kernel's merge flags.
__global__ void __launch_bounds__(256) wide8_q_prep_kernel(const __nv_bfloat16* __restrict__ q, uint8_t* __restrict__ q8,
                                                          float* __restrict__ qinv, int64_t rows, int* merge_flag,
                                                          int64_t n_flags) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  {
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i < n_flags) merge_flag[i] = 0;
  }
  if (row >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(q + row * kDqk);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 v = __ldg(src + lane + 32 * i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));  // the 16 lanes of a group
    int sh = 0;
    if (amax > 0.f) {
      int ea;
      const float m = frexpf(amax, &ea);  // amax = m 2^ea, m in [0.5, 1)
      sh = (m <= 0.875f ? 9 : 8) - ea;    // amax 2^sh in (224, 448]
      sh = max(-126, min(126, sh));
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) split2_f16(ldexpf(x[2 * k], sh), ldexpf(x[2 * k + 1], sh), hi[k], lo[k]);
    const int grp = (lane >> 4) + 2 * i;
    uint8_t* d = q8 + row * 1024 + grp * 256 + (lane & 15) * 8;
    *reinterpret_cast<uint2*>(d) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
    *reinterpret_cast<uint2*>(d + 128) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    if ((lane & 15) == 0) qinv[row * 4 + grp] = ldexpf(1.f, -sh);
  }
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }
// Workspace beyond the partial results: q8, qinv, then the merge flags and LSEs.
size_t q8_bytes(int T) { return round256((size_t)T * kHeads * 1024); }
size_t qinv_bytes(int T) { return round256((size_t)T * kHeads * 4 * 4); }
size_t merge_bytes(int T) { return round256((size_t)T * 4 * 4) + (size_t)T * 4 * kHeads * 4; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Tensor maps, all over bytes: the cache [NB * 64, 656] (m_code: 128-byte
// boxes, 128-byte swizzle; m_rope: 64-byte boxes, 64-byte swizzle), q8
// [T * 128, 1024] (128 x 128 boxes, 128-byte swizzle) and the input q
// [T * 128, 1152] (64 x 128 boxes, 64-byte swizzle).
cudaError_t make_maps(const uint8_t* cache, int64_t n_rows, const void* q8, const void* q, int T, CUtensorMap* m_code,
                      CUtensorMap* m_rope, CUtensorMap* q_map, CUtensorMap* q_rope_map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t rstride[1] = {(cuuint64_t)kRowBytes}, q8stride[1] = {1024}, qstride[1] = {(cuuint64_t)kDqk * 2};
  const cuuint32_t es[2] = {1, 1};
  const cuuint64_t r_dim[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)n_rows};
  const cuuint64_t q8_dim[2] = {1024, (cuuint64_t)T * kHeads};
  const cuuint64_t q_dim[2] = {(cuuint64_t)kDqk * 2, (cuuint64_t)T * kHeads};
  struct Spec {
    CUtensorMap* map;
    const void* base;
    const cuuint64_t* dim;
    const cuuint64_t* stride;
    cuuint32_t box0, box1;
    CUtensorMapSwizzle sw;
  } specs[4] = {{m_code, cache, r_dim, rstride, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B},
                {m_rope, cache, r_dim, rstride, 64, 1, CU_TENSOR_MAP_SWIZZLE_64B},
                {q_map, q8, q8_dim, q8stride, 128, kHeads, CU_TENSOR_MAP_SWIZZLE_128B},
                {q_rope_map, q, q_dim, qstride, 64, kHeads, CU_TENSOR_MAP_SWIZZLE_64B}};
  for (const Spec& sp : specs) {
    const cuuint32_t box[2] = {sp.box0, sp.box1};
    const CUresult r = enc(sp.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(sp.base), sp.dim, sp.stride,
                           box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sp.sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Pairs that can be resident at once (one CTA per SM), looked up once per device.
int resident_pairs(int num_sms) {
  static int cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaFuncSetAttribute(sparse_mla_wide8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)sparse_mla_wide8_kernel, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n <= 0) n = num_sms / 2;
  cached[dev] = n;
  return n;
}

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_set_wide8(long long* buf) {
  return (int)cudaMemcpyToSymbol(g_smla_trace_wide8, &buf, sizeof(buf));
}
#endif

// Pairs take contiguous, balanced ranges of the token-major tile sequence; a
// token split between two pairs is merged in the kernel when every range holds
// at least a whole token's tiles, otherwise by the combine kernel.
AttnPlan plan_decode_wide8(int T, int K, int num_splits, int num_sms) {
  AttnPlan pl;
  pl.HG = kHeads;
  pl.n_hg = 1;
  pl.nt = K > 0 ? (K + kRows - 1) / kRows : 1;
  pl.units = T;
  pl.total = pl.units * pl.nt;
  int64_t G = num_splits > 0 ? pl.units * (int64_t)num_splits : (int64_t)resident_pairs(num_sms);
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  pl.fused = pl.need_combine && pl.total / pl.G >= pl.nt;
  if (pl.fused) pl.need_combine = false;
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  pl.ws_bytes = kWsStatusBytes + round256((size_t)n_slots * kHeads * 4) + (size_t)n_slots * kHeads * kDv * 4 +
                q8_bytes(T) + qinv_bytes(T) + merge_bytes(T);
  return pl;
}

cudaError_t launch_decode_wide8(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  Params p{};
  p.cache = a.cache;
  p.indices = a.indices;
  p.block_table = a.block_table;
  p.req_id = a.req_id;
  p.R = a.R;
  p.MB = a.MB;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;
  p.lse = a.lse;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.status = reinterpret_cast<int*>(ws);
  const int64_t n_slots = (int64_t)plan.G + plan.units - 1;
  const size_t lse_bytes = round256((size_t)n_slots * kHeads * 4);
  p.part_lse = reinterpret_cast<float*>(ws + kWsStatusBytes);
  p.part_o = reinterpret_cast<float*>(ws + kWsStatusBytes + lse_bytes);
  uint8_t* q8 = ws + kWsStatusBytes + lse_bytes + (size_t)n_slots * kHeads * kDv * 4;
  float* qinv = reinterpret_cast<float*>(q8 + q8_bytes(a.T));
  uint8_t* mg = q8 + q8_bytes(a.T) + qinv_bytes(a.T);
  p.merge_flag = reinterpret_cast<int*>(mg);
  p.merge_lse = reinterpret_cast<float*>(mg + round256((size_t)a.T * 4 * 4));
  p.fused = plan.fused ? 1 : 0;
  p.qinv = qinv;
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.T = a.T;
  p.K = a.K;
  p.NB = a.NB;
  p.nt = plan.nt;
  p.total = plan.total;
  p.G = plan.G;
  const int64_t rows = (int64_t)a.T * kHeads;
  wide8_q_prep_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(a.q), q8, qinv,
                                                                      rows, p.merge_flag, (int64_t)a.T * 4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap m_code, m_rope, q_map, q_rope_map;
  e = make_maps(a.cache, a.NB * kBlock, q8, a.q, a.T, &m_code, &m_rope, &q_map, &q_rope_map);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sparse_mla_wide8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  sparse_mla_wide8_kernel<<<2 * plan.G, kThreads, kSmemAlloc, stream>>>(p, m_code, m_rope, q_map, q_rope_map);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  e = launch_combine<kHeads>(p.part_o, p.part_lse, p.out, p.lse, kHeads, 1, p.nt, p.total, p.G, plan.units, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
