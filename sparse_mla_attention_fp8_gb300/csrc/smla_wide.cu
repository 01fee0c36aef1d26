// BF16 sparse prefill for 128 heads on sm_103a: one cluster of two CTAs per
// work range, all 128 heads of a token in the M dimension of every MMA.
//
// What is computed (vLLM flashmla_sparse.py, FlashMLASparseImpl.forward on
// the prefill path): query token t attends with each of its 128 heads to its
// own K top-k rows of the bf16 latent buffer kv [N, 576] (MQA 576/512: all
// heads share the rows; V is the first 512 columns of each row).  Per head h:
//   s_j   = softmax_scale * <q[t,h,:], kv[i_j,:]>
//   out   = sum_j softmax(s)_j * kv[i_j, 0:512]     (bf16 [T, 128, 512])
//   lse   = log(sum_j exp(s_j))                       (fp32 [T, 128])
// Indices outside [0, N) are masked; a token with no valid row gets out = 0
// and lse = -inf.
//
// Why two CTAs: the output block O of one token is 128 heads x 512 fp32 =
// all of one SM's tensor memory, and its Q block (128 x 576 bf16, 144 KB)
// does not fit in shared memory next to the row tiles.  So CTA c of the pair
// owns value columns [256c, 256c + 256) and the features it needs: its four
// 64-feature value panels (features 256c .. 256c + 255, 128-byte swizzle) and
// half of the RoPE part (features 512 + 32c .. 512 + 32c + 31, 64-byte
// swizzle), so both CTAs do the same QK^T work.  Per 64-row tile:
//   * QK^T partial: S_c = Q[:, F_c] kv[rows, F_c]^T, M = 128 heads, N = 64
//     rows, K = the CTA's panels (tcgen05.mma kind::f16, fp32 in TMEM);
//   * the two partials are exchanged through distributed shared memory (each
//     exchange thread sends its head's 32 partial logits of a half tile to the
//     peer as 16-bit fixed point with st.async, whose bytes complete the
//     peer's barrier), and each CTA adds the peer's to its own: S = S_0 + S_1
//     up to 2^-16 of the largest partial of the head's half tile;
//   * softmax, one thread per head (the head's TMEM lane): online max and sum
//     in the log2 domain with lazy rescaling of O, P in bf16 written back to
//     TMEM;
//   * P.V: O_c += P V[rows, 256c : 256c + 256], A = P from TMEM, B = the
//     value panels of the same row tile (MN-major), N = 256.
// Warp roles: 0..3 softmax, 4..7 and 8..11 exchange of tile rows 0..31 and
// 32..63 (partial logits -> full, masked, log2-domain logits back in TMEM +
// the maximum), 12 QK^T issuer, 13 index translation + Q, 14..17 row loaders
// (TMA tile::gather4 straight into swizzled K-major operand tiles), 18 P.V
// issuer.
// Warp w of the first three groups handles heads 32 (w % 4) .. + 31 (its
// TMEM lane quarter), one per thread; the two halves' exchanges run side by
// side and overlap the softmax of the previous tile.  19 warps: at most 5 per
// sub-partition, so 96 registers per thread.  Work: pairs take contiguous balanced ranges of the
// token-major tile sequence; a token split over pairs goes through the
// LSE-weighted combine.
#include <cstdint>
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
constexpr int kHeads = 128;                 // heads per pair = M of every MMA
constexpr int kRows = 64;                   // top-k rows per tile
constexpr int kPanel = kRows * 128;         // 8 KB: 64 rows x 64 bf16
constexpr int kQPanel = kHeads * 128;       // 16 KB: 128 heads x 64 bf16
constexpr int kRopePanel = kRows * 64;      // 4 KB: 64 rows x 32 bf16 (this CTA's RoPE half)
constexpr int kQRopePanel = kHeads * 64;    // 8 KB: 128 heads x 32 bf16
constexpr int kKBuf = 4 * kPanel + kRopePanel;     // 36 KB
constexpr int kQBuf = 4 * kQPanel + kQRopePanel;   // 72 KB
// The peer's partial logits of one half tile (32 rows) as 16-bit fixed point:
// 64 bytes per head, then one fp32 step per head.
constexpr int kXData = kHeads * 64;         // 8 KB
constexpr int kXSlot = kXData + kHeads * 4;  // 8.5 KB
constexpr int kRowBytesBf16 = kDqk * 2;     // 1152
constexpr int kLoaders = 4;                 // loader lw gathers rows 16 lw .. 16 lw + 15
constexpr float kMaxSlack = 8.0f;           // log2 growth of a head's max tolerated before rescaling O

// FP8 rows: per 4-row group the staging holds codes 0..127 and 128..255 of
// the CTA's two scale groups (4 x 128 bytes each), the rows' four scales
// (4 x 16 bytes, padded to 128) and the CTA's RoPE halves (4 x 64 bytes);
// every part starts on a 128-byte boundary (TMA destinations).
constexpr int kRawRope = 1152;                      // offset of the RoPE halves in a group
constexpr int kRawGroup = kRawRope + 4 * 64;        // 1408
constexpr int kRawBuf = (kRows / 4) * kRawGroup;    // 22 KB per tile
constexpr int kRawRowBytes = 128 + 128 + 16 + 64;   // gathered into staging per row
constexpr int kSBufs = 3;                         // S buffers in tensor memory

// shared memory (offsets from a 1024-byte aligned base): Q, the bf16 operand
// tiles, FP8 staging (FP8 rows only), exchange slots, index ring, row flags,
// maxima, barriers
template <bool kFp8>
struct Lay {
  static constexpr int kKBufs = kFp8 ? 2 : 3;    // operand tiles in flight
  static constexpr int kRawBufs = kFp8 ? 2 : 0;  // FP8 staging slots
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBuf;
  static constexpr int kOffRaw = kOffK + kKBufs * kKBuf;
  static constexpr int kOffX = kOffRaw + kRawBufs * kRawBuf;
  static constexpr int kOffSlots = kOffX + 2 * kXSlot;            // int32 [4][64]
  static constexpr int kOffValid = kOffSlots + 4 * kRows * 4;      // uint8 [kKBufs][64]
  static constexpr int kOffRed = kOffValid + kKBufs * kRows;       // float [kSBufs][2 halves][128]: maxima (log2)
  static constexpr int kOffExp = kOffRed + kSBufs * 2 * kHeads * 4;  // int [kKBufs][4 quarters] (FP8 rows)
  static constexpr int kOffFac = kOffExp + kKBufs * 4 * 4;          // uint4 [loader][32] conversion factors (FP8 rows)
  static constexpr int kOffBar = kOffFac + (kFp8 ? kLoaders * 32 * 16 : 0);
  enum {
    kBarKFull = 0, kBarKEmpty = kBarKFull + kKBufs, kBarSFull = kBarKEmpty + kKBufs, kBarSReady = kBarSFull + kSBufs,
    kBarSFree = kBarSReady + kSBufs, kBarPFull = kBarSFree + kSBufs, kBarPDone = kBarPFull + 2,
    kBarXFull = kBarPDone + 2, kBarXFree = kBarXFull + 2, kBarIdxFull = kBarXFree + 2,
    kBarIdxEmpty = kBarIdxFull + 4, kBarQFull = kBarIdxEmpty + 4, kBarQEmpty = kBarQFull + 1,
    kBarOFree = kBarQEmpty + 1, kBarDrain = kBarOFree + 1, kBarDrainPv = kBarDrain + 1,
    kBarRawFull = kBarDrainPv + 1,  // [loader][staging slot], FP8 rows only
    kNumBars = kBarRawFull + 2 * kLoaders
  };
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemAlloc = kOffMisc + 16 + 1024;
  static_assert(kOffK % 1024 == 0 && kOffRaw % 128 == 0 && kKBuf % 1024 == 0, "operand alignment");
  static_assert(kOffBar % 8 == 0 && kOffRed % 16 == 0 && kOffX % 16 == 0, "alignment");
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};
static_assert((4 * kPanel) % 512 == 0 && (4 * kQPanel) % 512 == 0, "64-byte-swizzle atoms are 512 bytes");

// tensor memory columns
constexpr int kOCol = 0;    // O_c: 256 fp32 columns
constexpr int kSCol = 256;  // S: 3 buffers x 64 columns
constexpr int kPCol = 448;  // P: 2 buffers x 32 columns (bf16 pairs)
constexpr int kTmemCols = 512;

constexpr int kSoftWarps = 4, kXchgWarp0 = 4, kXchgWarps = 8, kMmaWarp = 12, kIndexWarp = 13, kLoadWarp0 = 14;
constexpr int kPvWarp = kLoadWarp0 + kLoaders;  // issues P.V (kMmaWarp issues QK^T)
constexpr int kNumWarps = kPvWarp + 1;
constexpr int kThreads = 32 * kNumWarps;

// Optional per-tile timeline for performance work: with SMLA_TRACE defined,
// roles record clock64() at their hand-off points into g_smla_trace_wide
// (set by the host through smla_trace_set_wide).  Compiled out otherwise.
#ifdef SMLA_TRACE
__device__ long long* g_smla_trace_wide = nullptr;
constexpr int kTraceTiles = 64, kTraceEvents = 20;
#define WIDE_TRACE(tl, ev)                                                                                   \
  do {                                                                                                       \
    if (trace_buf && (tl) < kTraceTiles)                                                                   \
      trace_buf[((size_t)blockIdx.x * kTraceTiles + (tl)) * kTraceEvents + (ev)] = clock64();             \
  } while (0)
#else
#define WIDE_TRACE(tl, ev) ((void)0)
#endif
// (the CTA's first instruction and its exit in tile 0's slots; a segment's
// epilogue start and end in its last tile's)
enum { kEvSFull = 0, kEvSLoaded, kEvXFree, kEvSent, kEvXFull, kEvPReady, kEvPFull, kEvQk, kEvPv, kEvIssue, kEvQkSeen,
       kEvKEmpty, kEvConverted, kEvRawFull, kEvXTop, kEvXKFull, kEvEnter, kEvEpiStart, kEvEpiEnd, kEvExit };

struct Params {
  const __nv_bfloat16* q;  // [T, 128, 576]
  const int32_t* indices;  // [T, K]: kv rows (bf16) or logical token indices (FP8)
  const int32_t* block_table;  // FP8 rows: [R, MB]
  const int32_t* req_id;       // FP8 rows: [T]
  const float* qinv;           // FP8 rows: [T, 128] 2^-s of each head's Q prescale
  int R, MB;
  __nv_bfloat16* out;      // [T, 128, 512]
  int out_v8;              // out is 32-byte aligned: a thread writes 16 output values in one store
  float* lse;              // [T, 128]
  float* part_o;           // [slots, 128, 512]
  float* part_lse;         // [slots, 128]
  // FP8 rows, every split token cut once (fused): the token's two parts merge
  // in the kernel.  Per (token, CTA of the pair, part: 0 = from the token's
  // first tile, 1 = to its last): a published flag and the part's LSEs.
  int* merge_flag;         // [T, 2, 2], zeroed by the Q preparation kernel
  float* merge_lse;        // [T, 2, 2, 128]
  int fused;
  int* status;
  float scale_log2;        // softmax_scale * log2(e)
  int T, K;
  int64_t N;               // kv rows (bf16) or physical 64-row blocks (FP8)
  int nt;                  // tiles per token
  int64_t total;           // T * nt
  int G;                   // pairs
};

struct TileInfo {
  int u, kt;
  bool seg_start, seg_end;
};

// st.async of raw 32-bit words into a peer CTA's shared memory, completing
// `bar` (cluster addresses) by the bytes written.
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

// 2^e for an integer e in [-127, 127] (-127 gives 0).
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// FP8 rows: exponent E of a 16-row quarter of a tile.  Its codes become f16
// values code * scale * 2^-E, and its RoPE values bf16 values RoPE * 2^-E;
// the logits and P take 2^E back in fp32.  E = floor(log2(largest scale of
// the quarter's four groups)) - 6 puts that scale in [64, 128), so every
// product stays below 448 * 128 < 65504 (the f16 maximum) and the quarter's
// large values are normal f16 numbers.  E is raised where needed so that the
// RoPE values times 2^-E stay below 2^101, and clamped to [-120, 120].
// smax = largest scale, rbits = largest |RoPE| as bf16 bits (0 = none).
__device__ __forceinline__ int quarter_exponent(float smax, uint32_t rbits) {
  int e = smax > 0.f ? (int)((__float_as_uint(smax) >> 23) & 0xFFu) - 127 - 6 : -1000;
  if (rbits != 0u) e = max(e, (int)((rbits >> 7) & 0xFFu) - 127 - 100);
  if (e == -1000) e = 0;  // nothing but zeros
  return min(max(e, -120), 120);
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ TileInfo tile_info(const Params& p, int64_t x, int64_t xbeg, int64_t xend) {
  TileInfo ti;
  ti.u = (int)(x / p.nt);
  ti.kt = (int)(x - (int64_t)ti.u * p.nt);
  ti.seg_start = (x == xbeg) || (ti.kt == 0);
  ti.seg_end = (x == xend - 1) || (ti.kt == p.nt - 1);
  return ti;
}

// Row maps: bf16 rows: m0 = 128-byte value panels (128-byte swizzle), m1
// unused, m2 = 64-byte RoPE halves (64-byte swizzle).  FP8 rows: m0 = 128
// bytes of codes, m1 = the 16 scale bytes, m2 = the 64-byte RoPE halves (all
// unswizzled, into staging).
template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(96)
    sparse_mla_wide_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap m0,
                           const __grid_constant__ CUtensorMap m1, const __grid_constant__ CUtensorMap m2,
                           const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap q_rope_map) {
  using L = Lay<kFp8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  grid_launch_dependents();  // the combine may be launched behind this grid right away
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + L::kOffSlots);
  uint8_t* valid = smem + L::kOffValid;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
#ifdef SMLA_TRACE
  // read once: a store through the global pointer would force a reload at every event
  long long* __restrict__ const trace_buf = g_smla_trace_wide;
  if (tid == 0) WIDE_TRACE(0, kEvEnter);
#endif
  const int lane = tid & 31;
  const int c = (int)cluster_ctarank();  // value half owned by this CTA
  const int pair = blockIdx.x >> 1;
  const int64_t xbeg = tile_begin(pair, p.total, p.G);
  const int64_t xend = tile_begin(pair + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);

  if (tid == 0) {
    for (int i = 0; i < L::kKBufs; ++i) {
      mbar_init(&bars[L::kBarKFull + i], kLoaders);
      mbar_init(&bars[L::kBarKEmpty + i], 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&bars[L::kBarSFull + i], 1);
      mbar_init(&bars[L::kBarSReady + i], 32 * kXchgWarps);
      mbar_init(&bars[L::kBarSFree + i], 32 * kSoftWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[L::kBarPFull + i], 32 * kSoftWarps);
      mbar_init(&bars[L::kBarPDone + i], 1);
    }
    for (int i = 0; i < 2; ++i) {               // exchange slot i carries half i of every tile
      mbar_init(&bars[L::kBarXFull + i], 1);           // own expect_tx + the peer's st.async bytes
      mbar_init(&bars[L::kBarXFree + i], kSoftWarps);  // one arrival per peer exchange warp
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[L::kBarIdxFull + i], 32);
      mbar_init(&bars[L::kBarIdxEmpty + i], kLoaders);
    }
    if (kFp8)
      for (int i = 0; i < 2 * kLoaders; ++i) mbar_init(&bars[L::kBarRawFull + i], 1);  // per loader and slot
    mbar_init(&bars[L::kBarQFull], 1);
    mbar_init(&bars[L::kBarQEmpty], 1);
    mbar_init(&bars[L::kBarOFree], 32 * kSoftWarps);
    mbar_init(&bars[L::kBarDrain], 1);
    mbar_init(&bars[L::kBarDrainPv], 1);
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
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      const int b4 = tl & 3;
      if (tl >= 4 && !SMLA_WAIT(L::kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
      const int32_t req = kFp8 ? __ldg(p.req_id + ti.u) : 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = lane + 32 * i;
        const int k = ti.kt * kRows + r;
        int32_t s = -1;
        if (k < p.K) {
          const int32_t idx = __ldg(p.indices + (int64_t)ti.u * p.K + k);
          if constexpr (kFp8)
            s = translate_slot(idx, req, p.block_table, p.R, p.MB, p.N);
          else
            s = (idx >= 0 && (int64_t)idx < p.N) ? idx : -1;
        }
        slots_ring[b4 * kRows + r] = s;
      }
      mbar_arrive(&bars[L::kBarIdxFull + b4]);
      if (ti.seg_start) {
        // the segment's Q block, once the previous segment's last QK^T is done
        if (seg >= 1 && !SMLA_WAIT(L::kBarQEmpty, (seg - 1) & 1)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[L::kBarQFull], (uint32_t)kQBuf);
          for (int b = 0; b < 4; ++b)
            tma_load_2d(smem_u32(smem + L::kOffQ + b * kQPanel), &q_map, 128 * (4 * c + b), ti.u * kHeads,
                        &bars[L::kBarQFull]);
          tma_load_2d(smem_u32(smem + L::kOffQ + 4 * kQPanel), &q_rope_map, 2 * kDv + 64 * c, ti.u * kHeads,
                      &bars[L::kBarQFull]);
        }
        __syncwarp();
        ++seg;
      }
    }
    // no Q copy may still be landing in shared memory when the CTA exits
    if (seg > 0 && lane == 0) mbar_wait_drain(&bars[L::kBarQFull], (seg - 1) & 1);
    __syncwarp();
  } else if (kFp8 && warp >= kLoadWarp0 && warp < kPvWarp) {
    // ------------------------------------------------------------ FP8 row loaders + converters
    // Loader lw owns tile rows 16 lw .. 16 lw + 15 (staging groups 4 lw ..
    // 4 lw + 3).  Two tiles ahead it gathers their codes (the CTA's two scale
    // groups), scales and RoPE halves into a staging slot, lane 4 g + b
    // issuing copy b of group g; when an operand tile is free it converts the
    // staged codes to f16 values code * scale * 2^-E with one rounding
    // (relative error at most 2^-11 plus a few units of 2^-22; E is the
    // quarter's exponent, which keeps every value inside f16's range whatever
    // the scales), lane l handling codes 8 l .. 8 l + 7 of each row, and copies
    // the RoPE halves (bf16, times 2^-E) into the tile's 64-byte-swizzled
    // panel.  Nothing on the way from a free tile to a full one waits for a
    // copy from global memory.
    const int lw = warp - kLoadWarp0;
    uint8_t* raw_base = smem + L::kOffRaw;
    const int rgrp = lane >> 2, rbox = lane & 3;
    int raw_issued = 0;
    auto issue_raw = [&](int t2) -> bool {
      const int b4 = t2 & 3, sl = t2 & 1;
      if (!SMLA_WAIT(L::kBarIdxFull + b4, (t2 >> 2) & 1)) return false;
      const int32_t s = lane < 16 ? slots_ring[b4 * kRows + 16 * lw + lane] : -1;
      const int r0 = __shfl_sync(kFullMask, s, (4 * rgrp) & 31), r1 = __shfl_sync(kFullMask, s, (4 * rgrp + 1) & 31);
      const int r2 = __shfl_sync(kFullMask, s, (4 * rgrp + 2) & 31), r3 = __shfl_sync(kFullMask, s, (4 * rgrp + 3) & 31);
      uint64_t* bar = &bars[L::kBarRawFull + 2 * lw + sl];
      if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(16 * kRawRowBytes));
      __syncwarp();
      if (lane < 16) {
        const uint32_t dst =
            smem_u32(raw_base + sl * kRawBuf + (4 * lw + rgrp) * kRawGroup + (rbox < 3 ? 512 * rbox : kRawRope));
        if (rbox < 2)
          tma_gather4_2d(dst, &m0, 256 * c + 128 * rbox, r0, r1, r2, r3, bar);
        else if (rbox == 2)
          tma_gather4_2d(dst, &m1, kScaleOff, r0, r1, r2, r3, bar);
        else
          tma_gather4_2d(dst, &m2, kRopeOff + 64 * c, r0, r1, r2, r3, bar);
      }
      ++raw_issued;
      return true;
    };
    bool ok = true;
    if (n_local > 0) ok = issue_raw(0);
    if (ok && n_local > 1) ok = issue_raw(1);
    int converted = 0;
    for (int tl = 0; ok && tl < n_local; ++tl) {
      const int b4 = tl & 3, kb = tl % L::kKBufs, use = tl / L::kKBufs, sl = tl & 1;
      if (!SMLA_WAIT(L::kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = lane < 16 ? slots_ring[b4 * kRows + 16 * lw + lane] : -1;
      const uint32_t vmask = __ballot_sync(kFullMask, slot >= 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[L::kBarIdxEmpty + b4]);
      if (!SMLA_WAIT(L::kBarRawFull + 2 * lw + sl, (tl >> 1) & 1)) break;
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvRawFull);
      const uint8_t* raw = raw_base + sl * kRawBuf;
      // the quarter's exponent E from its rows' four scales and RoPE values
      // (staged; the same bytes in both CTAs of the pair, so both take the same E)
      uint4 rv[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = lane + 32 * i, r = 16 * lw + (k >> 2), j = k & 3;
        rv[i] = *reinterpret_cast<const uint4*>(raw + (r >> 2) * kRawGroup + kRawRope + (r & 3) * 64 + 16 * j);
      }
      int q_exp;
      {
        float smax = 0.f;
        if (lane < 16) {
          const int r = 16 * lw + lane;
          const float4 s4 = *reinterpret_cast<const float4*>(raw + (r >> 2) * kRawGroup + 1024 + (r & 3) * 16);
          smax = fmaxf(fmaxf(s4.x, s4.y), fmaxf(s4.z, s4.w));
        }
        // |bf16| orders as its bits with the sign cleared
        uint32_t rb = 0u;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t w[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) rb = max(rb, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          smax = fmaxf(smax, __shfl_xor_sync(kFullMask, smax, o));
          rb = max(rb, __shfl_xor_sync(kFullMask, rb, o));
        }
        q_exp = quarter_exponent(smax, rb);
      }
      const float q_fac = exp2i(-q_exp);                                    // 2^-E (exact)
      const uint32_t q_fac_bf2 = (uint32_t)(127 - q_exp) * 0x00800080u;     // 2^-E as a bf16 pair
      // conversion factors of row 16 lw + (lane & 15), scale group 2 c + (lane >> 4):
      // s = scale * 2^-E (exact) is brought to t = s * 2^m in [1, 2) when
      // 0 < s < 1 (m <= 24) and split as t_hi = f16(t), t_lo = f16(t - t_hi)
      uint4* fac = reinterpret_cast<uint4*>(smem + L::kOffFac) + 32 * lw;
      bool all_m0;
      {
        const int r = 16 * lw + (lane & 15);
        const float sq =
            *reinterpret_cast<const float*>(raw + (r >> 2) * kRawGroup + 1024 + (r & 3) * 16 + 4 * (2 * c + (lane >> 4))) *
            q_fac;
        const int m = (sq < 1.f && sq > 0.f) ? min(127 - (int)((__float_as_uint(sq) >> 23) & 0xFFu), 24) : 0;
        const float t = sq * exp2i(m);
        const __half t_hi = __float2half_rn(t);
        const __half t_lo = __float2half_rn(t - __half2float(t_hi));
        // 2^-m as f16 (subnormal below 2^-14)
        const uint32_t sh = m <= 14 ? (uint32_t)(15 - m) << 10 : 1u << (24 - m);
        __syncwarp();  // the previous tile's factors have been read
        fac[lane] = make_uint4((uint32_t)__half_as_ushort(t_hi) * 0x00010001u,
                               (uint32_t)__half_as_ushort(t_lo) * 0x00010001u, sh * 0x00010001u, 0u);
        all_m0 = __all_sync(kFullMask, m == 0);
        __syncwarp();
      }
      if (use >= 1 && !SMLA_WAIT(L::kBarKEmpty + kb, (use + 1) & 1)) break;
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvKEmpty);
      if (lane < 16) valid[kb * kRows + 16 * lw + lane] = (uint8_t)((vmask >> lane) & 1u);
      if (lane == 0) reinterpret_cast<int*>(smem + L::kOffExp)[kb * 4 + lw] = q_exp;
      const uint32_t tile = smem_u32(smem + L::kOffK + kb * kKBuf);
      const int half = lane >> 4, pnl = lane >> 3, ch = lane & 7;
      // RoPE halves times 2^-E (exact): 16 rows x 4 chunks of 16 bytes, two per
      // lane, into the 64-byte swizzle (chunk j of row r at j ^ ((r >> 1) & 3)
      // in its 64 bytes)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int k = lane + 32 * i, r = 16 * lw + (k >> 2), j = k & 3;
        st_shared_v4(tile + 4 * kPanel + (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + ((j ^ ((r >> 1) & 3)) << 4)),
                     mul_bf16x2(rv[i].x, q_fac_bf2), mul_bf16x2(rv[i].y, q_fac_bf2), mul_bf16x2(rv[i].z, q_fac_bf2),
                     mul_bf16x2(rv[i].w, q_fac_bf2));
      }
      // 4 rows at a time: all their loads first, so that one load latency
      // covers 4 rows (the stores are ordered after them).  code * scale * 2^-E
      // in f16x2 with one rounding where the result is a normal f16:
      // fma(code, t_hi, code * t_lo) * 2^-m (the codes widen to f16 exactly;
      // the last product is exact unless its result is subnormal, and is
      // skipped when m = 0 for every row and group of the quarter).
#pragma unroll 1
      for (int rb = 0; rb < 16; rb += 4) {
        uint2 cw[4];
        uint4 f4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 16 * lw + rb + i;
          const uint8_t* grp = raw + (r >> 2) * kRawGroup;
          cw[i] = *reinterpret_cast<const uint2*>(grp + 512 * half + (r & 3) * 128 + 8 * (lane & 15));
          f4[i] = fac[rb + i + 16 * half];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 16 * lw + rb + i;
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint16_t pr = (uint16_t)(((k < 2 ? cw[i].x : cw[i].y) >> (16 * (k & 1))) & 0xFFFFu);
            uint32_t h2, t2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pr));  // exact
            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t2) : "r"(h2), "r"(f4[i].y));
            asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[k]) : "r"(h2), "r"(f4[i].x), "r"(t2));
          }
          if (!all_m0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[k]) : "r"(o[k]), "r"(f4[i].z));
          }
          st_shared_v4(tile + pnl * kPanel + (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4)), o[0],
                       o[1], o[2], o[3]);
        }
      }
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvConverted);
      // the tile's full barrier: this warp's arrival for its converted rows
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[L::kBarKFull + kb]);
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvIssue);
      converted = tl + 1;
      if (tl + 2 < n_local) ok = issue_raw(tl + 2);
    }
    // no copy may still be landing in shared memory when the CTA exits
    for (int t2 = converted; t2 < raw_issued; ++t2)
      if (lane == 0) mbar_wait_drain(&bars[L::kBarRawFull + 2 * lw + (t2 & 1)], (t2 >> 1) & 1);
    __syncwarp();
  } else if (warp >= kLoadWarp0 && warp < kPvWarp) {
    // ------------------------------------------------------------ row loaders
    // Loader lw gathers rows 16 lw .. 16 lw + 15 of every tile: 4 groups of 4
    // rows x 5 boxes (4 value panels, the RoPE half), lane 5 g + b issuing box
    // b of group g.  Its one arrival on the tile's full barrier carries the
    // bytes of its 16 rows and follows its writes of the rows' valid flags.
    const int lw = warp - kLoadWarp0;
    const int grp = lane / 5, box = lane - grp * 5;
    const int r_g = 16 * lw + 4 * grp;  // tile row of the lane's group
    int last_b = -1, last_use = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      const int b4 = tl & 3, kb = tl % L::kKBufs, use = tl / L::kKBufs;
      if (!SMLA_WAIT(L::kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = lane < 16 ? slots_ring[b4 * kRows + 16 * lw + lane] : -1;
      const uint32_t vmask = __ballot_sync(kFullMask, slot >= 0);
      const int g0 = __shfl_sync(kFullMask, slot, (4 * grp) & 31), g1 = __shfl_sync(kFullMask, slot, (4 * grp + 1) & 31);
      const int g2 = __shfl_sync(kFullMask, slot, (4 * grp + 2) & 31), g3 = __shfl_sync(kFullMask, slot, (4 * grp + 3) & 31);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[L::kBarIdxEmpty + b4]);
      if (use >= 1 && !SMLA_WAIT(L::kBarKEmpty + kb, (use + 1) & 1)) break;
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvKEmpty);
      if (lane < 16) valid[kb * kRows + 16 * lw + lane] = (uint8_t)((vmask >> lane) & 1u);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&bars[L::kBarKFull + kb], (uint32_t)(16 * (kKBuf / kRows)));
      __syncwarp();
      if (lane < 20) {
        const uint32_t tile = smem_u32(smem + L::kOffK + kb * kKBuf);
        if (box < 4)
          tma_gather4_2d(tile + box * kPanel + (uint32_t)((r_g >> 3) * 1024 + (r_g & 7) * 128), &m0,
                         128 * (4 * c + box), g0, g1, g2, g3, &bars[L::kBarKFull + kb]);
        else
          tma_gather4_2d(tile + 4 * kPanel + (uint32_t)((r_g >> 3) * 512 + (r_g & 7) * 64), &m2,
                         2 * kDv + 64 * c, g0, g1, g2, g3, &bars[L::kBarKFull + kb]);
      }
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvIssue);
      last_b = kb;
      last_use = use;
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (last_b >= 0) mbar_wait_drain(&bars[L::kBarKFull + last_b], last_use & 1);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ QK^T issuer
    // One thread: QK^T of each tile once its rows, the segment's Q and a free
    // S buffer are there (P.V has its own issuer warp, so it never waits
    // behind a QK^T).
    if (lane == 0 && n_local > 0) {
      // FP8 rows: value panels and Q's value part in f16; RoPE parts in bf16
      constexpr uint32_t id_qk = kFp8 ? make_idesc_f16(128, kRows, 0, 0) : make_idesc_bf16(128, kRows, 0, 0);
      constexpr uint32_t id_qkr = make_idesc_bf16(128, kRows, 0, 0);
      // shared-memory descriptors: constant high words, low words = base + offset / 16
      constexpr uint32_t kHi128 = sdesc_hi(1024, kLayoutSw128), kHi64 = sdesc_hi(512, kLayoutSw64);
      const uint32_t dq = sdesc_lo(smem_u32(smem + L::kOffQ), 16), dk0 = sdesc_lo(smem_u32(smem + L::kOffK), 16);
      int seg = 0, kt = (int)(xbeg % p.nt), issued = 0;
      for (int tl = 0; tl < n_local; ++tl) {
        const int kb = tl % L::kKBufs, sb = tl % kSBufs;
        const bool seg_start = tl == 0 || kt == 0;
        const bool seg_end = tl == n_local - 1 || kt == p.nt - 1;
        if (tl >= kSBufs && !SMLA_WAIT(L::kBarSFree + sb, ((tl / kSBufs) + 1) & 1)) break;
        if (seg_start && !SMLA_WAIT(L::kBarQFull, seg & 1)) break;
        if (!SMLA_WAIT(L::kBarKFull + kb, (tl / L::kKBufs) & 1)) break;
        WIDE_TRACE(tl, kEvQkSeen);
        tc_fence_after();
        const uint32_t dk = dk0 + ((kb * kKBuf) >> 4);
        const uint32_t sacc = tmem + kSCol + 64 * sb;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
          for (int s = 0; s < 4; ++s)
            mma_ss(sacc, sdesc_join<kHi128>(dq + ((b * kQPanel + 32 * s) >> 4)),
                   sdesc_join<kHi128>(dk + ((b * kPanel + 32 * s) >> 4)), id_qk, (b | s) != 0 ? 1u : 0u);
        }
#pragma unroll
        for (int s = 0; s < 2; ++s)  // RoPE half: 8-row atoms of 64 bytes
          mma_ss(sacc, sdesc_join<kHi64>(dq + ((4 * kQPanel + 32 * s) >> 4)),
                 sdesc_join<kHi64>(dk + ((4 * kPanel + 32 * s) >> 4)), id_qkr, 1u);
        mma_commit(&bars[L::kBarSFull + sb]);
        if (seg_end) {
          mma_commit(&bars[L::kBarQEmpty]);
          ++seg;
        }
        WIDE_TRACE(tl, kEvQk);
        ++issued;
        kt = kt + 1 == p.nt ? 0 : kt + 1;
      }
      // every issued tensor-core operation completes before tensor memory is released
      if (issued > 0) {
        mma_commit(&bars[L::kBarDrain]);
        mbar_wait_drain(&bars[L::kBarDrain], 0);
      }
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P.V issuer
    // One thread: O_c += P V of each tile once its P is written (and, first in
    // a segment, the previous segment's epilogue has read O).  Its completion
    // frees the row tile and the P buffer.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_pv = kFp8 ? make_idesc_f16(128, 256, 0, 1) : make_idesc_bf16(128, 256, 0, 1);
      constexpr uint32_t kHi128 = sdesc_hi(1024, kLayoutSw128);
      const uint32_t dv0 = sdesc_lo(smem_u32(smem + L::kOffK), kPanel);
      int seg_o = 0, kt = (int)(xbeg % p.nt), issued = 0;
      for (int tl = 0; tl < n_local; ++tl) {
        const int kb = tl % L::kKBufs, pb = tl & 1;
        const bool seg_start = tl == 0 || kt == 0;
        if (seg_start && seg_o > 0 && !SMLA_WAIT(L::kBarOFree, (seg_o - 1) & 1)) break;
        if (!SMLA_WAIT(L::kBarPFull + pb, (tl >> 1) & 1)) break;
        if (seg_start) ++seg_o;
        tc_fence_after();
        const uint32_t dv = dv0 + ((kb * kKBuf) >> 4);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          // B = V rows 16 s .. 16 s + 15 x 256 value columns, MN-major:
          // 64-column panels kPanel apart, 8-row groups 1024 bytes apart
          mma_ts(tmem + kOCol, tmem + kPCol + 32 * pb + 8 * s, sdesc_join<kHi128>(dv + ((2048 * s) >> 4)), id_pv,
                 (seg_start && s == 0) ? 0u : 1u);
        mma_commit(&bars[L::kBarKEmpty + kb]);
        mma_commit(&bars[L::kBarPDone + pb]);
        WIDE_TRACE(tl, kEvPv);
        ++issued;
        kt = kt + 1 == p.nt ? 0 : kt + 1;
      }
      if (issued > 0) {
        mma_commit(&bars[L::kBarDrainPv]);
        mbar_wait_drain(&bars[L::kBarDrainPv], 0);
      }
    }
    __syncwarp();
  } else {
    const int qd = warp & 3;
    const int h = 32 * qd + lane;  // head = TMEM lane of S, P and O
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    float* red = reinterpret_cast<float*>(smem + L::kOffRed);
    if (warp >= kXchgWarp0) {
      // ---------------------------------------------------------- exchange (warps 4..11)
      // Warp group e handles half e of every tile (rows 32 e .. 32 e + 31,
      // exchange slot e): the partial logits go to the peer (st.async into
      // its slot, the bytes completing its barrier), the peer's partial is
      // added, rows are masked and scaled to the log2 domain, and the result
      // is written back over the S buffer.  A half is sent once the peer has
      // read the same half of the previous tile.
      //
      // The SM-to-SM network moves about 12 bytes per cycle, so the partials
      // travel as 16-bit fixed point: each head's 32 values as integers
      // q = round(x * 32767 / a) with a the largest magnitude among them, plus
      // the step a / 32767.  The error of a received value is at most a / 65534
      // (plus fp32 rounding), i.e. 2^-16 of the half row's largest partial.
      // The codes are q + 32768 (offset binary); both conversions stay on the
      // full-rate pipes: fma(x, 32767 / a, 1.5 * 2^23 + 32768) rounds to the
      // nearest integer and leaves the code in its low 16 bits, and a code u
      // placed under the exponent of 2^23 reads as 2^23 + u.
      // The 16-byte chunk i of head h sits at position (i + h / 2) % 4 of the
      // head's 64 bytes, so that eight consecutive heads cover all banks.
      const uint32_t peer = (uint32_t)(c ^ 1);
      const uint32_t x_chunk = (uint32_t)(h * 64);
      const uint32_t x_remote = mapa_shared(smem_u32(smem + L::kOffX), peer);
      const uint32_t xfull_remote = mapa_shared(smem_u32(&bars[L::kBarXFull]), peer);
      const uint32_t xfree_remote = mapa_shared(smem_u32(&bars[L::kBarXFree]), peer);
      const int e = (warp - kXchgWarp0) >> 2;
      const bool lead = lane == 0 && qd == 0;  // registers the slot's expected bytes
      bool dead = false;
      int u = (int)(xbeg / p.nt), kt = (int)(xbeg - (int64_t)u * p.nt);
      for (int tl = 0; tl < n_local; ++tl) {
        // FP8 rows: Q was scaled by 2^s per head; the logits take 2^-s back
        const float sl2 = kFp8 ? p.scale_log2 * __ldg(p.qinv + (int64_t)u * kHeads + h) : p.scale_log2;
        if (++kt == p.nt) {
          kt = 0;
          ++u;
        }
        const int sb = tl % kSBufs, kb = tl % L::kKBufs;
        if (tid == 32 * kXchgWarp0) WIDE_TRACE(tl, kEvXTop);
        // row validity (written by the loaders before the tile's full barrier)
        if (!dead) dead = !SMLA_WAIT(L::kBarKFull + kb, (tl / L::kKBufs) & 1);
        if (tid == 32 * kXchgWarp0) WIDE_TRACE(tl, kEvXKFull);
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
        // FP8 rows: the half's two quarters hold logits times 2^-E0 and
        // 2^-E1; both are brought to 2^-max(E0, E1) (the same in both CTAs),
        // and the scale to the log2 domain takes 2^max(E0, E1) back
        float qf0 = 1.f, qf1 = 1.f, sl2t = sl2;
        if constexpr (kFp8) {
          const int* qe = reinterpret_cast<const int*>(smem + L::kOffExp) + kb * 4 + 2 * e;
          const int e0 = qe[0], e1 = qe[1], eh = max(e0, e1);
          qf0 = exp2i(max(e0 - eh, -127));
          qf1 = exp2i(max(e1 - eh, -127));
          sl2t = sl2 * exp2i(eh);
        }
        if (!dead) dead = !SMLA_WAIT(L::kBarSFull + sb, (tl / kSBufs) & 1);
        if (tid == 32 * kXchgWarp0) WIDE_TRACE(tl, kEvSFull);
        tc_fence_after();
        float mt = -INFINITY;
        {
          const uint32_t scol = tmem + lane_base + kSCol + 64 * sb + 32 * e;
          if (lead) mbar_arrive_expect_tx(&bars[L::kBarXFull + e], (uint32_t)kXSlot);
          float s[32];
          {
            uint32_t r0[16], r1[16];
            tmem_ld16(scol, r0);
            tmem_ld16(scol + 16, r1);
            tmem_ld_wait();
            reg_fence16(r0);
            reg_fence16(r1);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              s[j] = __uint_as_float(r0[j]);
              s[16 + j] = __uint_as_float(r1[j]);
            }
            if (kFp8 && (qf0 != 1.f || qf1 != 1.f)) {  // uniform: the tile's exponents
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                s[j] *= qf0;
                s[16 + j] *= qf1;
              }
            }
          }
          // 16-bit fixed point relative to the largest magnitude
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(s[j]));
          // (a magnitude below 2^-100 sends zeros)
          const float inv = amax > 0x1p-100f ? __fdividef(32767.f, amax) : 0.f;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = __byte_perm(__float_as_uint(fmaf(s[2 * j], inv, 12615680.f)),
                                __float_as_uint(fmaf(s[2 * j + 1], inv, 12615680.f)), 0x5410);
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvSLoaded);
          if (tl >= 1 && !dead) dead = !SMLA_WAIT_X(L::kBarXFree + e, (tl - 1) & 1);
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvXFree);
          if (!dead) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              st_async_v4_b32(x_remote + e * kXSlot + x_chunk + 16 * ((i + (h >> 1)) & 3), pk[4 * i],
                              pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3], xfull_remote + 8 * e);
            st_async_b32(x_remote + e * kXSlot + kXData + 4 * h, __float_as_uint(amax * (1.f / 32767.f)),
                         xfull_remote + 8 * e);
          }
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvSent);
          if (!dead) dead = !SMLA_WAIT_X(L::kBarXFull + e, tl & 1);
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvXFull);
          if (!dead) {
            const uint8_t* src = smem + L::kOffX + e * kXSlot;
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
          uint32_t r[2][16];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = (vb >> j) & 1u ? s[j] * sl2t : -INFINITY;
            mt = fmaxf(mt, x);
            r[j >> 4][j & 15] = __float_as_uint(x);
          }
          tc_fence_after();
          tmem_st16(scol, r[0]);
          tmem_st16(scol + 16, r[1]);
        }
        tmem_st_wait();
        red[(sb * 2 + e) * kHeads + h] = mt;
        tc_fence_before();
        mbar_arrive(&bars[L::kBarSReady + sb]);
        if (tid == 32 * kXchgWarp0) WIDE_TRACE(tl, kEvPReady);
      }
    } else {
      // ---------------------------------------------------------- softmax + epilogue (warps 0..3)
      float m_used = -INFINITY, l_sum = 0.f;
      int n_seg_tiles = 0;
      int e_run = 0;  // FP8 rows: O holds sum_j p_j V_j * 2^-e_run
      bool dead = false;
      int u = (int)(xbeg / p.nt), kt = (int)(xbeg - (int64_t)u * p.nt);
      for (int tl = 0; tl < n_local; ++tl) {
        const bool seg_start = tl == 0 || kt == 0;
        const bool seg_end = tl == n_local - 1 || kt == p.nt - 1;
        const int sb = tl % kSBufs, pb = tl & 1;
        if (seg_start) {
          m_used = -INFINITY;
          l_sum = 0.f;
          n_seg_tiles = 0;
        }
        // full, masked log2-domain logits of the tile and their maximum
        if (!dead) dead = !SMLA_WAIT(L::kBarSReady + sb, (tl / kSBufs) & 1);
        tc_fence_after();
        const float mt = fmaxf(red[(sb * 2) * kHeads + h], red[(sb * 2 + 1) * kHeads + h]);
        // A head whose max grew by more than kMaxSlack takes the new max; when
        // O already holds earlier tiles of the segment its row is scaled by
        // a = 2^(m_used - m_new).
        const bool need = mt > m_used + kMaxSlack || (m_used == -INFINITY && mt > -INFINITY);
        const bool scale_m = need && n_seg_tiles > 0 && m_used > -INFINITY;
        const float dm = scale_m ? m_used - mt : 0.f;
        if (need) m_used = mt;
        // FP8 rows: quarter q of the tile carries V * 2^-E_q.  O stays in units
        // of 2^e_run, raised (O rescaled) when a tile's largest E_q exceeds it
        // by more than 7, so that P' = p * 2^(E_q - e_run) <= 2^8 * 2^7 stays
        // inside f16.  P' is formed as 2^(logit - mu_q) with
        // mu_q = m_used - (E_q - e_run) (the shift floored at -64, where P'
        // weighs less than 2^-40 of the largest value O can hold), and the row
        // sum takes the shift back.
        bool e_up = false;
        float de = 0.f, mu_q[4] = {m_used, m_used, m_used, m_used}, w_q[4] = {1.f, 1.f, 1.f, 1.f};
        if constexpr (kFp8) {
          const int* qe = reinterpret_cast<const int*>(smem + L::kOffExp) + (tl % L::kKBufs) * 4;
          const int eq[4] = {qe[0], qe[1], qe[2], qe[3]};
          const int emax = max(max(eq[0], eq[1]), max(eq[2], eq[3]));
          if (seg_start) {
            e_run = emax;
          } else if (emax > e_run + 7) {
            de = (float)(e_run - emax);
            e_run = emax;
            e_up = true;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int d = max(eq[q] - e_run, -64);
            mu_q[q] = m_used - (float)d;
            w_q[q] = exp2i(-d);
          }
        }
        const bool scale_o = scale_m || e_up;
        const float a_l = scale_m ? ex2_approx(dm) : 1.f;        // row sums
        const float a = scale_o ? ex2_approx(dm + de) : 1.f;     // O
        // TMEM access is warp-wide: a warp with any head to rescale runs the
        // pass (factor 1 for its other heads), once P.V(tl - 1) has landed in O
        if (__any_sync(kFullMask, scale_o)) {
          if (!dead) dead = !SMLA_WAIT(L::kBarPDone + ((tl - 1) & 1), ((tl - 1) >> 1) & 1);
          tc_fence_after();
#pragma unroll 1
          for (int q = 0; q < 256 / 16; ++q) {
            uint32_t r[16];
            tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a);
            tmem_st16(tmem + lane_base + kOCol + 16 * q, r);
          }
        }
        // P (bf16 pairs) into TMEM, 32 rows at a time, once P.V(tl - 2) has
        // read the buffer
        if (tl >= 2 && !dead) dead = !SMLA_WAIT(L::kBarPDone + pb, ((tl >> 1) + 1) & 1);
        tc_fence_after();
        const bool none = m_used == -INFINITY;
        float lt = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t r0[16], r1[16];
          tmem_ld16(tmem + lane_base + kSCol + 64 * sb + 32 * e, r0);
          tmem_ld16(tmem + lane_base + kSCol + 64 * sb + 32 * e + 16, r1);
          tmem_ld_wait();
          reg_fence16(r0);
          reg_fence16(r1);
          uint32_t pk[16];
          float l0 = 0.f, l1 = 0.f;
          const float mu0 = mu_q[2 * e], mu1 = mu_q[2 * e + 1];  // r0: quarter 2e, r1: quarter 2e + 1
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float p0 = none ? 0.f : ex2_approx(__uint_as_float(r0[2 * j]) - mu0);
            const float p1 = none ? 0.f : ex2_approx(__uint_as_float(r0[2 * j + 1]) - mu0);
            const float p2 = none ? 0.f : ex2_approx(__uint_as_float(r1[2 * j]) - mu1);
            const float p3 = none ? 0.f : ex2_approx(__uint_as_float(r1[2 * j + 1]) - mu1);
            l0 += p0 + p1;
            l1 += p2 + p3;
            pk[j] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            pk[8 + j] = kFp8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3);
          }
          lt += l0 * w_q[2 * e] + l1 * w_q[2 * e + 1];
          tmem_st16(tmem + lane_base + kPCol + 32 * pb + 16 * e, pk);
        }
        tc_fence_before();
        mbar_arrive(&bars[L::kBarSFree + sb]);
        l_sum = l_sum * a_l + lt;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[L::kBarPFull + pb]);
        if (tid == 0) WIDE_TRACE(tl, kEvPFull);
        ++n_seg_tiles;
        // epilogue at the end of a segment
        if (seg_end) {
          if (!dead) dead = !SMLA_WAIT(L::kBarPDone + pb, (tl >> 1) & 1);
          tc_fence_after();
          if (tid == 0) WIDE_TRACE(tl, kEvEpiStart);
          const bool full_unit = n_seg_tiles == p.nt;  // the whole token ran in this pair
          // approximate reciprocal and logarithms (a few ulp): the correctly rounded
          // library forms are long, cold code in an epilogue
          const float inv = l_sum > 0.f ? (kFp8 ? exp2i(e_run) : 1.f) * __fdividef(1.f, l_sum) : 0.f;
          const float lse_v = l_sum > 0.f ? (m_used + __log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
          const int64_t slot = (int64_t)pair + u;
          // A fused part's normalized output in the slot's block for CTA c,
          // lane-major so that a warp's accesses are contiguous: columns
          // 256 c + 16 q + 4 j .. + 3 of head h at float4 (4 q + j) * 128 + h.
          auto fused_block = [&](int64_t sl) {
            return reinterpret_cast<float4*>(p.part_o + (sl * kHeads + 64 * c) * kDv);
          };
          auto write_part = [&](float4* base) {
#pragma unroll 1
            for (int q = 0; q < 256 / 16; ++q) {
              uint32_t r[16];
              tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                base[(4 * q + j) * kHeads + h] =
                    make_float4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                                __uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv);
            }
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
          if (kFp8 && p.fused && !full_unit) {
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
            volatile int* bc = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 8);
            int merge = 0;
            if (!dead) {
              if (tid == 0) *bc = ld_acquire_gpu(flag_oth);
              named_bar_sync(1, 32 * kSoftWarps);
              merge = *bc;
              named_bar_sync(1, 32 * kSoftWarps);
              if (!merge) {
                write_part(fused_block(slot));
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
          mbar_arrive(&bars[L::kBarOFree]);
          if (tid == 0) WIDE_TRACE(tl, kEvEpiEnd);
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
#ifdef SMLA_TRACE
  if (tid == 0) WIDE_TRACE(0, kEvExit);
#endif
}

// Q of the FP8 path: each (token, head) row of 576 bf16 values is scaled by
// 2^s, s chosen so that its largest magnitude lands in [2^14, 2^15), and
// stored as f16 (value part, exact for the bf16 values in range) and bf16
// (RoPE part, exact power-of-two scaling); qinv = 2^-s.  One warp per row.
__global__ void __launch_bounds__(256) wide_q_prep_kernel(const __nv_bfloat16* __restrict__ q, uint16_t* __restrict__ q16,
                                                         float* __restrict__ qinv, int64_t rows, int* merge_flag,
                                                         int64_t n_flags) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  {  // the attention kernel's merge flags start each call at zero
    const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (i < n_flags) merge_flag[i] = 0;
  }
  if (row >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(q + row * kDqk);  // 72 chunks of 8 values
  uint4 v[3];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int ch = lane + 32 * i;
    v[i] = ch < 72 ? __ldg(src + ch) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
  int sh = 0;
  if (amax > 0.f) {
    int ex;
    frexpf(32768.f / amax, &ex);  // 32768 / amax = m * 2^ex, m in [0.5, 1)
    sh = ex - 1;
  }
  const float pre = ldexpf(1.f, sh);
  uint4* dst = reinterpret_cast<uint4*>(q16 + row * kDqk);
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int ch = lane + 32 * i;
    if (ch >= 72) continue;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16) * pre, hi = __uint_as_float(w[k] & 0xFFFF0000u) * pre;
      o[k] = ch < 64 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
    }
    dst[ch] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0) qinv[row] = ldexpf(1.f, -sh);
}

// Workspace of the FP8 path beyond the partial results: the prepared Q and
// the heads' inverse prescales.
size_t q_prep_bytes(int T) {
  return (((size_t)T * kHeads * kDqk * 2 + 255) / 256) * 256 + (((size_t)T * kHeads * 4 + 255) / 256) * 256;
}
// the fused merge's flags and LSEs (after the prepared Q)
size_t merge_bytes(int T) { return (((size_t)T * 4 * 4 + 255) / 256) * 256 + (size_t)T * 4 * kHeads * 4; }

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

// Tensor maps, all over bytes.  bf16 rows (kv [N, 576]): m0 gathers one
// 128-byte value panel of single rows (128-byte swizzle), m2 one 64-byte RoPE
// half (64-byte swizzle).  FP8 rows (the [NB * 64, 656] cache): m0 gathers
// 128 bytes of codes, m1 the 16 scale bytes (unswizzled, into staging), m2
// the 64-byte RoPE half (64-byte swizzle).  q [T * 128, 576] bf16: the same
// slices of 128 consecutive head rows.
template <bool kFp8>
cudaError_t make_maps(const void* rows, int64_t n_rows, const void* q, int T, CUtensorMap* m0, CUtensorMap* m1,
                      CUtensorMap* m2, CUtensorMap* q_map, CUtensorMap* q_rope_map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t row_bytes = kFp8 ? (cuuint64_t)kRowBytes : (cuuint64_t)kRowBytesBf16;
  const cuuint64_t rstride[1] = {row_bytes}, qstride[1] = {(cuuint64_t)kRowBytesBf16};
  const cuuint32_t es[2] = {1, 1};
  const cuuint64_t r_dim[2] = {row_bytes, (cuuint64_t)n_rows};
  const cuuint64_t q_dim[2] = {(cuuint64_t)kRowBytesBf16, (cuuint64_t)T * kHeads};
  struct Spec {
    CUtensorMap* map;
    const void* base;
    const cuuint64_t* dim;
    const cuuint64_t* stride;
    cuuint32_t box0, box1;
    CUtensorMapSwizzle sw;
  } specs[5] = {{m0, rows, r_dim, rstride, 128, 1, kFp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B},
                {m1, rows, r_dim, rstride, kFp8 ? 16u : 128u, 1, kFp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B},
                {m2, rows, r_dim, rstride, 64, 1, kFp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B},
                {q_map, q, q_dim, qstride, 128, kHeads, CU_TENSOR_MAP_SWIZZLE_128B},
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
template <bool kFp8>
int resident_pairs(int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaFuncSetAttribute(sparse_mla_wide_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay<kFp8>::kSmemAlloc) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Lay<kFp8>::kSmemAlloc;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)sparse_mla_wide_kernel<kFp8>, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n <= 0) n = num_sms / 2;
  cached[dev] = n;
  return n;
}

AttnPlan plan_wide(bool fp8, int T, int K, int num_splits, int num_sms) {
  AttnPlan pl;
  pl.HG = kHeads;
  pl.n_hg = 1;
  pl.nt = K > 0 ? (K + kRows - 1) / kRows : 1;
  pl.units = T;
  pl.total = pl.units * pl.nt;
  const int pairs = fp8 ? resident_pairs<true>(num_sms) : resident_pairs<false>(num_sms);
  int64_t G = num_splits > 0 ? pl.units * (int64_t)num_splits : (int64_t)pairs;
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  // FP8 rows: when every pair's range holds at least a whole token's tiles, a
  // split token has two parts, merged in the kernel
  pl.fused = fp8 && pl.need_combine && pl.total / pl.G >= pl.nt;
  if (pl.fused) pl.need_combine = false;
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  const size_t lse_bytes = (size_t)(((n_slots * kHeads * 4) + 255) / 256) * 256;
  pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * kHeads * kDv * 4;
  if (fp8) pl.ws_bytes += q_prep_bytes(T) + merge_bytes(T);
  return pl;
}

template <bool kFp8>
cudaError_t launch_wide(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  Params p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
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
  const size_t lse_bytes = (size_t)(((n_slots * kHeads * 4) + 255) / 256) * 256;
  p.part_lse = reinterpret_cast<float*>(ws + kWsStatusBytes);
  p.part_o = reinterpret_cast<float*>(ws + kWsStatusBytes + lse_bytes);
  p.scale_log2 = a.sm_scale * 1.4426950408889634f;
  p.T = a.T;
  p.K = a.K;
  p.N = a.NB;
  p.nt = plan.nt;
  p.total = plan.total;
  p.G = plan.G;
  const void* qsrc = a.q;
  if (kFp8) {
    // prepared Q after the partial results (256-byte aligned)
    uint8_t* qp = ws + kWsStatusBytes + lse_bytes + (size_t)n_slots * kHeads * kDv * 4;
    uint16_t* q16 = reinterpret_cast<uint16_t*>(qp);
    float* qinv = reinterpret_cast<float*>(qp + (((size_t)a.T * kHeads * kDqk * 2 + 255) / 256) * 256);
    const int64_t rows = (int64_t)a.T * kHeads;
    uint8_t* mg = qp + q_prep_bytes(a.T);
    p.merge_flag = reinterpret_cast<int*>(mg);
    p.merge_lse = reinterpret_cast<float*>(mg + (((size_t)a.T * 4 * 4 + 255) / 256) * 256);
    p.fused = plan.fused ? 1 : 0;
    wide_q_prep_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(a.q), q16,
                                                                     qinv, rows, p.merge_flag, (int64_t)a.T * 4);
    cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
    p.qinv = qinv;
    qsrc = q16;
  }
  CUtensorMap m0, m1, m2, q_map, q_rope_map;
  const void* rows = kFp8 ? static_cast<const void*>(a.cache) : a.kv;
  const int64_t n_rows = kFp8 ? a.NB * kBlock : a.NB;
  cudaError_t e = make_maps<kFp8>(rows, n_rows, qsrc, a.T, &m0, &m1, &m2, &q_map, &q_rope_map);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sparse_mla_wide_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Lay<kFp8>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  sparse_mla_wide_kernel<kFp8><<<2 * plan.G, kThreads, Lay<kFp8>::kSmemAlloc, stream>>>(p, m0, m1, m2, q_map,
                                                                                         q_rope_map);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  e = launch_combine<kHeads>(p.part_o, p.part_lse, p.out, p.lse, kHeads, 1, p.nt, p.total, p.G, plan.units, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_set_wide(long long* buf) {
  return (int)cudaMemcpyToSymbol(g_smla_trace_wide, &buf, sizeof(buf));
}
#endif

bool wide_supported(int H) { return H == kHeads; }

AttnPlan plan_prefill_wide(int T, int K, int num_splits, int num_sms) {
  return plan_wide(false, T, K, num_splits, num_sms);
}
AttnPlan plan_decode_wide(int T, int K, int num_splits, int num_sms) {
  return plan_wide(true, T, K, num_splits, num_sms);
}
cudaError_t launch_prefill_wide(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  return launch_wide<false>(a, plan, stream);
}
cudaError_t launch_decode_wide(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  return launch_wide<true>(a, plan, stream);
}

}  // namespace smla
