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
//   * the two fp32 partials are exchanged through distributed shared memory
//     (each softmax thread sends its head's 64 partial logits to the peer with
//     st.async, whose bytes complete the peer's barrier), so both CTAs hold
//     the same S = S_0 + S_1 and take identical softmax decisions;
//   * softmax, one thread per head (the head's TMEM lane): online max and sum
//     in the log2 domain with lazy rescaling of O, P in bf16 written back to
//     TMEM;
//   * P.V: O_c += P V[rows, 256c : 256c + 256], A = P from TMEM, B = the
//     value panels of the same row tile (MN-major), N = 256.
// Warp roles: 0..3 softmax, 4..7 and 8..11 exchange of tile rows 0..31 and
// 32..63 (partial logits -> full, masked, log2-domain logits back in TMEM +
// the maximum), 12 tensor-core issuer, 13 index translation + Q, 14..17 row
// loaders (TMA tile::gather4 straight into swizzled K-major operand tiles).
// Warp w of the first three groups handles heads 32 (w % 4) .. + 31 (its
// TMEM lane quarter), one per thread; the two halves' exchanges run side by
// side and overlap the softmax of the previous tile.  18 warps: at most 5 per
// sub-partition, so 96 registers per thread.  Work: pairs take contiguous balanced ranges of the
// token-major tile sequence; a token split over pairs goes through the
// LSE-weighted combine.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
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
constexpr int kKBufs = 3;                   // row tiles in flight
constexpr int kKBuf = 4 * kPanel + kRopePanel;     // 36 KB
constexpr int kQBuf = 4 * kQPanel + kQRopePanel;   // 72 KB
constexpr int kXSlot = kHeads * 32 * 4;     // 16 KB: the peer's partial logits of one half tile (32 rows)
constexpr int kRowBytesBf16 = kDqk * 2;     // 1152
constexpr int kLoaders = 4;                 // loader lw gathers rows 16 lw .. 16 lw + 15
constexpr float kMaxSlack = 8.0f;           // log2 growth of a head's max tolerated before rescaling O

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBuf;
constexpr int kOffX = kOffK + kKBufs * kKBuf;
constexpr int kOffSlots = kOffX + 2 * kXSlot;      // int32 [4][64]
constexpr int kOffValid = kOffSlots + 4 * kRows * 4;  // uint8 [2][64]
constexpr int kSBufs = 3;                              // S buffers in tensor memory
constexpr int kOffRed = kOffValid + kKBufs * kRows;    // float [kSBufs][2 halves][128]: maxima (log2 domain)
constexpr int kOffBar = kOffRed + kSBufs * 2 * kHeads * 4;
enum {
  kBarKFull = 0, kBarKEmpty = kBarKFull + kKBufs, kBarSFull = kBarKEmpty + kKBufs, kBarSReady = kBarSFull + kSBufs,
  kBarSFree = kBarSReady + kSBufs, kBarPFull = kBarSFree + kSBufs, kBarPDone = kBarPFull + 2, kBarXFull = kBarPDone + 2,
  kBarXFree = kBarXFull + 2, kBarIdxFull = kBarXFree + 2, kBarIdxEmpty = kBarIdxFull + 4, kBarQFull = kBarIdxEmpty + 4,
  kBarQEmpty = kBarQFull + 1, kBarOFree = kBarQEmpty + 1, kBarDrain = kBarOFree + 1, kNumBars = kBarDrain + 1
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kOffK % 1024 == 0 && kOffX % 1024 == 0 && kKBuf % 1024 == 0, "operand alignment");
static_assert((4 * kPanel) % 512 == 0 && (4 * kQPanel) % 512 == 0, "64-byte-swizzle atoms are 512 bytes");
static_assert(kOffBar % 8 == 0 && kOffRed % 16 == 0, "alignment");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// tensor memory columns
constexpr int kOCol = 0;    // O_c: 256 fp32 columns
constexpr int kSCol = 256;  // S: 3 buffers x 64 columns
constexpr int kPCol = 448;  // P: 2 buffers x 32 columns (bf16 pairs)
constexpr int kTmemCols = 512;

constexpr int kSoftWarps = 4, kXchgWarp0 = 4, kXchgWarps = 8, kMmaWarp = 12, kIndexWarp = 13, kLoadWarp0 = 14;
constexpr int kNumWarps = kLoadWarp0 + kLoaders;
constexpr int kThreads = 32 * kNumWarps;

// Optional per-tile timeline for performance work: with SMLA_TRACE defined,
// roles record clock64() at their hand-off points into g_smla_trace_wide
// (set by the host through smla_trace_set_wide).  Compiled out otherwise.
#ifdef SMLA_TRACE
__device__ long long* g_smla_trace_wide = nullptr;
constexpr int kTraceTiles = 64, kTraceEvents = 12;
#define WIDE_TRACE(tl, ev)                                                                                   \
  do {                                                                                                       \
    if (g_smla_trace_wide && (tl) < kTraceTiles)                                                           \
      g_smla_trace_wide[((size_t)blockIdx.x * kTraceTiles + (tl)) * kTraceEvents + (ev)] = clock64();     \
  } while (0)
#else
#define WIDE_TRACE(tl, ev) ((void)0)
#endif
enum { kEvSFull = 0, kEvSLoaded, kEvXFree, kEvSent, kEvXFull, kEvPReady, kEvPFull, kEvQk, kEvPv, kEvIssue, kEvQkSeen,
       kEvKEmpty };

struct Params {
  const __nv_bfloat16* q;  // [T, 128, 576]
  const int32_t* indices;  // [T, K]
  __nv_bfloat16* out;      // [T, 128, 512]
  float* lse;              // [T, 128]
  float* part_o;           // [slots, 128, 512]
  float* part_lse;         // [slots, 128]
  int* status;
  float scale_log2;        // softmax_scale * log2(e)
  int T, K;
  int64_t N;               // kv rows
  int nt;                  // tiles per token
  int64_t total;           // T * nt
  int G;                   // pairs
};

struct TileInfo {
  int u, kt;
  bool seg_start, seg_end;
};

__device__ __forceinline__ TileInfo tile_info(const Params& p, int64_t x, int64_t xbeg, int64_t xend) {
  TileInfo ti;
  ti.u = (int)(x / p.nt);
  ti.kt = (int)(x - (int64_t)ti.u * p.nt);
  ti.seg_start = (x == xbeg) || (ti.kt == 0);
  ti.seg_end = (x == xend - 1) || (ti.kt == p.nt - 1);
  return ti;
}

__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(96)
    sparse_mla_wide_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap kv_map,
                           const __grid_constant__ CUtensorMap kv_rope_map, const __grid_constant__ CUtensorMap q_map,
                           const __grid_constant__ CUtensorMap q_rope_map) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + kOffSlots);
  uint8_t* valid = smem + kOffValid;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = (int)cluster_ctarank();  // value half owned by this CTA
  const int pair = blockIdx.x >> 1;
  const int64_t xbeg = tile_begin(pair, p.total, p.G);
  const int64_t xend = tile_begin(pair + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);

  if (tid == 0) {
    for (int i = 0; i < kKBufs; ++i) {
      mbar_init(&bars[kBarKFull + i], kLoaders);
      mbar_init(&bars[kBarKEmpty + i], 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarSReady + i], 32 * kXchgWarps);
      mbar_init(&bars[kBarSFree + i], 32 * kSoftWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarPFull + i], 32 * kSoftWarps);
      mbar_init(&bars[kBarPDone + i], 1);
    }
    for (int i = 0; i < 2; ++i) {               // exchange slot i carries half i of every tile
      mbar_init(&bars[kBarXFull + i], 1);           // own expect_tx + the peer's st.async bytes
      mbar_init(&bars[kBarXFree + i], kSoftWarps);  // one arrival per peer exchange warp
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarIdxFull + i], 32);
      mbar_init(&bars[kBarIdxEmpty + i], kLoaders);
    }
    mbar_init(&bars[kBarQFull], 1);
    mbar_init(&bars[kBarQEmpty], 1);
    mbar_init(&bars[kBarOFree], 32 * kSoftWarps);
    mbar_init(&bars[kBarDrain], 1);
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
      if (tl >= 4 && !SMLA_WAIT(kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = lane + 32 * i;
        const int k = ti.kt * kRows + r;
        int32_t s = -1;
        if (k < p.K) {
          const int32_t idx = __ldg(p.indices + (int64_t)ti.u * p.K + k);
          s = (idx >= 0 && (int64_t)idx < p.N) ? idx : -1;
        }
        slots_ring[b4 * kRows + r] = s;
      }
      mbar_arrive(&bars[kBarIdxFull + b4]);
      if (ti.seg_start) {
        // the segment's Q block, once the previous segment's last QK^T is done
        if (seg >= 1 && !SMLA_WAIT(kBarQEmpty, (seg - 1) & 1)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[kBarQFull], (uint32_t)kQBuf);
          for (int b = 0; b < 4; ++b)
            tma_load_2d(smem_u32(smem + kOffQ + b * kQPanel), &q_map, 128 * (4 * c + b), ti.u * kHeads,
                        &bars[kBarQFull]);
          tma_load_2d(smem_u32(smem + kOffQ + 4 * kQPanel), &q_rope_map, 2 * kDv + 64 * c, ti.u * kHeads,
                      &bars[kBarQFull]);
        }
        __syncwarp();
        ++seg;
      }
    }
    // no Q copy may still be landing in shared memory when the CTA exits
    if (seg > 0 && lane == 0) mbar_wait_drain(&bars[kBarQFull], (seg - 1) & 1);
    __syncwarp();
  } else if (warp >= kLoadWarp0) {
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
      const int b4 = tl & 3, kb = tl % kKBufs, use = tl / kKBufs;
      if (!SMLA_WAIT(kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = lane < 16 ? slots_ring[b4 * kRows + 16 * lw + lane] : -1;
      const uint32_t vmask = __ballot_sync(kFullMask, slot >= 0);
      const int g0 = __shfl_sync(kFullMask, slot, (4 * grp) & 31), g1 = __shfl_sync(kFullMask, slot, (4 * grp + 1) & 31);
      const int g2 = __shfl_sync(kFullMask, slot, (4 * grp + 2) & 31), g3 = __shfl_sync(kFullMask, slot, (4 * grp + 3) & 31);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarIdxEmpty + b4]);
      if (use >= 1 && !SMLA_WAIT(kBarKEmpty + kb, (use + 1) & 1)) break;
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvKEmpty);
      if (lane < 16) valid[kb * kRows + 16 * lw + lane] = (uint8_t)((vmask >> lane) & 1u);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarKFull + kb], (uint32_t)(16 * (kKBuf / kRows)));
      __syncwarp();
      if (lane < 20) {
        const uint32_t tile = smem_u32(smem + kOffK + kb * kKBuf);
        if (box < 4)
          tma_gather4_2d(tile + box * kPanel + (uint32_t)((r_g >> 3) * 1024 + (r_g & 7) * 128), &kv_map,
                         128 * (4 * c + box), g0, g1, g2, g3, &bars[kBarKFull + kb]);
        else
          tma_gather4_2d(tile + 4 * kPanel + (uint32_t)((r_g >> 3) * 512 + (r_g & 7) * 64), &kv_rope_map,
                         2 * kDv + 64 * c, g0, g1, g2, g3, &bars[kBarKFull + kb]);
      }
      if (lane == 0 && lw == 0) WIDE_TRACE(tl, kEvIssue);
      last_b = kb;
      last_use = use;
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (last_b >= 0) mbar_wait_drain(&bars[kBarKFull + last_b], last_use & 1);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor-core issuer
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_qk = make_idesc_bf16(128, kRows, 0, 0);
      constexpr uint32_t id_pv = make_idesc_bf16(128, 256, 0, 1);
      const uint32_t q0 = smem_u32(smem + kOffQ), k0 = smem_u32(smem + kOffK);  // 1024-byte aligned
      int seg_q = 0, seg_o = 0, next_qk = 0, next_pv = 0;
      const int kt0 = (int)(xbeg % p.nt);
      int kt_qk = kt0, kt_pv = kt0;
      uint64_t t_idle = 0;
      uint32_t idle_polls = 0;
      // shared-memory descriptors: constant high words, low words = base + offset / 16
      constexpr uint32_t kHi128 = sdesc_hi(1024, kLayoutSw128), kHi64 = sdesc_hi(512, kLayoutSw64);
      const uint32_t dq = sdesc_lo(q0, 16), dk0 = sdesc_lo(k0, 16), dv0 = sdesc_lo(k0, kPanel);
      // P.V of tile next_pv once its P is written (and, first in a segment, O
      // is free).  Tried before every QK^T panel too: its completion frees the
      // row tile the loaders wait for, so it never waits out a whole QK^T.
      auto try_pv = [&]() -> bool {
        if (next_pv >= next_qk) return false;
        const int tl = next_pv, kb = tl % kKBufs, pb = tl & 1;
        const bool seg_start = tl == 0 || kt_pv == 0;
        const bool o_ok = !seg_start || seg_o == 0 || mbar_test_wait(&bars[kBarOFree], (seg_o - 1) & 1);
        if (!o_ok || !mbar_test_wait(&bars[kBarPFull + pb], (tl >> 1) & 1)) return false;
        if (seg_start) ++seg_o;
        tc_fence_after();
        const uint32_t dv = dv0 + ((kb * kKBuf) >> 4);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          // B = V rows 16 s .. 16 s + 15 x 256 value columns, MN-major:
          // 64-column panels kPanel apart, 8-row groups 1024 bytes apart
          mma_ts(tmem + kOCol, tmem + kPCol + 32 * pb + 8 * s, sdesc_join<kHi128>(dv + ((2048 * s) >> 4)), id_pv,
                 (seg_start && s == 0) ? 0u : 1u);
        mma_commit(&bars[kBarKEmpty + kb]);
        mma_commit(&bars[kBarPDone + pb]);
        WIDE_TRACE(tl, kEvPv);
        ++next_pv;
        kt_pv = kt_pv + 1 == p.nt ? 0 : kt_pv + 1;
        return true;
      };
      while (next_pv < n_local) {
        bool progressed = try_pv();
        // QK^T of tile next_qk: its rows, the segment's Q and a free S buffer
        if (next_qk < n_local) {
          const int tl = next_qk, kb = tl % kKBufs, sb = tl % kSBufs;
          const bool seg_start = tl == 0 || kt_qk == 0;
          const bool seg_end = tl == n_local - 1 || kt_qk == p.nt - 1;
          const int seg = seg_start ? seg_q : seg_q - 1;
          const bool s_ok = tl < kSBufs || mbar_test_wait(&bars[kBarSFree + sb], ((tl / kSBufs) + 1) & 1);
          const bool q_ok = !seg_start || mbar_test_wait(&bars[kBarQFull], seg & 1);
          if (s_ok && q_ok && mbar_test_wait(&bars[kBarKFull + kb], (tl / kKBufs) & 1)) {
            if (seg_start) ++seg_q;
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
              try_pv();
            }
#pragma unroll
            for (int s = 0; s < 2; ++s)  // RoPE half: 8-row atoms of 64 bytes
              mma_ss(sacc, sdesc_join<kHi64>(dq + ((4 * kQPanel + 32 * s) >> 4)),
                     sdesc_join<kHi64>(dk + ((4 * kPanel + 32 * s) >> 4)), id_qk, 1u);
            mma_commit(&bars[kBarSFull + sb]);
            if (seg_end) mma_commit(&bars[kBarQEmpty]);
            WIDE_TRACE(tl, kEvQk);
            ++next_qk;
            kt_qk = kt_qk + 1 == p.nt ? 0 : kt_qk + 1;
            progressed = true;
          }
        }
        if (progressed) {
          t_idle = 0;
          idle_polls = 0;
        } else if ((++idle_polls & 255u) == 0u) {
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
      // every issued tensor-core operation completes before tensor memory is released
      if (next_qk > 0) {
        mma_commit(&bars[kBarDrain]);
        mbar_wait_drain(&bars[kBarDrain], 0);
      }
    }
    __syncwarp();
  } else {
    const int qd = warp & 3;
    const int h = 32 * qd + lane;  // head = TMEM lane of S, P and O
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    if (warp >= kXchgWarp0) {
      // ---------------------------------------------------------- exchange (warps 4..11)
      // Warp group e handles half e of every tile (rows 32 e .. 32 e + 31,
      // exchange slot e): the
      // partial logits go to the peer (st.async into its slot, the bytes
      // completing its barrier; chunk i of head h at 16-byte slot (i + h) % 8 so
      // a warp's stores spread over the banks, the reader using the same
      // placement), the peer's partial is added, rows are masked and scaled to
      // the log2 domain, and the result is written back over the S buffer.  A
      // half is sent once the peer has read the same half of the previous tile.
      const uint32_t peer = (uint32_t)(c ^ 1);
      const uint32_t x_local = smem_u32(smem + kOffX) + (uint32_t)(h * 128);
      const uint32_t x_remote = mapa_shared(x_local, peer);
      const uint32_t xfull_remote = mapa_shared(smem_u32(&bars[kBarXFull]), peer);
      const uint32_t xfree_remote = mapa_shared(smem_u32(&bars[kBarXFree]), peer);
      const int e = (warp - kXchgWarp0) >> 2;
      const bool lead = lane == 0 && qd == 0;  // registers the slot's expected bytes
      bool dead = false;
      for (int tl = 0; tl < n_local; ++tl) {
        const int sb = tl % kSBufs, kb = tl % kKBufs;
        // row validity (written by the loaders before the tile's full barrier)
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
        if (!dead) dead = !SMLA_WAIT(kBarSFull + sb, (tl / kSBufs) & 1);
        if (tid == 32 * kXchgWarp0) WIDE_TRACE(tl, kEvSFull);
        tc_fence_after();
        float mt = -INFINITY;
        {
          const uint32_t scol = tmem + lane_base + kSCol + 64 * sb + 32 * e;
          if (lead) mbar_arrive_expect_tx(&bars[kBarXFull + e], (uint32_t)kXSlot);
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
          }
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvSLoaded);
          if (tl >= 1 && !dead) dead = !SMLA_WAIT_X(kBarXFree + e, (tl - 1) & 1);
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvXFree);
          if (!dead) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              st_async_v4(x_remote + e * kXSlot + 16 * ((i + h) & 7), s[4 * i], s[4 * i + 1], s[4 * i + 2],
                          s[4 * i + 3], xfull_remote + 8 * e);
          }
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvSent);
          if (!dead) dead = !SMLA_WAIT_X(kBarXFull + e, tl & 1);
          if (tid == 32 * kXchgWarp0 && e == 0) WIDE_TRACE(tl, kEvXFull);
          if (!dead) {
            const uint8_t* src = smem + kOffX + e * kXSlot + h * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 v = *reinterpret_cast<const float4*>(src + 16 * ((i + h) & 7));
              s[4 * i] += v.x;
              s[4 * i + 1] += v.y;
              s[4 * i + 2] += v.z;
              s[4 * i + 3] += v.w;
            }
          }
          // the slot's values are in registers: the peer may overwrite it
          __syncwarp();
          if (!dead && lane == 0) mbar_arrive_cluster_relaxed(xfree_remote + 8 * e);
          uint32_t r[2][16];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = (vb >> j) & 1u ? s[j] * p.scale_log2 : -INFINITY;
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
        mbar_arrive(&bars[kBarSReady + sb]);
        if (tid == 32 * kXchgWarp0) WIDE_TRACE(tl, kEvPReady);
      }
    } else {
      // ---------------------------------------------------------- softmax + epilogue (warps 0..3)
      float m_used = -INFINITY, l_sum = 0.f;
      int n_seg_tiles = 0;
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
        if (!dead) dead = !SMLA_WAIT(kBarSReady + sb, (tl / kSBufs) & 1);
        tc_fence_after();
        const float mt = fmaxf(red[(sb * 2) * kHeads + h], red[(sb * 2 + 1) * kHeads + h]);
        // A head whose max grew by more than kMaxSlack takes the new max; when
        // O already holds earlier tiles of the segment its row is scaled by
        // a = 2^(m_used - m_new).
        const bool need = mt > m_used + kMaxSlack || (m_used == -INFINITY && mt > -INFINITY);
        const bool scale_o = need && n_seg_tiles > 0 && m_used > -INFINITY;
        const float a = scale_o ? ex2_approx(m_used - mt) : 1.f;
        if (need) m_used = mt;
        // TMEM access is warp-wide: a warp with any head to rescale runs the
        // pass (factor 1 for its other heads), once P.V(tl - 1) has landed in O
        if (__any_sync(kFullMask, scale_o)) {
          if (!dead) dead = !SMLA_WAIT(kBarPDone + ((tl - 1) & 1), ((tl - 1) >> 1) & 1);
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
        if (tl >= 2 && !dead) dead = !SMLA_WAIT(kBarPDone + pb, ((tl >> 1) + 1) & 1);
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
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float p0 = none ? 0.f : ex2_approx(__uint_as_float(r0[2 * j]) - m_used);
            const float p1 = none ? 0.f : ex2_approx(__uint_as_float(r0[2 * j + 1]) - m_used);
            const float p2 = none ? 0.f : ex2_approx(__uint_as_float(r1[2 * j]) - m_used);
            const float p3 = none ? 0.f : ex2_approx(__uint_as_float(r1[2 * j + 1]) - m_used);
            l0 += p0 + p2;
            l1 += p1 + p3;
            pk[j] = pack_bf16x2(p0, p1);
            pk[8 + j] = pack_bf16x2(p2, p3);
          }
          lt += l0 + l1;
          tmem_st16(tmem + lane_base + kPCol + 32 * pb + 16 * e, pk);
        }
        tc_fence_before();
        mbar_arrive(&bars[kBarSFree + sb]);
        l_sum = l_sum * a + lt;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars[kBarPFull + pb]);
        if (tid == 0) WIDE_TRACE(tl, kEvPFull);
        ++n_seg_tiles;
        // epilogue at the end of a segment
        if (seg_end) {
          if (!dead) dead = !SMLA_WAIT(kBarPDone + pb, (tl >> 1) & 1);
          tc_fence_after();
          const bool full_unit = n_seg_tiles == p.nt;  // the whole token ran in this pair
          const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
          const int64_t slot = (int64_t)pair + u;
          for (int q = 0; q < 256 / 16; ++q) {
            uint32_t r[16];
            tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
            if (dead) continue;
            if (full_unit) {
              uint32_t ow[8];
#pragma unroll
              for (int j = 0; j < 8; ++j)
                ow[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
              uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)u * kHeads + h) * kDv + 256 * c + 16 * q);
              dst[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
              dst[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
            } else {
              float4* dst = reinterpret_cast<float4*>(p.part_o + (slot * kHeads + h) * kDv + 256 * c + 16 * q);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_float4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                                     __uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv);
            }
          }
          if (!dead && c == 0) {
            const float lse_v = l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
            if (full_unit)
              p.lse[(int64_t)u * kHeads + h] = lse_v;
            else
              p.part_lse[slot * kHeads + h] = lse_v;
          }
          tc_fence_before();
          mbar_arrive(&bars[kBarOFree]);
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
}

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

// kv [N, 576] bf16 and q [T * 128, 576] bf16, both as bytes.  The kv maps
// gather single rows: one 128-byte value panel (128-byte swizzle) or one
// 64-byte RoPE half (64-byte swizzle); the q maps load the same slices of
// 128 consecutive head rows.
cudaError_t make_maps(const void* kv, int64_t N, const void* q, int T, CUtensorMap* kv_map, CUtensorMap* kv_rope_map,
                      CUtensorMap* q_map, CUtensorMap* q_rope_map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gstride[1] = {(cuuint64_t)kRowBytesBf16};
  const cuuint32_t es[2] = {1, 1};
  const cuuint64_t kv_dim[2] = {(cuuint64_t)kRowBytesBf16, (cuuint64_t)N};
  const cuuint64_t q_dim[2] = {(cuuint64_t)kRowBytesBf16, (cuuint64_t)T * kHeads};
  struct Spec {
    CUtensorMap* map;
    const void* base;
    const cuuint64_t* dim;
    cuuint32_t box0, box1;
    CUtensorMapSwizzle sw;
  } specs[4] = {{kv_map, kv, kv_dim, 128, 1, CU_TENSOR_MAP_SWIZZLE_128B},
                {kv_rope_map, kv, kv_dim, 64, 1, CU_TENSOR_MAP_SWIZZLE_64B},
                {q_map, q, q_dim, 128, kHeads, CU_TENSOR_MAP_SWIZZLE_128B},
                {q_rope_map, q, q_dim, 64, kHeads, CU_TENSOR_MAP_SWIZZLE_64B}};
  for (const Spec& sp : specs) {
    const cuuint32_t box[2] = {sp.box0, sp.box1};
    const CUresult r = enc(sp.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(sp.base), sp.dim, gstride, box,
                           es, CU_TENSOR_MAP_INTERLEAVE_NONE, sp.sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Pairs that can be resident at once (one CTA per SM), looked up once per device.
int resident_pairs(int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaFuncSetAttribute(sparse_mla_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    if (cudaOccupancyMaxActiveClusters(&n, (void*)sparse_mla_wide_kernel, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n <= 0) n = num_sms / 2;
  cached[dev] = n;
  return n;
}

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_set_wide(long long* buf) {
  return (int)cudaMemcpyToSymbol(g_smla_trace_wide, &buf, sizeof(buf));
}
#endif

bool wide_prefill_supported(int H) { return H == kHeads; }

AttnPlan plan_prefill_wide(int T, int K, int num_splits, int num_sms) {
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
  const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
  const size_t lse_bytes = (size_t)(((n_slots * kHeads * 4) + 255) / 256) * 256;
  pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * kHeads * kDv * 4;
  return pl;
}

cudaError_t launch_prefill_wide(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  Params p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.indices = a.indices;
  p.out = static_cast<__nv_bfloat16*>(a.out);
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
  CUtensorMap kv_map, kv_rope_map, q_map, q_rope_map;
  cudaError_t e = make_maps(a.kv, a.NB, a.q, a.T, &kv_map, &kv_rope_map, &q_map, &q_rope_map);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sparse_mla_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  sparse_mla_wide_kernel<<<2 * plan.G, kThreads, kSmemAlloc, stream>>>(p, kv_map, kv_rope_map, q_map, q_rope_map);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  combine_kernel<kHeads><<<(unsigned)(plan.units * combine_split<kHeads>()), combine_threads<kHeads>(), 0, stream>>>(
      p.part_o, p.part_lse, p.out, p.lse, kHeads, 1, p.nt, p.total, p.G);
  return cudaGetLastError();
}

}  // namespace smla
