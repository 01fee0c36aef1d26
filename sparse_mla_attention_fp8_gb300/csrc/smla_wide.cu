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
// owns value columns [256c, 256c + 256) and the feature panels it needs:
//   CTA 0: value panels 0..3 (features 0..255) and the RoPE panel (512..575),
//   CTA 1: value panels 4..7 (features 256..511),
// each panel being 64 features.  Per 64-row tile:
//   * QK^T partial: S_c = Q[:, F_c] kv[rows, F_c]^T, M = 128 heads, N = 64
//     rows, K = the CTA's panels (tcgen05.mma kind::f16, fp32 in TMEM);
//   * the two fp32 partials are exchanged through distributed shared memory
//     (each softmax thread stores its head's 64 partial logits into the peer
//     and arrives on the peer's barrier), so both CTAs hold the same
//     S = S_0 + S_1 and take identical softmax decisions;
//   * softmax, one thread per head (the head's TMEM lane): online max and sum
//     in the log2 domain with lazy rescaling of O, P in bf16 written back to
//     TMEM;
//   * P.V: O_c += P V[rows, 256c : 256c + 256], A = P from TMEM, B = the
//     value panels of the same row tile (MN-major), N = 256.
// Warp roles: 0..3 softmax, 4 tensor-core issuer, 5 index translation + Q,
// 6..13 row loaders (TMA tile::gather4 straight into 128-byte-swizzled
// K-major operand tiles).  Work: pairs take contiguous balanced ranges of the
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
constexpr int kPanels = 5;                  // panel slots per CTA (CTA 1 uses 4)
constexpr int kKBufs = 2;                   // row tiles in flight
constexpr int kKBuf = kPanels * kPanel;     // 40 KB
constexpr int kQBuf = kPanels * kQPanel;    // 80 KB
constexpr int kXBuf = kHeads * kRows * 4;   // 32 KB: the peer's partial logits
constexpr int kRowBytesBf16 = kDqk * 2;     // 1152
constexpr int kLoaders = 8;                 // loader lw gathers rows 8 lw .. 8 lw + 7
constexpr float kMaxSlack = 8.0f;           // log2 growth of a head's max tolerated before rescaling O

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBuf;
constexpr int kOffX = kOffK + kKBufs * kKBuf;
constexpr int kOffSlots = kOffX + 2 * kXBuf;       // int32 [4][64]
constexpr int kOffValid = kOffSlots + 4 * kRows * 4;  // uint8 [2][64]
constexpr int kOffBar = kOffValid + kKBufs * kRows;
enum {
  kBarKFull = 0, kBarKEmpty = kBarKFull + kKBufs, kBarSFull = kBarKEmpty + kKBufs, kBarSFree = kBarSFull + 2,
  kBarPFull = kBarSFree + 2, kBarPDone = kBarPFull + 2, kBarXFull = kBarPDone + 2, kBarXFree = kBarXFull + 2,
  kBarIdxFull = kBarXFree + 2, kBarIdxEmpty = kBarIdxFull + 4, kBarQFull = kBarIdxEmpty + 4,
  kBarQEmpty = kBarQFull + 1, kBarOFree = kBarQEmpty + 1, kBarDrain = kBarOFree + 1, kNumBars = kBarDrain + 1
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kOffK % 1024 == 0 && kOffX % 1024 == 0 && kKBuf % 1024 == 0, "operand alignment");
static_assert(kOffBar % 8 == 0, "barrier alignment");
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// tensor memory columns
constexpr int kOCol = 0;    // O_c: 256 fp32 columns
constexpr int kSCol = 256;  // S: 2 buffers x 64 columns
constexpr int kPCol = 384;  // P: 2 buffers x 32 columns (bf16 pairs)
constexpr int kTmemCols = 512;

constexpr int kSoftWarps = 4, kMmaWarp = 4, kIndexWarp = 5, kLoadWarp0 = 6;
constexpr int kNumWarps = kLoadWarp0 + kLoaders;
constexpr int kThreads = 32 * kNumWarps;

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

// Global feature panel held in panel slot b of CTA c.
__device__ __forceinline__ int global_panel(int c, int b) { return c == 0 ? (b < 4 ? b : 8) : 4 + b; }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    sparse_mla_wide_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap kv_map,
                           const __grid_constant__ CUtensorMap q_map) {
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
  const int np = c == 0 ? 5 : 4;         // feature panels of this CTA
  const int pair = blockIdx.x >> 1;
  const int64_t xbeg = tile_begin(pair, p.total, p.G);
  const int64_t xend = tile_begin(pair + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);

  if (tid == 0) {
    for (int i = 0; i < kKBufs; ++i) {
      mbar_init(&bars[kBarKFull + i], kLoaders);
      mbar_init(&bars[kBarKEmpty + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarSFree + i], 32 * kSoftWarps);
      mbar_init(&bars[kBarPFull + i], 32 * kSoftWarps);
      mbar_init(&bars[kBarPDone + i], 1);
      mbar_init(&bars[kBarXFull + i], 32 * kSoftWarps);
      mbar_init(&bars[kBarXFree + i], 32 * kSoftWarps);
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
          mbar_arrive_expect_tx(&bars[kBarQFull], (uint32_t)(np * kQPanel));
          for (int b = 0; b < np; ++b)
            tma_load_2d(smem_u32(smem + kOffQ + b * kQPanel), &q_map, 128 * global_panel(c, b), ti.u * kHeads,
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
    // Loader lw gathers rows 8 lw .. 8 lw + 7 of every tile: 2 groups of 4
    // rows x np panels, lane np * g + b issuing panel b of group g.  Its one
    // arrival on the tile's full barrier carries the bytes of its 8 rows and
    // follows its writes of the rows' valid flags.
    const int lw = warp - kLoadWarp0;
    const int grp = lane / np, box = lane - grp * np;
    const int r_g = 8 * lw + 4 * grp;  // tile row of the lane's group
    int last_b = -1, last_use = 0;
    for (int tl = 0; tl < n_local; ++tl) {
      const int b4 = tl & 3, kb = tl & 1, use = tl >> 1;
      if (!SMLA_WAIT(kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = lane < 8 ? slots_ring[b4 * kRows + 8 * lw + lane] : -1;
      const uint32_t vmask = __ballot_sync(kFullMask, slot >= 0);
      const int g0 = __shfl_sync(kFullMask, slot, (4 * grp) & 31), g1 = __shfl_sync(kFullMask, slot, (4 * grp + 1) & 31);
      const int g2 = __shfl_sync(kFullMask, slot, (4 * grp + 2) & 31), g3 = __shfl_sync(kFullMask, slot, (4 * grp + 3) & 31);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarIdxEmpty + b4]);
      if (use >= 1 && !SMLA_WAIT(kBarKEmpty + kb, (use + 1) & 1)) break;
      if (lane < 8) valid[kb * kRows + 8 * lw + lane] = (uint8_t)((vmask >> lane) & 1u);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarKFull + kb], (uint32_t)(8 * np * 128));
      __syncwarp();
      if (lane < 2 * np) {
        const uint32_t dst = smem_u32(smem + kOffK + kb * kKBuf + box * kPanel) + (uint32_t)((r_g >> 3) * 1024 + (r_g & 7) * 128);
        tma_gather4_2d(dst, &kv_map, 128 * global_panel(c, box), g0, g1, g2, g3, &bars[kBarKFull + kb]);
      }
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
      const uint32_t q0 = smem_u32(smem + kOffQ), k0 = smem_u32(smem + kOffK);
      int seg_q = 0, seg_o = 0, next_qk = 0, next_pv = 0;
      const int kt0 = (int)(xbeg % p.nt);
      int kt_qk = kt0, kt_pv = kt0;
      uint64_t t_idle = 0;
      uint32_t idle_polls = 0;
      while (next_pv < n_local) {
        bool progressed = false;
        // QK^T of tile next_qk: its rows, the segment's Q and a free S buffer
        if (next_qk < n_local && next_qk < next_pv + 2) {
          const int tl = next_qk, kb = tl & 1;
          const bool seg_start = tl == 0 || kt_qk == 0;
          const bool seg_end = tl == n_local - 1 || kt_qk == p.nt - 1;
          const int seg = seg_start ? seg_q : seg_q - 1;
          const bool s_ok = tl < 2 || mbar_test_wait(&bars[kBarSFree + kb], ((tl >> 1) + 1) & 1);
          const bool q_ok = !seg_start || mbar_test_wait(&bars[kBarQFull], seg & 1);
          if (s_ok && q_ok && mbar_test_wait(&bars[kBarKFull + kb], (tl >> 1) & 1)) {
            if (seg_start) ++seg_q;
            tc_fence_after();
            const uint32_t kt = k0 + kb * kKBuf;
            for (int b = 0; b < np; ++b) {
#pragma unroll
              for (int s = 0; s < 4; ++s) {
                const uint64_t da = make_sdesc(q0 + b * kQPanel + 32 * s, 16, 1024, kLayoutSw128);
                const uint64_t db = make_sdesc(kt + b * kPanel + 32 * s, 16, 1024, kLayoutSw128);
                mma_ss(tmem + kSCol + 64 * kb, da, db, id_qk, (b | s) != 0 ? 1u : 0u);
              }
            }
            mma_commit(&bars[kBarSFull + kb]);
            if (seg_end) mma_commit(&bars[kBarQEmpty]);
            ++next_qk;
            kt_qk = kt_qk + 1 == p.nt ? 0 : kt_qk + 1;
            progressed = true;
          }
        }
        // P.V of tile next_pv: its P (and, first in a segment, a free O)
        if (next_pv < next_qk) {
          const int tl = next_pv, kb = tl & 1;
          const bool seg_start = tl == 0 || kt_pv == 0;
          const bool o_ok = !seg_start || seg_o == 0 || mbar_test_wait(&bars[kBarOFree], (seg_o - 1) & 1);
          if (o_ok && mbar_test_wait(&bars[kBarPFull + kb], (tl >> 1) & 1)) {
            if (seg_start) ++seg_o;
            tc_fence_after();
            const uint32_t kt = k0 + kb * kKBuf;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              // B = V rows 16 s .. 16 s + 15 x 256 value columns, MN-major:
              // 64-column panels kPanel apart, 8-row groups 1024 bytes apart
              const uint64_t db = make_sdesc(kt + 2048 * s, kPanel, 1024, kLayoutSw128);
              mma_ts(tmem + kOCol, tmem + kPCol + 32 * kb + 8 * s, db, id_pv, (seg_start && s == 0) ? 0u : 1u);
            }
            mma_commit(&bars[kBarKEmpty + kb]);
            mma_commit(&bars[kBarPDone + kb]);
            ++next_pv;
            kt_pv = kt_pv + 1 == p.nt ? 0 : kt_pv + 1;
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
    // ------------------------------------------------------------ softmax + epilogue (warps 0..3)
    // Thread (w, lane) owns head h = 32 w + lane: TMEM lane h of S, P and O.
    const int h = tid;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const uint32_t peer = (uint32_t)(c ^ 1);
    // this head's row of the peer's partial-logit buffers, and the peer's barriers
    const uint32_t x_local = smem_u32(smem + kOffX) + (uint32_t)h * (kRows * 4);
    const uint32_t x_remote = mapa_shared(x_local, peer);
    const uint32_t xfull_remote = mapa_shared(smem_u32(&bars[kBarXFull]), peer);
    const uint32_t xfree_remote = mapa_shared(smem_u32(&bars[kBarXFree]), peer);
    float m_used = -INFINITY, l_sum = 0.f;
    int n_seg_tiles = 0;
    bool dead = false;
    int64_t x = xbeg;
    for (int tl = 0; tl < n_local; ++tl, ++x) {
      const TileInfo ti = tile_info(p, x, xbeg, xend);
      const int kb = tl & 1;
      if (ti.seg_start) {
        m_used = -INFINITY;
        l_sum = 0.f;
        n_seg_tiles = 0;
      }
      // 1. own partial logits
      if (!dead) dead = !SMLA_WAIT(kBarSFull + kb, (tl >> 1) & 1);
      tc_fence_after();
      float s[kRows];
      {
        uint32_t r[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tmem + lane_base + kSCol + 64 * kb + 16 * q, r[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          reg_fence16(r[q]);
#pragma unroll
          for (int j = 0; j < 16; ++j) s[16 * q + j] = __uint_as_float(r[q][j]);
        }
      }
      tc_fence_before();
      mbar_arrive(&bars[kBarSFree + kb]);
      // 2. exchange with the peer: store ours into its buffer kb (chunk i of
      // head h at 16-byte slot (i + h) % 16, so a warp's stores spread over the
      // banks; the reader uses the same placement)
      if (tl >= 2 && !dead) dead = !SMLA_WAIT_X(kBarXFree + kb, ((tl >> 1) + 1) & 1);
      if (!dead) {
        const uint32_t dst = x_remote + (uint32_t)kb * kXBuf;
#pragma unroll
        for (int i = 0; i < kRows / 4; ++i)
          st_cluster_v4(dst + 16 * ((i + h) & (kRows / 4 - 1)), s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
        mbar_arrive_cluster(xfull_remote + 8 * kb);
      }
      if (!dead) dead = !SMLA_WAIT_X(kBarXFull + kb, (tl >> 1) & 1);
      if (!dead) {
        const uint8_t* src = smem + kOffX + kb * kXBuf + h * (kRows * 4);
#pragma unroll
        for (int i = 0; i < kRows / 4; ++i) {
          const float4 v = *reinterpret_cast<const float4*>(src + 16 * ((i + h) & (kRows / 4 - 1)));
          s[4 * i] += v.x;
          s[4 * i + 1] += v.y;
          s[4 * i + 2] += v.z;
          s[4 * i + 3] += v.w;
        }
        mbar_arrive_cluster(xfree_remote + 8 * kb);
      }
      // 3. row validity (written by the loaders before the tile's full barrier)
      if (!dead) dead = !SMLA_WAIT(kBarKFull + kb, (tl >> 1) & 1);
      uint32_t vbits[2] = {0u, 0u};
      {
        const uint4* vf = reinterpret_cast<const uint4*>(valid + kb * kRows);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 w4 = vf[i];
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // bytes are 0 or 1: gather bit 0 of each byte
            uint32_t b = w[k] & 0x01010101u;
            b = (b | (b >> 7)) & 0x00030003u;
            b = (b | (b >> 14)) & 0xFu;
            vbits[i >> 1] |= b << (4 * (4 * (i & 1) + k));
          }
        }
      }
      // 4. online softmax in the log2 domain
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        const bool ok = (vbits[j >> 5] >> (j & 31)) & 1u;
        s[j] = ok ? s[j] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
      // A head whose max grew by more than kMaxSlack takes the new max; when
      // O already holds earlier tiles of the segment its row is scaled by
      // 2^(m_used - m_new).  TMEM access is warp-wide, so a warp with any such
      // head runs the scaling pass (factor 1 for its other heads).
      const bool need = mt > m_used + kMaxSlack || (m_used == -INFINITY && mt > -INFINITY);
      if (__any_sync(kFullMask, need)) {
        const float m_new = need ? mt : m_used;
        const bool scale_o = need && n_seg_tiles > 0 && m_used > -INFINITY;
        if (__any_sync(kFullMask, scale_o)) {
          // O holds P.V of the segment's earlier tiles once the last one is done
          if (!dead) dead = !SMLA_WAIT(kBarPDone + ((tl - 1) & 1), ((tl - 1) >> 1) & 1);
          tc_fence_after();
          const float a = scale_o ? exp2f(m_used - m_new) : 1.f;
#pragma unroll 1
          for (int q = 0; q < 256 / 16; ++q) {
            uint32_t r[16];
            tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * a);
            tmem_st16(tmem + lane_base + kOCol + 16 * q, r);
          }
          tmem_st_wait();
          l_sum *= a;
        }
        m_used = m_new;
      }
      uint32_t pk[kRows / 2];
      float lt = 0.f;
#pragma unroll
      for (int j = 0; j < kRows; j += 2) {
        const float p0 = m_used == -INFINITY ? 0.f : exp2f(s[j] - m_used);
        const float p1 = m_used == -INFINITY ? 0.f : exp2f(s[j + 1] - m_used);
        lt += p0 + p1;
        pk[j >> 1] = pack_bf16x2(p0, p1);
      }
      l_sum += lt;
      // 5. P into TMEM once P.V(tl - 2) has read the buffer
      if (tl >= 2 && !dead) dead = !SMLA_WAIT(kBarPDone + kb, ((tl >> 1) + 1) & 1);
      tc_fence_after();
      {
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          lo[j] = pk[j];
          hi[j] = pk[16 + j];
        }
        tmem_st16(tmem + lane_base + kPCol + 32 * kb, lo);
        tmem_st16(tmem + lane_base + kPCol + 32 * kb + 16, hi);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bars[kBarPFull + kb]);
      ++n_seg_tiles;
      // 6. epilogue at the end of a segment
      if (ti.seg_end) {
        if (!dead) dead = !SMLA_WAIT(kBarPDone + kb, (tl >> 1) & 1);
        tc_fence_after();
        const bool full_unit = n_seg_tiles == p.nt;  // the whole token ran in this pair
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const float lse_v = l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
        const int64_t slot = (int64_t)pair + ti.u;
        for (int q = 0; q < 256 / 16; ++q) {
          uint32_t r[16];
          tmem_ld16_sync(tmem + lane_base + kOCol + 16 * q, r);
          if (dead) continue;
          if (full_unit) {
            uint4 o[2];
            uint32_t* ow = reinterpret_cast<uint32_t*>(o);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ow[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * inv, __uint_as_float(r[2 * j + 1]) * inv);
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)ti.u * kHeads + h) * kDv + 256 * c + 16 * q);
            dst[0] = o[0];
            dst[1] = o[1];
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + (slot * kHeads + h) * kDv + 256 * c + 16 * q);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                                   __uint_as_float(r[4 * j + 2]) * inv, __uint_as_float(r[4 * j + 3]) * inv);
          }
        }
        if (!dead && c == 0) {
          if (full_unit)
            p.lse[(int64_t)ti.u * kHeads + h] = lse_v;
          else
            p.part_lse[slot * kHeads + h] = lse_v;
        }
        tc_fence_before();
        mbar_arrive(&bars[kBarOFree]);
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

// kv [N, 576] bf16 and q [T * 128, 576] bf16, both as bytes: the kv map
// gathers one 128-byte panel of single rows, the q map loads one panel of
// 128 consecutive head rows; both with the 128-byte swizzle.
cudaError_t make_maps(const void* kv, int64_t N, const void* q, int T, CUtensorMap* kv_map, CUtensorMap* q_map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t gstride[1] = {(cuuint64_t)kRowBytesBf16};
  const cuuint32_t es[2] = {1, 1};
  const cuuint64_t kv_dim[2] = {(cuuint64_t)kRowBytesBf16, (cuuint64_t)N};
  const cuuint32_t kv_box[2] = {128, 1};
  CUresult r = enc(kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(kv), kv_dim, gstride, kv_box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const cuuint64_t q_dim[2] = {(cuuint64_t)kRowBytesBf16, (cuuint64_t)T * kHeads};
  const cuuint32_t q_box[2] = {128, kHeads};
  r = enc(q_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(q), q_dim, gstride, q_box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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
  CUtensorMap kv_map, q_map;
  cudaError_t e = make_maps(a.kv, a.NB, a.q, a.T, &kv_map, &q_map);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(sparse_mla_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  sparse_mla_wide_kernel<<<2 * plan.G, kThreads, kSmemAlloc, stream>>>(p, kv_map, q_map);
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  combine_kernel<kHeads><<<(unsigned)(plan.units * combine_split<kHeads>()), combine_threads<kHeads>(), 0, stream>>>(
      p.part_o, p.part_lse, p.out, p.lse, kHeads, 1, p.nt, p.total, p.G);
  return cudaGetLastError();
}

}  // namespace smla
