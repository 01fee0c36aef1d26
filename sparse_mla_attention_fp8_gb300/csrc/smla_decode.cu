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
// Design: the tensor cores read the cache codes as stored, with no
// dequantization pass, 128 top-k rows per tile (M = 128 in every MMA).
//  * Transport: the loader warps copy the rows with 16-byte cp.async (LSU
//    path, L2 only): one instruction moves 128 codes of 4 rows into a code
//    panel with the 128-byte swizzle, nine move the scales and RoPE values of
//    32 rows.  A buffer's RoPE panel and scales are refilled once the softmax
//    has read its previous tile's, and each code panel once the P.V of that
//    tile has read it.  The tensor cores read the tile after each loader has
//    waited for its own copies and made them visible to the async proxy.
//    Invalid rows are zero-filled.  Two operand tiles (4 code panels of 128
//    rows x 128 bytes, a RoPE panel and the 128 rows' scales: 82 KB each).
//  * Q is split once per (token, 16-head group) into two e4m3 terms,
//    q * 2^s_hg = hi + lo (s_hg a power of two per head and 128-column scale
//    group g putting the group's max |q| near 448), exact for all but
//    components far below their group's largest; hi and lo are the two halves
//    of an N = 32 operand.  QK^T for scale group g is kind::f8f6f4
//    S_g = E_g [Q_hi Q_lo]^T (M = 128 rows, N = 32, K = 128 codes in 4 steps),
//    the RoPE part a bf16 product (N = 16); the softmax combines
//    s = sum_g scale_g 2^-s_hg (S_g,hi + S_g,lo) + S_rope in fp32.
//  * P.V for value chunk q (= scale group q) is kind::f8f6f4
//    O_q^T += E_q^T P'_q with the same code panel read MN-major (M = 128 value
//    columns, N = 32, K = 32 rows per step) and P'_q = 2^7 p * scale_q / R_q
//    split into e4m3 hi + lo (R_q a running power-of-two bound of the group's
//    scales).  The running max of a head is refreshed (to 2^0.75 above the
//    tile's maximum) only when a tile's maximum exceeds it by more than
//    2^1.75, so p <= 2^1.75 and P' < 430 stays at the top of the e4m3 range
//    (max 448), where hi + lo carries 8 significant bits.  O is rescaled in
//    tensor memory when R_q or a running max changes.
//  * 36 MMAs per 128 rows: 16 QK^T, 4 RoPE, 16 P.V.
//  * Softmax: thread = tile row (its TMEM lane), 8 heads; tile maxima by
//    warp reductions and a named barrier per half of the heads.
//  * Warp roles: softmax / epilogue (8 warps: one per TMEM lane quarter and
//    half of the 16 heads), tensor-core issuer (1 thread), index translation
//    (1 warp), loaders (4 warps), Q preparation (2 warps).
#include <cstdint>
#include <algorithm>
#include <mutex>
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

// Optional per-tile timeline for performance work: built with SMLA_TRACE
// defined (the separate traced library that trace.py builds), roles record
// %globaltimer at their hand-off points into g_smla_trace_fp8, set by the host
// through smla_trace_set_fp8.  Compiled out otherwise.
#ifdef SMLA_TRACE
__device__ unsigned long long* g_smla_trace_fp8 = nullptr;
constexpr int kTraceTiles = 16, kTraceEvents = 23;
#define SMLA_TRACE_SET(tl, ev)                                                                                  \
  do {                                                                                                          \
    if (trace_buf && (tl) < kTraceTiles)                                                                        \
      trace_buf[((size_t)blockIdx.x * kTraceTiles + (tl)) * kTraceEvents + (ev)] = globaltimer_ns();            \
  } while (0)
#else
#define SMLA_TRACE_SET(tl, ev) ((void)0)
#endif
// events: index translated, loader 0 past its free-buffer wait, loader 0
// copies issued, loader 0 copies landed, tile full (seen by the QK^T issuer),
// QK^T issued, softmax start (S ready), softmax past the tile-max barrier, P'
// written (warp 0), P.V issued, epilogue done, Q of a segment ready (at the
// segment's first tile), epilogue past the last P.V, cluster merge: before
// the wait for the other CTA, after it; the CTA's first instruction and its
// exit (tile 0's slots); cluster merge steps: sums and LSEs done, readiness
// signalled, the others' readiness seen, values sent, output written; set-up
// done (barriers initialised, tensor memory allocated, cluster synchronised)
enum { kEvIdx = 0, kEvBufFree, kEvIssued, kEvLanded, kEvOpFull, kEvQk, kEvSoftStart, kEvSoftBar, kEvPWritten, kEvPv,
       kEvEpi, kEvQReady, kEvEpiStart, kEvMergeWait, kEvMergeGo, kEvEnter, kEvExit, kEvEpiLse, kEvEpiSignal,
       kEvEpiReady, kEvEpiSent, kEvEpiWritten, kEvSetup };

constexpr int HG = 16;                 // heads per CTA work unit
constexpr int kRows = 128;             // top-k rows per tile
constexpr int kLoaders = 4;            // loader lw copies rows 32 lw .. 32 lw + 31 of every tile
constexpr int kOpBufs = 2;             // operand tiles
constexpr float kMaxSlack = 1.75f;     // log2 growth of a head's max tolerated before rescaling O (p <= 2^1.75)
constexpr float kMaxOvershoot = 0.75f; // a refreshed running max is set this far above the tile max
constexpr float kPScale = 128.0f;      // P' = kPScale * p * scale / R  <=  128 * 2^1.75 < 430 (e4m3 max 448)
constexpr float kPScaleInv = 1.0f / 128.0f;

// ---- shared memory layout (offsets from a 1024-byte aligned base)
constexpr int kPanel = kRows * 128;                   // 16 KB: 128 rows x 128 bytes, 128-byte swizzle
constexpr int kOpRope = 4 * kPanel;                   // RoPE panel after the 4 code panels
constexpr int kOpScale = 5 * kPanel;                  // scales: 128 rows x 16 bytes
constexpr int kOpBuf = 5 * kPanel + kRows * 16;       // 83968
constexpr int kQPanel = 32 * 128;                     // 32 operand rows (hi, lo) x 128 codes
constexpr int kQRope = 4 * kQPanel;                   // 16 rows x 64 bf16
constexpr int kQBuf = 4 * kQPanel + HG * 128;         // 18432
constexpr int kQBufs = 2;                             // Q blocks: the next segment's is prepared ahead
constexpr int kPGroup = kRows * 32;                   // P'_q: 128 rows x 32 codes
constexpr int kPBuf = 4 * kPGroup;                    // 16384
constexpr int kPBufs = 1;                             // P' buffers
constexpr int kOffOp = 0;
constexpr int kOffQ = kOffOp + kOpBufs * kOpBuf;
constexpr int kOffP = kOffQ + kQBufs * kQBuf;
constexpr int kOffSlots = kOffP + kPBufs * kPBuf;                   // int32 [4][128]
constexpr int kOffValid = kOffSlots + 4 * kRows * 4;                // uint8 [2][128]
constexpr int kOffPre = kOffValid + kOpBufs * kRows;                // float [4 segments][4 groups][16 heads]
constexpr int kOffRedMax = kOffPre + 4 * 4 * HG * 4;                // float [2 tiles][2 halves][4 quarters][8 heads]
constexpr int kOffRedSc = kOffRedMax + 2 * 2 * 4 * 8 * 4;           // uint32 [2 tiles][2 halves][4 quarters][4 groups]
constexpr int kOffRedSum = kOffRedSc + 2 * 2 * 4 * 4 * 4;           // float [2 halves][4 quarters][8 heads]
constexpr int kOffBar = kOffRedSum + 2 * 4 * 8 * 4;
enum {
  // kBarOpEmpty + 4 ob + q: code panel q of operand tile ob has been read by its P.V
  kBarOpFull = 0, kBarOpEmpty = kBarOpFull + kOpBufs, kBarSFull = kBarOpEmpty + 4 * kOpBufs, kBarSFree = kBarSFull + 2,
  kBarPFull = kBarSFree + 2, kBarPvDone = kBarPFull + kPBufs, kBarIdxFull = kBarPvDone + kPBufs,
  kBarIdxEmpty = kBarIdxFull + 4, kBarQFull = kBarIdxEmpty + 4, kBarQEmpty = kBarQFull + kQBufs,
  kBarOFree = kBarQEmpty + kQBufs, kBarDrain = kBarOFree + 1, kBarDrainPv = kBarDrain + 1,
  kBarReady = kBarDrainPv + 1,  // cluster merge: every other CTA's receive buffer is free (arrived remotely)
  kBarRecv = kBarReady + 1,     // cluster merge: the other parts' values of this CTA's chunks have arrived
  kNumBars = kBarRecv + 1
};
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
// cluster merge: CTA c of a cluster of S writes the value chunks q (128
// columns each) with q % S == c; it receives every other CTA's normalized
// values of those chunks (128 columns x 16 heads fp32 per chunk) and its 16
// LSEs in its operand tiles (free by then)
constexpr int kMaxCluster = 4;
constexpr int kChunkBytes = kRows * HG * 4;  // 8 KB: one value chunk of one part, [column][head]
// two-part clusters: a CTA sends its raw values of the other's two chunks and
// its heads' running maxima and sums (fp32), staged after its own receive buffer
constexpr int kTwoPartBytes = 2 * kChunkBytes + 2 * HG * 4;
constexpr int kSendOff = 3 * kChunkBytes;
static_assert(kSendOff >= kTwoPartBytes && kSendOff + kTwoPartBytes <= kOpBufs * kOpBuf && kTwoPartBytes % 16 == 0,
              "two-part send staging");
static_assert((kMaxCluster - 1) * (2 * kChunkBytes + HG * 4) <= kOpBufs * kOpBuf, "cluster receive buffer");
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kOpBuf % 1024 == 0, "operand alignment");
static_assert(kOffBar % 8 == 0, "barriers 8-byte aligned");
static_assert(kOffPre % 16 == 0 && kOffRedMax % 16 == 0 && kOffRedSc % 16 == 0 && kOffRedSum % 16 == 0, "float4");
static_assert(kSmemAlloc <= 232448, "shared memory budget");
static_assert(kOpBufs == 2, "operand tile tl uses S buffer tl % 2 as well");

// ---- tensor memory columns
constexpr int kSCols = 4 * 32 + HG;   // per S buffer: 4 groups x (hi, lo) x 16 heads + RoPE
constexpr int kOCol = 2 * kSCols;     // O^T: 4 chunks x (hi, lo) x 16 heads
constexpr int kTmemCols = 512;
static_assert(kOCol + 4 * 32 <= kTmemCols, "tensor memory budget");

// ---- warp roles (16 warps; 128 registers per thread).  Warp w runs on
// sub-partition w % 4: each sub-partition carries two softmax warps (one per
// head half), a loader and one more role.  Each tensor-core issuer blocks on
// its own barriers, so no warp spins.
constexpr int kSoftWarps = 8, kLoadWarp0 = 8, kMmaWarp = 12, kPvWarp = 13, kIndexWarp = 14, kQWarp = 15;
constexpr int kNumWarps = 16;
constexpr int kThreads = 32 * kNumWarps;
static_assert(kLoadWarp0 + kLoaders == kMmaWarp && kQWarp + 1 == kNumWarps, "warp roles");

__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

struct Params {
  const __nv_bfloat16* q;
  const uint8_t* cache;
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
  int cluster;  // > 1: the parts of a unit are the CTAs of one cluster, merged by its first CTA
};

struct TileInfo {
  int u, kt, t, hg;
  bool seg_start, seg_end;
};

// Top-k tile index of tile x within its unit (x mod nt).
__device__ __forceinline__ int tile_kt(const Params& p, int64_t x) {
  return (int)(x - udiv_fast(x, p.nt) * p.nt);
}

__device__ __forceinline__ TileInfo tile_info(const Params& p, int64_t x, int64_t xbeg, int64_t xend) {
  TileInfo ti;
  ti.u = (int)udiv_fast(x, p.nt);
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

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}


__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
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

// Two floats -> e4m3 hi and lo pairs (low byte from x0), x ~ hi + lo; the
// split runs in f16x2 (11 significant bits, more than the 8 that hi + lo keep).
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

__device__ __forceinline__ float pow2_ceil(float x) {  // smallest power of two >= x (x > 0)
  const uint32_t u = __float_as_uint(x);
  const uint32_t e = u & 0x7F800000u;
  return __uint_as_float((u & 0x007FFFFFu) ? e + 0x00800000u : e);
}

// 1 / x for a power of two x in the normal range (exact).
__device__ __forceinline__ float rcp_pow2(float x) { return __uint_as_float(0x7F000000u - __float_as_uint(x)); }

// Warp-wide maxima: floats through an order-preserving map to signed
// integers (negative floats reversed), non-negative floats as their bits.
__device__ __forceinline__ float warp_max_f32(float x) {
  int k = __float_as_int(x);
  k = k >= 0 ? k : k ^ 0x7FFFFFFF;
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(k));
  return __int_as_float(r >= 0 ? r : r ^ 0x7FFFFFFF);
}
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t x) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(x));
  return r;
}

// 16-byte cp.async global -> shared through L2 (src_bytes = 0 writes zeros).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Offset of 16-byte column `ch` (0..7) of row r in a 128-byte-swizzled panel.
__device__ __forceinline__ uint32_t sw128(int r, int ch) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4));
}

// Q of head h of one (token, 16-head group) into a Q buffer, by NSUB threads
// per (head, scale group `part`) on consecutive lanes: thread `sub` converts
// columns [128 part + W sub, + W), W = 128 / NSUB.  q * 2^s = hi + lo in e4m3,
// s chosen so that the largest |q * 2^s| over the group's 128 columns is at
// most 448; hi goes to operand row h, lo to row 16 + h; the RoPE chunks are
// copied as they are; pre[part * 16 + h] = 2^-s.
template <int NSUB>
__device__ __forceinline__ void prep_q(const __nv_bfloat16* __restrict__ qrow, int h, int part, int sub, uint32_t qbuf,
                                       float* pre) {
  constexpr int W = 128 / NSUB, NV = W / 8;
  const uint4* src = reinterpret_cast<const uint4*>(qrow);
  uint4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = __ldg(src + (128 * part + W * sub) / 8 + i);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k)
      amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 1; o < NSUB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, o));
  int sh = 0;
  if (amax > 0.f) {
    int e;
    frexpf(448.f / amax, &e);  // 448 / amax = m * 2^e, m in [0.5, 1)
    sh = e - 1;
  }
  const float pre_s = ldexpf(1.f, sh);
  const uint32_t qpanel = qbuf + part * kQPanel;
#pragma unroll
  for (int ch = 0; ch < W / 16; ++ch) {  // 16 codes per chunk = two uint4 of bf16
    uint32_t hi[4], lo[4];
    const uint32_t w8[8] = {v[2 * ch].x,     v[2 * ch].y,     v[2 * ch].z,     v[2 * ch].w,
                            v[2 * ch + 1].x, v[2 * ch + 1].y, v[2 * ch + 1].z, v[2 * ch + 1].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t h0, l0, h1, l1;
      split2(__uint_as_float(w8[2 * k] << 16) * pre_s, __uint_as_float(w8[2 * k] & 0xFFFF0000u) * pre_s, h0, l0);
      split2(__uint_as_float(w8[2 * k + 1] << 16) * pre_s, __uint_as_float(w8[2 * k + 1] & 0xFFFF0000u) * pre_s, h1, l1);
      hi[k] = h0 | (h1 << 16);
      lo[k] = l0 | (l1 << 16);
    }
    const int c16 = (W * sub) / 16 + ch;
    sts128(qpanel + sw128_chunk(32, h, c16), make_uint4(hi[0], hi[1], hi[2], hi[3]));
    sts128(qpanel + sw128_chunk(32, 16 + h, c16), make_uint4(lo[0], lo[1], lo[2], lo[3]));
  }
  for (int rc = part * NSUB + sub; rc < 8; rc += 4 * NSUB)
    sts128(qbuf + kQRope + sw128_chunk(HG, h, rc), __ldg(src + 64 + rc));
  if (sub == 0) pre[part * HG + h] = ldexpf(1.f, -sh);
}

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_decode_fp8_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  grid_launch_dependents();  // the combine may be launched behind this grid right away
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* slots_ring = reinterpret_cast<int32_t*>(smem + kOffSlots);
  uint8_t* valid = smem + kOffValid;
  float* pre_ring = reinterpret_cast<float*>(smem + kOffPre);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#ifdef SMLA_TRACE
  unsigned long long* __restrict__ const trace_buf = g_smla_trace_fp8;
  if (tid == 0) SMLA_TRACE_SET(0, kEvEnter);
#endif
  const int64_t xbeg = tile_begin(blockIdx.x, p.total, p.G);
  const int64_t xend = tile_begin(blockIdx.x + 1, p.total, p.G);
  const int n_local = (int)(xend - xbeg);
  // the index warp's loads for the first tile go out before the set-up below,
  // so their memory latency overlaps it
  int32_t idx0[4] = {-1, -1, -1, -1}, req0 = 0;
  if (warp == kIndexWarp && n_local > 0) {
    const TileInfo t0 = tile_info(p, xbeg, xbeg, xend);
    req0 = __ldg(p.req_id + t0.t);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int k = t0.kt * kRows + lane + 32 * i;
      idx0[i] = k < p.K ? __ldg(p.indices + (int64_t)t0.t * p.K + k) : -1;
    }
  }

  if (tid == 0) {
    for (int i = 0; i < kOpBufs; ++i) {
      mbar_init(&bars[kBarOpFull + i], kLoaders);  // one arrival per loader once its copies are visible
      for (int q = 0; q < 4; ++q) mbar_init(&bars[kBarOpEmpty + 4 * i + q], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarSFree + i], kSoftWarps);
    }
    for (int i = 0; i < kPBufs; ++i) {
      mbar_init(&bars[kBarPFull + i], kSoftWarps);
      mbar_init(&bars[kBarPvDone + i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarIdxFull + i], 32);
      mbar_init(&bars[kBarIdxEmpty + i], kLoaders);
    }
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(&bars[kBarQFull + i], 1);
      mbar_init(&bars[kBarQEmpty + i], 1);
    }
    mbar_init(&bars[kBarOFree], kSoftWarps);
    mbar_init(&bars[kBarDrain], 1);
    mbar_init(&bars[kBarDrainPv], 1);
    mbar_init(&bars[kBarReady], p.cluster > 1 ? p.cluster - 1 : 1);
    mbar_init(&bars[kBarRecv], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if (p.cluster > 1)
    cluster_sync_relaxed();  // every CTA's barriers (fenced above) are initialised before another CTA uses them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) SMLA_TRACE_SET(0, kEvSetup);
  // Launched as a programmatic dependent (of the cache store, typically): the
  // index translation and the Q split read only this call's inputs and write
  // only shared memory, so they start at once; every other role reads the
  // cache or writes global memory, and first waits for the preceding grid.
  if (warp >= kSoftWarps && warp != kIndexWarp && warp != kQWarp) grid_dependency_wait();

#define SMLA_WAIT(bar_idx, parity) mbar_wait(&bars[(bar_idx)], (parity), abort_flag, p.status, kDevWaitTimeout)

  if (warp == kIndexWarp) {
    // ------------------------------------------------------------ index translation
    // The next tile's indices are loaded before this tile's block-table reads,
    // so each tile costs about one memory round trip.
    int32_t cur[4] = {idx0[0], idx0[1], idx0[2], idx0[3]}, nxt[4], req_cur = req0, req_nxt = 0;
    auto load_idx = [&](int tl, int32_t (&v)[4], int32_t& rq) {
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      rq = __ldg(p.req_id + ti.t);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = ti.kt * kRows + lane + 32 * i;
        v[i] = k < p.K ? __ldg(p.indices + (int64_t)ti.t * p.K + k) : -1;
      }
    };
    for (int tl = 0; tl < n_local; ++tl) {
      if (tl + 1 < n_local) load_idx(tl + 1, nxt, req_nxt);
      const int b4 = tl & 3;
      if (tl >= 4 && !SMLA_WAIT(kBarIdxEmpty + b4, ((tl >> 2) + 1) & 1)) break;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        slots_ring[b4 * kRows + lane + 32 * i] = translate_slot(cur[i], req_cur, p.block_table, p.R, p.MB, p.NB);
      mbar_arrive(&bars[kBarIdxFull + b4]);
      if (lane == 0) SMLA_TRACE_SET(tl, kEvIdx);
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
      req_cur = req_nxt;
    }
  } else if (warp >= kLoadWarp0 && warp < kLoadWarp0 + kLoaders) {
    // ------------------------------------------------------------ loaders
    // Loader lw copies rows 32 lw .. 32 lw + 31 of every tile with 16-byte
    // cp.async: nine instructions for the 32 rows' scales and RoPE values
    // (chunk 0 of a row's 144 bytes from byte 512 is its scales, chunks 1..8
    // its RoPE values), as soon as the softmax has read the buffer's previous
    // tile; then, per code panel q as soon as that tile's P.V has read it,
    // eight instructions for the rows' codes 128 q .. 128 q + 127 (128-byte
    // swizzle).  Invalid rows are zero-filled.  Its arrival on the
    // tile's full barrier follows its own copies' completion and a proxy
    // fence (the tensor cores read the tile through the async proxy), and its
    // writes of the rows' valid flags.
    const int lw = warp - kLoadWarp0;
    const int rw = 32 * lw;  // first tile row of this loader
    // Codes: instruction i of panel q moves rows 4 i .. 4 i + 3 (of this
    // loader's 32) x 128 codes; lane l copies 16-byte column l % 8 of row
    // 4 i + l / 8, to column (l % 8) ^ (row % 8) of the panel's row.  The
    // row's place in its 8-row group is 4 (i % 2) + l / 8: one offset per
    // parity of i.
    uint32_t code_off[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int rr = 4 * e + (lane >> 3);
      code_off[e] = (uint32_t)((rw >> 3) * 1024 + rr * 128 + (((lane & 7) ^ rr) << 4));
    }
    const uint8_t* cache_lane = p.cache + 16 * (lane & 7);
    for (int tl = 0; tl < n_local; ++tl) {
      const int b4 = tl & 3, ob = tl % kOpBufs, use = tl / kOpBufs;
      if (!SMLA_WAIT(kBarIdxFull + b4, (tl >> 2) & 1)) break;
      const int32_t slot = slots_ring[b4 * kRows + rw + lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarIdxEmpty + b4]);  // this loader's slots read
      // The tile two before in this buffer has been through QK^T and the
      // softmax has read its rows' flags and scales (its S buffer is free
      // again): the RoPE panel, the scales and the flags can take this tile's
      // while the codes are still being read by its P.V.
      if (use >= 1 && !SMLA_WAIT(kBarSFree + (tl & 1), ((tl - 2) >> 1) & 1)) break;
      valid[ob * kRows + rw + lane] = slot >= 0 ? 1 : 0;
      const uint32_t op = smem_u32(smem + kOffOp + ob * kOpBuf);
#pragma unroll
      for (int it = 0; it < 9; ++it) {
        const int idx = 32 * it + lane;
        const int i = idx / 9, k = idx - 9 * i;
        const int32_t s = __shfl_sync(kFullMask, slot, i);
        const int r = rw + i;
        const uint8_t* src = p.cache + (int64_t)(s >= 0 ? s : 0) * kRowBytes + kScaleOff + 16 * k;
        const uint32_t dst = k == 0 ? op + kOpScale + 16 * r : op + kOpRope + sw128(r, k - 1);
        cp_async_16(dst, src, s >= 0 ? 16u : 0u);
      }
      // code panel q is free once that tile's P.V has read it (its chunk q)
      bool gone = false;
#pragma unroll 1
      for (int q = 0; q < 4 && !gone; ++q) {
        if (use >= 1 && !SMLA_WAIT(kBarOpEmpty + 4 * ob + q, (use + 1) & 1)) gone = true;
        if (lane == 0 && lw == 0 && q == 0) SMLA_TRACE_SET(tl, kEvBufFree);
        if (gone) break;
        const uint32_t panel = op + q * kPanel;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int32_t s = __shfl_sync(kFullMask, slot, 4 * i + (lane >> 3));
          const uint8_t* src = cache_lane + (size_t)(uint32_t)max(s, 0) * kRowBytes + 128 * q;
          cp_async_16(panel + code_off[i & 1] + (uint32_t)((i >> 1) * 1024), src, s >= 0 ? 16u : 0u);
        }
      }
      if (gone) break;
      if (lane == 0 && lw == 0) SMLA_TRACE_SET(tl, kEvIssued);
      asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
      if (lane == 0 && lw == 0) SMLA_TRACE_SET(tl, kEvLanded);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarOpFull + ob]);
    }
  } else if (warp == kQWarp) {
    // ------------------------------------------------------------ Q preparation
    // Every segment after the first (the softmax warps prepare the first one
    // at start-up): four passes of 4 heads, lane 8 j + 2 part + sub handling
    // half `sub` of head j (+ 4 pass) and scale group `part`.  Two Q buffers: segment s uses buffer
    // s % 2, so the next segment's Q is ready before the current one ends.
    int tl = 0, seg = 0;
    while (true) {
      // the next segment starts at the next tile with top-k tile index 0
      do {
        ++tl;
      } while (tl < n_local && tile_info(p, xbeg + tl, xbeg, xend).kt != 0);
      if (tl >= n_local) break;
      ++seg;
      const int qb = seg % kQBufs;
      if (seg >= kQBufs && !SMLA_WAIT(kBarQEmpty + qb, ((seg / kQBufs) - 1) & 1)) break;
      const TileInfo ti = tile_info(p, xbeg + tl, xbeg, xend);
      const uint32_t qbuf = smem_u32(smem + kOffQ + qb * kQBuf);
#pragma unroll 1
      for (int pass = 0; pass < 4; ++pass) {
        const int h = (lane >> 3) + 4 * pass;
        prep_q<2>(p.q + ((int64_t)ti.t * p.H + ti.hg * HG + h) * kDqk, h, (lane >> 1) & 3, lane & 1, qbuf,
                  pre_ring + (seg & 3) * 4 * HG);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarQFull + qb]);
      if (lane == 0) SMLA_TRACE_SET(tl, kEvQReady);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ QK^T issuer
    // One thread: QK^T of each tile once its rows, the segment's Q and a free
    // S buffer (the softmax has read the tile two before out of it) are there.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_qk8 = idesc_e4m3(128, 32, 0, 0);
      constexpr uint32_t id_qkr = make_idesc_bf16(128, HG, 0, 0);
      // Shared-memory descriptors are built once; an operand at a byte offset
      // o from a base is that descriptor + o / 16 (the start-address field holds
      // bits 4..17 of the address, and no offset here carries out of it).
      const uint64_t dK0 = make_sdesc(smem_u32(smem + kOffOp), 16, 1024, kLayoutSw128);
      const uint64_t dQ = make_sdesc(smem_u32(smem + kOffQ), 16, 1024, kLayoutSw128);
      int seg = 0, kt = tile_kt(p, xbeg), issued = 0;
      for (int tl = 0; tl < n_local; ++tl) {
        const int sbuf = tl & 1, ob = tl % kOpBufs;
        const bool seg_start = tl == 0 || kt == 0;
        const bool seg_end = tl == n_local - 1 || kt == p.nt - 1;
        if (tl >= 2 && !SMLA_WAIT(kBarSFree + sbuf, ((tl - 2) >> 1) & 1)) break;
        const int qb = seg % kQBufs;
        if (seg_start && !SMLA_WAIT(kBarQFull + qb, (seg / kQBufs) & 1)) break;
        if (!SMLA_WAIT(kBarOpFull + ob, (tl / kOpBufs) & 1)) break;
        SMLA_TRACE_SET(tl, kEvOpFull);
        tc_fence_after();
        const uint64_t dk = dK0 + (uint64_t)((ob * kOpBuf) >> 4);
        const uint64_t dq = dQ + (uint64_t)((qb * kQBuf) >> 4);
        const uint32_t sb = tmem + sbuf * kSCols;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_f8(sb + 32 * g, dk + ((g * kPanel + 32 * k) >> 4), dq + ((g * kQPanel + 32 * k) >> 4), id_qk8,
                   k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(sb + 128, dk + ((kOpRope + 32 * k) >> 4), dq + ((kQRope + 32 * k) >> 4), id_qkr, k > 0 ? 1u : 0u);
        mma_commit(&bars[kBarSFull + sbuf]);
        if (seg_end) {
          mma_commit(&bars[kBarQEmpty + qb]);
          ++seg;
        }
        SMLA_TRACE_SET(tl, kEvQk);
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
    // One thread: O^T += E^T P' of each tile once its P' is written (and,
    // first in a segment, the previous segment's epilogue has read O).  The
    // completion of its value chunk q frees code panel q of the operand tile
    // (QK^T of the tile completed before its P' could be written); that of
    // the whole tile frees the P' buffer.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t id_pv = idesc_e4m3(128, 32, 1, 1);
      const uint64_t dV0 = make_sdesc(smem_u32(smem + kOffOp), kPanel, 1024, kLayoutSw128);
      const uint64_t dP0 = make_sdesc(smem_u32(smem + kOffP), 256, 128, kLayoutNone);
      int seg_o = 0, kt = tile_kt(p, xbeg), issued = 0;
      for (int tl = 0; tl < n_local; ++tl) {
        const int ob = tl % kOpBufs, pb = tl % kPBufs;
        const bool seg_start = tl == 0 || kt == 0;
        if (seg_start && seg_o > 0 && !SMLA_WAIT(kBarOFree, (seg_o - 1) & 1)) break;
        if (!SMLA_WAIT(kBarPFull + pb, (tl / kPBufs) & 1)) break;
        if (seg_start) ++seg_o;
        tc_fence_after();
        const uint64_t dv = dV0 + (uint64_t)((ob * kOpBuf) >> 4), dp = dP0 + (uint64_t)((pb * kPBuf) >> 4);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            // A = codes^T (value column c x row j), MN-major; B = P'_q (row j x 32), MN-major
            mma_f8(tmem + kOCol + 32 * q, dv + ((q * kPanel + 4096 * k) >> 4), dp + ((q * kPGroup + 1024 * k) >> 4),
                   id_pv, (seg_start && k == 0) ? 0u : 1u);
          mma_commit(&bars[kBarOpEmpty + 4 * ob + q]);  // code panel q read (QK^T of the tile completed earlier)
        }
        mma_commit(&bars[kBarPvDone + pb]);
        SMLA_TRACE_SET(tl, kEvPv);
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
    // ------------------------------------------------------------ softmax / epilogue (warps 0..7)
    // QK^T with M = 128 leaves tile row r in TMEM lane r.  Warp w reads lane
    // quarter qd = w % 4 (rows 32 qd .. 32 qd + 31, one per thread) and the
    // columns of heads 8 hh .. 8 hh + 7, hh = w / 4.  Every thread of a half
    // keeps the running maxima of its 8 heads (the same in all of them) and
    // its own row's share of the running sums.  The two halves share nothing
    // but the barriers on S, P' and O: each decides its own rescales and
    // rescales its own columns of O.  For the P.V output (M = 128) thread
    // lane of warp w owns value column 32 qd + lane of each chunk, for the
    // columns of its half.
    const int w = warp, qd = w & 3, hh = w >> 2;
    const int r = 32 * qd + lane;
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    const uint32_t p0 = smem_u32(smem + kOffP);
    const int bar_id = 1 + hh;  // named barrier of the half (4 warps)
    float* red_max = reinterpret_cast<float*>(smem + kOffRedMax);
    uint32_t* red_sc = reinterpret_cast<uint32_t*>(smem + kOffRedSc);
    float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
    float m[8], l[8], Rq[4];
    int seg = -1, seg_first_kt = 0, n_seg_tiles = 0;
    bool dead = false;
    // waits of this role keep `dead` warp-uniform: the tensor-memory accesses
    // and reductions it guards are warp-collective
    auto wait_s = [&](int bar_idx, uint32_t parity) {
      if (!dead) dead = !SMLA_WAIT(bar_idx, parity);
      dead = __any_sync(kFullMask, dead);
    };
    TileInfo ti = tile_info(p, xbeg, xbeg, xend);
    if (n_local > 0) {
      // Q of the first segment (buffer 0), 4 threads per (head, scale group):
      // it reads only q, so it runs before the wait for the preceding grid
      prep_q<4>(p.q + ((int64_t)ti.t * p.H + ti.hg * HG + (tid >> 4)) * kDqk, tid >> 4, (tid >> 2) & 3, tid & 3,
                smem_u32(smem + kOffQ), pre_ring);
      fence_proxy_async_smem();
      named_bar_sync(3, 32 * kSoftWarps);
      if (tid == 0) mbar_arrive(&bars[kBarQFull]);
      if (tid == 0) SMLA_TRACE_SET(0, kEvQReady);
    }
    grid_dependency_wait();  // the epilogue writes global memory
    for (int tl = 0; tl < n_local; ++tl) {
      if (tl > 0) {  // advance the tile position without divisions
        ti.seg_start = ++ti.kt == p.nt;
        if (ti.seg_start) {
          ti.kt = 0;
          ++ti.u;
          if (++ti.hg == p.n_hg) {
            ti.hg = 0;
            ++ti.t;
          }
        }
        ti.seg_end = tl == n_local - 1 || ti.kt == p.nt - 1;
      }
      const int ob = tl % kOpBufs, sbuf = tl & 1, pb = tl % kPBufs, puse = tl / kPBufs;
      if (ti.seg_start) {
        ++seg;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          m[h] = -INFINITY;
          l[h] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) Rq[g] = 0.f;
        seg_first_kt = ti.kt;
        n_seg_tiles = 0;
      }
      wait_s(kBarOpFull + ob, (tl / kOpBufs) & 1);  // row flags and scales
      wait_s(kBarSFull + sbuf, (tl >> 1) & 1);
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftStart);
      tc_fence_after();
      const bool ok = !dead && valid[ob * kRows + r] != 0;
      const float4 s4 = ok ? *reinterpret_cast<const float4*>(smem + kOffOp + ob * kOpBuf + kOpScale + 16 * r)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      const float sc[4] = {s4.x, s4.y, s4.z, s4.w};
      // logits (log2 units): sum_g scale_g 2^-s_hg (S_g,hi + S_g,lo) + S_rope
      float sl[8];
      {
        const uint32_t sa = tmem + lane_base + sbuf * kSCols + 8 * hh;
        const float* pre = pre_ring + (seg & 3) * 4 * HG + 8 * hh;
        float acc[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) acc[h] = 0.f;
        if (!dead) {
#pragma unroll
          for (int gp = 0; gp < 2; ++gp) {  // scale groups 2 gp, 2 gp + 1 (and the RoPE part with the second pair)
            uint32_t hi[2][8], lo[2][8], rp[8];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              tmem_ld8(sa + 32 * (2 * gp + e), hi[e]);
              tmem_ld8(sa + 32 * (2 * gp + e) + 16, lo[e]);
            }
            if (gp == 1) tmem_ld8(sa + 128, rp);
            tmem_ld_wait();
            if (gp == 1) {
              // S of this tile is in registers: its buffer may take QK^T of tile tl + 2
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&bars[kBarSFree + sbuf]);
              reg_fence8(rp);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              reg_fence8(hi[e]);
              reg_fence8(lo[e]);
              const int g = 2 * gp + e;
              const float4 i0 = *reinterpret_cast<const float4*>(pre + g * HG);
              const float4 i1 = *reinterpret_cast<const float4*>(pre + g * HG + 4);
              const float ip[8] = {i0.x, i0.y, i0.z, i0.w, i1.x, i1.y, i1.z, i1.w};
#pragma unroll
              for (int h = 0; h < 8; ++h)
                acc[h] = fmaf(sc[g] * ip[h], __uint_as_float(hi[e][h]) + __uint_as_float(lo[e][h]), acc[h]);
            }
            if (gp == 1) {
#pragma unroll
              for (int h = 0; h < 8; ++h) acc[h] += __uint_as_float(rp[h]);
            }
          }
        } else if (lane == 0) {
          mbar_arrive(&bars[kBarSFree + sbuf]);
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) sl[h] = ok ? acc[h] * p.scale_log2 : -INFINITY;
      }
      // tile maxima: per head (logits) and per scale group (scales), across the 128 rows
      float* redm = red_max + ((tl & 1) * 2 + hh) * 4 * 8;
      uint32_t* reds = red_sc + ((tl & 1) * 2 + hh) * 4 * 4;
      {
        float mx[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) mx[h] = warp_max_f32(sl[h]);
        uint32_t ms[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) ms[g] = warp_max_u32(__float_as_uint(sc[g]));  // scales are >= 0
        if (lane == 0) {
          *reinterpret_cast<float4*>(redm + qd * 8) = make_float4(mx[0], mx[1], mx[2], mx[3]);
          *reinterpret_cast<float4*>(redm + qd * 8 + 4) = make_float4(mx[4], mx[5], mx[6], mx[7]);
          *reinterpret_cast<uint4*>(reds + qd * 4) = make_uint4(ms[0], ms[1], ms[2], ms[3]);
        }
      }
      named_bar_sync(bar_id, 128);
      if (tid == 0) SMLA_TRACE_SET(tl, kEvSoftBar);
      // running maxima of the half's heads (lazy: refreshed only when the tile
      // maximum exceeds them by more than kMaxSlack) and power-of-two bounds
      // of the scale groups
      float alpha[8], beta[4];
      bool up_any = false, rq_changed = false;
      {
        float tmax[8];
        uint32_t smax[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int h = 0; h < 8; ++h) tmax[h] = -INFINITY;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 a0 = *reinterpret_cast<const float4*>(redm + v * 8);
          const float4 a1 = *reinterpret_cast<const float4*>(redm + v * 8 + 4);
          const uint4 c = *reinterpret_cast<const uint4*>(reds + v * 4);
          tmax[0] = fmaxf(tmax[0], a0.x);
          tmax[1] = fmaxf(tmax[1], a0.y);
          tmax[2] = fmaxf(tmax[2], a0.z);
          tmax[3] = fmaxf(tmax[3], a0.w);
          tmax[4] = fmaxf(tmax[4], a1.x);
          tmax[5] = fmaxf(tmax[5], a1.y);
          tmax[6] = fmaxf(tmax[6], a1.z);
          tmax[7] = fmaxf(tmax[7], a1.w);
          smax[0] = max(smax[0], c.x);
          smax[1] = max(smax[1], c.y);
          smax[2] = max(smax[2], c.z);
          smax[3] = max(smax[3], c.w);
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const float nm = fmaxf(m[h], tmax[h]);
          const bool up = nm > m[h] + kMaxSlack;
          const float mnew = nm + kMaxOvershoot;
          alpha[h] = up ? ex2_approx(m[h] - mnew) : 1.f;
          m[h] = up ? mnew : m[h];
          l[h] *= alpha[h];
          up_any |= up;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float sm = __uint_as_float(smax[g]);
          const bool grow = sm > Rq[g];
          const float rn = grow ? pow2_ceil(sm) : Rq[g];
          beta[g] = (grow && Rq[g] > 0.f) ? Rq[g] * rcp_pow2(rn) : 1.f;
          rq_changed |= grow && Rq[g] > 0.f;
          Rq[g] = rn;
        }
      }
      // every thread of a half sees the same shared maxima: the decision is
      // uniform over the half
      if ((up_any || rq_changed) && n_seg_tiles > 0) {
        // O^T holds this segment's earlier P.V: wait for the latest and rescale
        // this half's columns in place (column 8 hh + h and 16 + 8 hh + h: head 8 hh + h)
        wait_s(kBarPvDone + (tl - 1) % kPBufs, ((tl - 1) / kPBufs) & 1);  // P.V(tl - 1) and all before
        if (!dead) {
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t oh[8], ol[8];
            const uint32_t addr = tmem + lane_base + kOCol + 32 * q + 8 * hh;
            tmem_ld8(addr, oh);
            tmem_ld8(addr + 16, ol);
            tmem_ld_wait();
            reg_fence8(oh);
            reg_fence8(ol);
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const float f = alpha[h] * beta[q];
              oh[h] = __float_as_uint(__uint_as_float(oh[h]) * f);
              ol[h] = __float_as_uint(__uint_as_float(ol[h]) * f);
            }
            tmem_st8(addr, oh);
            tmem_st8(addr + 16, ol);
          }
          tmem_st_wait();
        }
      }
      // probabilities and this row's share of the running sums
      float pr[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        pr[h] = ok ? ex2_approx(sl[h] - m[h]) : 0.f;
        l[h] += pr[h];
      }
      if (tl >= kPBufs) wait_s(kBarPvDone + pb, (puse + 1) & 1);  // P buffer free: P.V(tl - 2) done
      // P'_q = kPScale * p * scale_q / R_q as e4m3 hi + lo: MN-major core
      // matrices of 8 rows x 16 codes (heads), hi and lo blocks 128 B apart,
      // row blocks 256 B apart; this thread writes its row's 8 heads
      if (!dead) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float f = sc[g] * (Rq[g] > 0.f ? kPScale * rcp_pow2(Rq[g]) : 0.f);
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) split2_f16(pr[2 * j] * f, pr[2 * j + 1] * f, hw[j], lw[j]);
          const uint32_t base = p0 + pb * kPBuf + g * kPGroup + (r >> 3) * 256 + (r & 7) * 16 + 8 * hh;
          sts64(base, hw[0] | (hw[1] << 16), hw[2] | (hw[3] << 16));
          sts64(base + 128, lw[0] | (lw[1] << 16), lw[2] | (lw[3] << 16));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && !dead) mbar_arrive(&bars[kBarPFull + pb]);
      if (tid == 0) SMLA_TRACE_SET(tl, kEvPWritten);
      ++n_seg_tiles;

      if (ti.seg_end) {
        // the heads' sums over the tile rows: warp butterflies, then the half's
        // four warps through shared memory
        float* rs = red_sum + hh * 4 * 8;
        {
          float v[8];
#pragma unroll
          for (int h = 0; h < 8; ++h) v[h] = l[h];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int h = 0; h < 8; ++h) v[h] += __shfl_xor_sync(kFullMask, v[h], off);
          if (lane == 0) {
            *reinterpret_cast<float4*>(rs + qd * 8) = make_float4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<float4*>(rs + qd * 8 + 4) = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
        named_bar_sync(bar_id, 128);
        wait_s(kBarPvDone + pb, puse & 1);  // last P.V of the segment
        tc_fence_after();
        if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiStart);
        const bool full = (seg_first_kt == 0) && (ti.kt == p.nt - 1);
        const int64_t slot = (int64_t)blockIdx.x + ti.u;
        const int64_t row0 = (int64_t)ti.t * p.H + ti.hg * HG + 8 * hh;  // first head of this half
        // the heads' sums over the segment's rows; a two-part cluster merges raw
        // sums and values (below), the other paths normalize here
        float inv[8], lse_own[8], lt[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) lt[h] = 0.f;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 a0 = *reinterpret_cast<const float4*>(rs + v * 8);
          const float4 a1 = *reinterpret_cast<const float4*>(rs + v * 8 + 4);
          lt[0] += a0.x;
          lt[1] += a0.y;
          lt[2] += a0.z;
          lt[3] += a0.w;
          lt[4] += a1.x;
          lt[5] += a1.y;
          lt[6] += a1.z;
          lt[7] += a1.w;
        }
        const bool two_parts = p.cluster == 2;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          // approximate reciprocal and log2 (a few ulp; lt >= 2^-0.75 here): the
          // correctly rounded library forms cost about a microsecond of cold code
          inv[h] = two_parts ? 1.f : (lt[h] > 0.f ? __fdividef(1.f, lt[h]) : 0.f);
          lse_own[h] = two_parts || !(lt[h] > 0.f) ? -INFINITY : (m[h] + __log2f(lt[h])) * 0.69314718055994530942f;
        }
        // The epilogue runs once per CTA, so its code is fetched cold: it is
        // kept compact (rolled loops over chunks and parts, no divisions).
        // load_out2: this thread's output values of chunks q and (normalized,
        // except in a two-part cluster)
        // chunk q + 1 (one tensor-memory round trip), head 8 hh + h, value column
        // 128 q' + 32 qd + lane.
        auto load_out2 = [&](int q, float (&va)[8], float (&vb)[8]) {
          uint32_t ah[8], al[8], bh[8], bl[8];
          const uint32_t o = tmem + lane_base + kOCol + 32 * q + 8 * hh;
          tmem_ld8(o, ah);
          tmem_ld8(o + 16, al);
          tmem_ld8(o + 32, bh);
          tmem_ld8(o + 48, bl);
          tmem_ld_wait();
          reg_fence8(ah);
          reg_fence8(al);
          reg_fence8(bh);
          reg_fence8(bl);
          const float ra = (q == 0 ? Rq[0] : Rq[2]) * kPScaleInv, rb = (q == 0 ? Rq[1] : Rq[3]) * kPScaleInv;
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            va[h] = (__uint_as_float(ah[h]) + __uint_as_float(al[h])) * ra * inv[h];
            vb[h] = (__uint_as_float(bh[h]) + __uint_as_float(bl[h])) * rb * inv[h];
          }
        };
        const int c0 = 32 * qd + lane;
        if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiLse);
        if (p.cluster > 1) {
          // The unit's parts are the cluster's S CTAs (2 <= S <= 4, one
          // segment each).  CTA `rank` writes the value chunks q with
          // q % S == rank (rank and rank + S).  Every CTA, its last P.V done,
          // tells the others that its operand tiles are free and sends its
          // values of each chunk it does not write to the chunk's CTA, counted
          // on that CTA's receive barrier; each CTA merges what it receives for
          // its own chunks (CTA 0 writes the LSE).  Three or four parts send
          // normalized values and LSEs by 16-byte st.async and merge as
          // M = max_r lse_r, w_r = exp(lse_r - M), out = sum_r w_r out_r /
          // sum_r w_r, lse = M + log sum_r w_r; two parts send raw values and
          // their heads' running maxima and sums by one bulk copy (below).
          // Receive layout of a CTA owning n chunks: the part in peer slot ps
          // (the other ranks in order) has chunk j at (ps * n + j) *
          // kChunkBytes, column c and head h at (c * 16 + h) * 4; the LSEs (or
          // the maxima and sums) follow all values, 64 (128) bytes per slot.
          const int rank = (int)cluster_ctarank();
          const int S = p.cluster;
          const int n_own = rank < 4 - S ? 2 : 1;
          const uint32_t recv = smem_u32(smem + kOffOp);
          const uint32_t recv_bar = smem_u32(&bars[kBarRecv]);
          if (tid == 0 && !dead) {
            mbar_arrive_expect_tx(&bars[kBarRecv], (uint32_t)(S == 2 ? kTwoPartBytes
                                                                    : (S - 1) * (n_own * kChunkBytes + HG * 4)));
#pragma unroll 1
            for (int r = 0; r < S; ++r)
              if (r != rank) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&bars[kBarReady]), (uint32_t)r));
          }
          if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiSignal);
          float own0[8], own1[8];  // this thread's values of chunks rank and rank + S
#pragma unroll
          for (int h = 0; h < 8; ++h) own0[h] = own1[h] = 0.f;
          if (S == 2) {
            // Two parts: this CTA's raw (unnormalized) values of the other's
            // chunks (rank ^ 1 and rank ^ 1 + 2) and its heads' running maxima
            // and sums go to a staging area laid out as the other CTA's receive
            // buffer, then one bulk copy moves them once the other CTA is ready.
            // The staging area follows the receive buffer in the free operand
            // tiles.
            const uint32_t stage = recv + (uint32_t)kSendOff;
            if (!dead) {
#pragma unroll 1
              for (int q2 = 0; q2 < 4; q2 += 2) {
                float vals[2][8];
                load_out2(q2, vals[0], vals[1]);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int q = q2 + e, j = q >> 1;
                  const float(&val)[8] = vals[e];
                  if ((q & 1) == rank) {
#pragma unroll
                    for (int h = 0; h < 8; ++h) {
                      own0[h] = j == 0 ? val[h] : own0[h];
                      own1[h] = j == 0 ? own1[h] : val[h];
                    }
                  } else {
                    const uint32_t dst = stage + (uint32_t)((j * kRows + c0) * (HG * 4) + 32 * hh);
                    st_shared_v4(dst, __float_as_uint(val[0]), __float_as_uint(val[1]), __float_as_uint(val[2]),
                                 __float_as_uint(val[3]));
                    st_shared_v4(dst + 16, __float_as_uint(val[4]), __float_as_uint(val[5]), __float_as_uint(val[6]),
                                 __float_as_uint(val[7]));
                  }
                }
              }
              if (qd == 0 && lane == 0) {
                const uint32_t dst = stage + (uint32_t)(2 * kChunkBytes + 64 * hh);
                st_shared_v4(dst, __float_as_uint(m[0]), __float_as_uint(m[1]), __float_as_uint(m[2]),
                             __float_as_uint(m[3]));
                st_shared_v4(dst + 16, __float_as_uint(m[4]), __float_as_uint(m[5]), __float_as_uint(m[6]),
                             __float_as_uint(m[7]));
                st_shared_v4(dst + 32, __float_as_uint(lt[0]), __float_as_uint(lt[1]), __float_as_uint(lt[2]),
                             __float_as_uint(lt[3]));
                st_shared_v4(dst + 48, __float_as_uint(lt[4]), __float_as_uint(lt[5]), __float_as_uint(lt[6]),
                             __float_as_uint(lt[7]));
              }
            }
            fence_proxy_async_smem();  // the bulk copy reads the staging area through the async proxy
            named_bar_sync(3, 32 * kSoftWarps);
            if (tid == 0) SMLA_TRACE_SET(tl, kEvMergeWait);
            if (tid == 0 && !dead) {
              if (SMLA_WAIT(kBarReady, 0)) {
                if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiReady);
                const uint32_t other = (uint32_t)(rank ^ 1);
                bulk_copy_to_peer(mapa_shared(recv, other), stage, (uint32_t)kTwoPartBytes, mapa_shared(recv_bar, other));
              }
            }
          } else {
          if (tid == 0) SMLA_TRACE_SET(tl, kEvMergeWait);
          if (!dead) dead = !SMLA_WAIT(kBarReady, 0);
          dead = __any_sync(kFullMask, dead);
          if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiReady);
          if (!dead) {
#pragma unroll 1
            for (int q2 = 0; q2 < 4; q2 += 2) {
              float vals[2][8];
              load_out2(q2, vals[0], vals[1]);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int q = q2 + e;
                const float(&val)[8] = vals[e];
                const int o = q < S ? q : q - S, j = q < S ? 0 : 1;  // the chunk's CTA and its index there
                if (o == rank) {
#pragma unroll
                  for (int h = 0; h < 8; ++h) {
                    own0[h] = j == 0 ? val[h] : own0[h];
                    own1[h] = j == 0 ? own1[h] : val[h];
                  }
                } else {
                  const int n_o = o < 4 - S ? 2 : 1, ps = rank < o ? rank : rank - 1;
                  const uint32_t dst =
                      mapa_shared(recv + (uint32_t)(((ps * n_o + j) * kRows + c0) * (HG * 4) + 32 * hh), (uint32_t)o);
                  const uint32_t bar = mapa_shared(recv_bar, (uint32_t)o);
                  st_async_v4(dst, val[0], val[1], val[2], val[3], bar);
                  st_async_v4(dst + 16, val[4], val[5], val[6], val[7], bar);
                }
              }
            }
            if (qd == 0 && lane == 0) {
#pragma unroll 1
              for (int o = 0; o < S; ++o) {
                if (o == rank) continue;
                const int n_o = o < 4 - S ? 2 : 1, ps = rank < o ? rank : rank - 1;
                const uint32_t dst = mapa_shared(
                    recv + (uint32_t)((S - 1) * n_o * kChunkBytes + ps * HG * 4 + 32 * hh), (uint32_t)o);
                const uint32_t bar = mapa_shared(recv_bar, (uint32_t)o);
                st_async_v4(dst, lse_own[0], lse_own[1], lse_own[2], lse_own[3], bar);
                st_async_v4(dst + 16, lse_own[4], lse_own[5], lse_own[6], lse_own[7], bar);
              }
            }
          }
          }
          if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiSent);
          if (!dead) dead = !SMLA_WAIT(kBarRecv, 0);
          dead = __any_sync(kFullMask, dead);
          if (tid == 0) SMLA_TRACE_SET(tl, kEvMergeGo);
          if (!dead && S == 2) {
            // Two parts (the usual cluster): straight-line code, since it runs
            // once per CTA and is fetched cold.  Each CTA owns chunks rank and
            // rank + 2; the other part's raw values are in peer slot 0, its
            // maxima and sums after them.  Per head, with d = m_own - m_peer
            // (log2 units): the smaller part is scaled by e = 2^-|d|, the sum is
            // L = l_own a_own + l_peer a_peer and out = (O_own a_own + O_peer
            // a_peer) / L, lse = ln 2 (max(m_own, m_peer) + log2 L): one
            // exponential and one reciprocal per head.
            const uint32_t ml_base = recv + (uint32_t)(2 * kChunkBytes) + 64 * hh;
            const float4 ma = lds_f32x4(ml_base), mb = lds_f32x4(ml_base + 16);
            const float4 la = lds_f32x4(ml_base + 32), lb = lds_f32x4(ml_base + 48);
            const float mp[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
            const float lp[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
            float w1[8], m_mine = -INFINITY, s_mine = 1.f;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const float M = fmaxf(m[h], mp[h]);
              const bool own_big = m[h] >= mp[h];
              const float e = M == -INFINITY ? 0.f : ex2_approx(-fabsf(m[h] - mp[h]));
              const float a_own = own_big ? 1.f : e, a_peer = own_big ? e : 1.f;
              const float L = lt[h] * a_own + lp[h] * a_peer;
              const float r = L > 0.f ? __fdividef(1.f, L) : 0.f;
              const float ro = a_own * r;
              own0[h] *= ro;  // the own part's weighted values
              own1[h] *= ro;
              w1[h] = a_peer * r;
              m_mine = lane == h ? M : m_mine;
              s_mine = lane == h ? L : s_mine;
            }
            if (rank == 0 && qd == 0 && lane < 8)
              p.lse[row0 + lane] =
                  s_mine > 0.f ? (m_mine + __log2f(s_mine)) * 0.69314718055994530942f : -INFINITY;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const uint32_t src = recv + (uint32_t)((j * kRows + c0) * (HG * 4) + 32 * hh);
              const float4 x0 = lds_f32x4(src), x1 = lds_f32x4(src + 16);
              const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
              const int q = rank + 2 * j;
#pragma unroll
              for (int h = 0; h < 8; ++h)
                p.out[(row0 + h) * kDv + 128 * q + c0] =
                    __float2bfloat16_rn(fmaf(w1[h], x[h], j == 0 ? own0[h] : own1[h]));
            }
          } else if (!dead) {
            // merge weights per head: the maximum M, 1 / sum_r w_r and the own
            // part's weight are kept; a received part's weight is recomputed
            // from its LSE where it is used
            const uint32_t lse_base = recv + (uint32_t)((S - 1) * n_own * kChunkBytes) + 32 * hh;
            float mx[8], iw[8], w0[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              mx[h] = lse_own[h];
              iw[h] = 0.f;
            }
#pragma unroll 1
            for (int ps = 0; ps < S - 1; ++ps) {
              const float4 a = lds_f32x4(lse_base + ps * HG * 4), b = lds_f32x4(lse_base + ps * HG * 4 + 16);
              const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
              for (int h = 0; h < 8; ++h) mx[h] = fmaxf(mx[h], v[h]);
            }
#pragma unroll 1
            for (int ps = 0; ps < S - 1; ++ps) {
              const float4 a = lds_f32x4(lse_base + ps * HG * 4), b = lds_f32x4(lse_base + ps * HG * 4 + 16);
              const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
              for (int h = 0; h < 8; ++h) iw[h] += mx[h] == -INFINITY ? 0.f : __expf(v[h] - mx[h]);
            }
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              w0[h] = mx[h] == -INFINITY ? 0.f : __expf(lse_own[h] - mx[h]);
              const float wsum = iw[h] + w0[h];
              iw[h] = wsum > 0.f ? __fdividef(1.f, wsum) : 0.f;  // wsum in [1, S]
              w0[h] *= iw[h];
              if (rank == 0 && qd == 0 && lane == h) p.lse[row0 + h] = wsum > 0.f ? mx[h] + __logf(wsum) : -INFINITY;
            }
#pragma unroll 1
            for (int j = 0; j < n_own; ++j) {
              float acc[8];
#pragma unroll
              for (int h = 0; h < 8; ++h) acc[h] = w0[h] * (j == 0 ? own0[h] : own1[h]);
#pragma unroll 1
              for (int ps = 0; ps < S - 1; ++ps) {
                const float4 a = lds_f32x4(lse_base + ps * HG * 4), b = lds_f32x4(lse_base + ps * HG * 4 + 16);
                const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                const uint32_t src = recv + (uint32_t)(((ps * n_own + j) * kRows + c0) * (HG * 4) + 32 * hh);
                const float4 x0 = lds_f32x4(src), x1 = lds_f32x4(src + 16);
                const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                for (int h = 0; h < 8; ++h)
                  acc[h] = fmaf(mx[h] == -INFINITY ? 0.f : __expf(v[h] - mx[h]) * iw[h], x[h], acc[h]);
              }
              const int q = rank + j * S;
#pragma unroll
              for (int h = 0; h < 8; ++h) p.out[(row0 + h) * kDv + 128 * q + c0] = __float2bfloat16_rn(acc[h]);
            }
          }
          if (tid == 0) SMLA_TRACE_SET(tl, kEvEpiWritten);
        } else {
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            if (qd == 0 && lane == h && !dead) {
              if (full)
                p.lse[row0 + h] = lse_own[h];
              else
                p.part_lse[slot * HG + 8 * hh + h] = lse_own[h];
            }
          }
          if (!dead) {
#pragma unroll 1
            for (int q2 = 0; q2 < 4; q2 += 2) {
              float vals[2][8];
              load_out2(q2, vals[0], vals[1]);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int q = q2 + e;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                  if (full)
                    p.out[(row0 + h) * kDv + 128 * q + c0] = __float2bfloat16_rn(vals[e][h]);
                  else
                    p.part_o[(slot * HG + 8 * hh + h) * kDv + 128 * q + c0] = vals[e][h];
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !dead) mbar_arrive(&bars[kBarOFree]);
        if (tid == 0) SMLA_TRACE_SET(tl, kEvEpi);
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
  // no CTA leaves while another CTA of its cluster may still write into its shared memory
  if (p.cluster > 1) cluster_sync_relaxed();
  if (tid == 0) SMLA_TRACE_SET(0, kEvExit);
}

// Per-device flag: the kernel's dynamic shared memory limit has been raised.
std::once_flag g_attr_once[64];
cudaError_t g_attr_err[64];

}  // namespace

#ifdef SMLA_TRACE
extern "C" int smla_trace_set_fp8(unsigned long long* buf) {
  return (int)cudaMemcpyToSymbol(g_smla_trace_fp8, &buf, sizeof(buf));
}
#endif

namespace {

cudaError_t set_smem_attr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_attr_once[dev], [dev] {
    g_attr_err[dev] =
        cudaFuncSetAttribute(sparse_mla_decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  });
  return g_attr_err[dev];
}

// Clusters of s CTAs of the decode kernel that the GPU holds at once (one CTA
// per SM; a cluster lives on one GPC, so fewer than SMs / s when the GPCs'
// SM counts are not multiples of s), cached per device.  0 when unknown.
int max_active_clusters(int s) {
  static std::mutex mu;
  static int cached[64][kMaxCluster + 1] = {};
  int dev = 0;
  if (s < 2 || s > kMaxCluster || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev][s] != 0) return cached[dev][s] > 0 ? cached[dev][s] : 0;
  int n = 0;
  if (set_smem_attr() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)s, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)s;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_decode_fp8_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
  }
  cached[dev][s] = n > 0 ? n : -1;
  return n;
}

// Units cut into s parts run as clusters when all of them are resident at
// once (if the query failed, assume they are).
bool clusters_fit(int64_t units, int s) {
  const int n = max_active_clusters(s);
  return n <= 0 || units <= n;
}

}  // namespace

AttnPlan plan_decode_fp8(int T, int H, int K, int num_splits, int num_sms) {
  if (wide_supported(H)) return plan_decode_wide(T, K, num_splits, num_sms);
  AttnPlan pl;
  pl.HG = HG;
  pl.n_hg = H / HG;
  pl.nt = K > 0 ? (K + kRows - 1) / kRows : 1;
  pl.units = (int64_t)T * pl.n_hg;
  pl.total = pl.units * pl.nt;
  int64_t G;
  if (num_splits > 0) {
    G = pl.units * (int64_t)num_splits;
  } else {
    // Automatic.  Candidates: equal contiguous ranges over all SMs, or every
    // unit cut into s parts (one segment per CTA: one Q preparation and one
    // epilogue each).  Parts of a unit are merged on chip by a cluster when
    // 2 <= s <= kMaxCluster and all the clusters are resident at once, else
    // by the combine kernel.  Cost in tiles: the largest range or part, one
    // tile per segment boundary inside a range, kCombineTiles when the
    // combine runs (measured: about two tiles); on a tie the on-chip merge.
    constexpr int64_t kCombineTiles = 2;
    const int64_t tpc = (pl.total + num_sms - 1) / num_sms;
    const bool range_cut = !(pl.total % num_sms == 0 && (pl.total / num_sms) % pl.nt == 0);
    int64_t best = 2 * (tpc + (tpc + pl.nt - 1) / pl.nt + (range_cut ? kCombineTiles : 0)) + (range_cut ? 1 : 0);
    G = num_sms;
    const int64_t s_max = pl.units > 0 ? std::min<int64_t>(num_sms / pl.units, pl.nt) : 0;
    for (int64_t s = s_max; s >= 1; --s) {
      const bool on_chip = s == 1 || (s <= kMaxCluster && clusters_fit(pl.units, (int)s));
      const int64_t cost = 2 * ((pl.nt + s - 1) / s + (on_chip ? 0 : kCombineTiles)) + (on_chip ? 0 : 1);
      if (cost < best) {
        best = cost;
        G = pl.units * s;
      }
    }
  }
  if (G > pl.total) G = pl.total;
  if (G < 1) G = 1;
  pl.G = (int)G;
  pl.need_combine = !(pl.total % pl.G == 0 && (pl.total / pl.G) % pl.nt == 0);
  // every unit cut into s parts aligned with the CTA ranges: a cluster of s
  // CTAs per unit merges them in distributed shared memory
  if (pl.need_combine && pl.G % pl.units == 0) {
    const int64_t s = pl.G / pl.units;
    if (s >= 2 && s <= kMaxCluster && clusters_fit(pl.units, (int)s)) {
      pl.cluster = (int)s;
      pl.need_combine = false;
    }
  }
  if (pl.need_combine) {
    const int64_t n_slots = (int64_t)pl.G + pl.units - 1;
    const size_t lse_bytes = (size_t)(((n_slots * HG * 4) + 255) / 256) * 256;
    pl.ws_bytes = kWsStatusBytes + lse_bytes + (size_t)n_slots * HG * kDv * 4;
  } else {
    pl.ws_bytes = kWsStatusBytes;  // the status word
  }
  return pl;
}

cudaError_t launch_decode_fp8(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream) {
  if (plan.HG == 128) return launch_decode_wide(a, plan, stream);
  cudaError_t e = set_smem_attr();
  if (e != cudaSuccess) return e;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  const int64_t n_slots = (int64_t)plan.G + plan.units - 1;
  Params p;
  p.cluster = plan.cluster;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.cache = a.cache;
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.G, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)plan.cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = plan.cluster > 1 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, sparse_mla_decode_fp8_kernel, p);
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess || !plan.need_combine) return e;
  e = launch_combine<HG>(p.part_o, p.part_lse, p.out, p.lse, p.H, p.n_hg, p.nt, p.total, p.G, plan.units, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace smla
