// Internal launch interface between the C-ABI layer and the CUDA kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace smla {

cudaError_t launch_quantize_store(const void* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T, int64_t NB,
                                  cudaStream_t stream);

cudaError_t launch_translate(const int32_t* indices, const int32_t* block_table, const int32_t* req_id,
                             int32_t* slots, int T, int K, int R, int MB, int64_t NB, cudaStream_t stream);

// Separate-mode FP8 prefill: index translation with a prefill workspace, and
// the gather + up-convert of prefill requests' cache rows into a bf16 workspace.
cudaError_t launch_translate_ws(const int32_t* indices, const int32_t* block_table, const int32_t* req_id,
                                const int32_t* prefill_req_id, const int32_t* starts, int P, int32_t* out, int T,
                                int K, int R, int MB, int64_t NB, cudaStream_t stream);
cudaError_t launch_gather_upconvert(const uint8_t* cache, int64_t NB, const int32_t* block_table, int R, int MB,
                                    const int32_t* seq_lens, const int32_t* starts, void* ws, int64_t N,
                                    int num_sms, cudaStream_t stream);

// MLA weight absorption around the attention (smla_absorb.cu): per-head GEMMs
// on the tensor cores.  status: a device word that a timed-out wait sets.
cudaError_t launch_absorb_q(const void* q, const void* w_uk_t, void* q_out, int T, int H, int P, int* status,
                            cudaStream_t stream);
cudaError_t launch_v_up_proj(const void* attn_out, const void* w_uv, void* out, int T, int H, int V, int* status,
                             cudaStream_t stream);

// Work decomposition of one sparse-attention call: units are (token, head
// group) pairs, each split into nt tiles of 64 top-k rows; G persistent CTAs
// take contiguous, balanced ranges of the unit-major tile sequence.
struct AttnPlan {
  int HG;             // heads per work unit
  int n_hg;           // head groups per token
  int nt;             // tiles per unit
  int64_t units;      // T * n_hg
  int64_t total;      // units * nt
  int G;              // CTAs
  bool need_combine;  // some unit spans more than one CTA, merged by the combine kernel
  size_t ws_bytes;    // workspace bytes (status word + partial results)
  int cluster = 1;    // > 1: every unit is split into `cluster` parts run by one thread-block
                      // cluster, merged in distributed shared memory (no combine kernel)
  bool fused = false; // 128-head FP8 decode: every split unit has two parts, merged in the
                      // attention kernel by whichever part finishes second (no combine kernel)
};

AttnPlan plan_attention(bool fp8, int T, int H, int K, int num_splits, int num_sms);
AttnPlan plan_decode_fp8(int T, int H, int K, int num_splits, int num_sms);
AttnPlan plan_prefill_bf16(int T, int H, int K, int num_splits, int num_sms);

struct AttnArgs {
  const void* q;
  const uint8_t* cache;      // FP8 decode: [NB, 64, 656]
  const void* kv;            // BF16 prefill: [N, 576]
  const int32_t* indices;    // [T, K]
  const int32_t* block_table;
  const int32_t* req_id;
  void* out;                 // bf16 [T, H, 512]
  float* lse;                // [T, H]
  void* workspace;
  float sm_scale;
  int T, H, K, R, MB;
  int64_t NB;                // physical blocks (FP8) or kv rows (BF16)
};

cudaError_t launch_attention(bool fp8, const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);

// Attention with all 128 heads of a token per CTA pair (smla_wide.cu), over
// the bf16 latent buffer (prefill) or the FP8 paged cache (decode).
bool wide_supported(int H);
AttnPlan plan_prefill_wide(int T, int K, int num_splits, int num_sms);
AttnPlan plan_decode_wide(int T, int K, int num_splits, int num_sms);
cudaError_t launch_prefill_wide(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);
cudaError_t launch_decode_wide(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);
cudaError_t launch_decode_fp8(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);

// The 128-head FP8 decode with the query quantized to e4m3 (two terms) and
// both products on the FP8 tensor path, the row scales folded into P
// (smla_wide8.cu).
AttnPlan plan_decode_wide8(int T, int K, int num_splits, int num_sms);
cudaError_t launch_decode_wide8(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);
cudaError_t launch_prefill_bf16(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);

// The NVFP4 cache (smla_nvfp4.cu): quantize-and-store, and the decode's
// staging of each token's top-k rows as exact bf16 rows ([T * K] row indices,
// -1 = invalid, then [T * K, 576] bf16 rows; nvfp4_stage_bytes in all).
cudaError_t launch_nvfp4_store(const void* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T, int64_t NB,
                               cudaStream_t stream);
size_t nvfp4_stage_bytes(int T, int K);
cudaError_t launch_nvfp4_stage(const uint8_t* cache, int64_t NB, const int32_t* indices, const int32_t* block_table,
                               const int32_t* req_id, int T, int K, int R, int MB, void* stage, cudaStream_t stream);
// The native NVFP4 decode (smla_attn.cu) below 128 heads, in 16-head groups:
// a.cache is the NVFP4 cache, a.NB its blocks.
bool nvfp4_native_supported(int H);
AttnPlan plan_decode_nvfp4(int T, int H, int K, int num_splits, int num_sms);
cudaError_t launch_decode_nvfp4(const AttnArgs& a, const AttnPlan& plan, cudaStream_t stream);

// Offsets inside the workspace.
constexpr size_t kWsStatusBytes = 256;

}  // namespace smla
