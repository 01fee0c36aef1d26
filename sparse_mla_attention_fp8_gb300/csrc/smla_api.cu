// C-ABI entry points: argument validation, work planning, workspace handling
// and kernel dispatch.  Every function returns a status code; nothing throws
// and nothing synchronizes the host on the launch path.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/smla.h"
#include "smla_kernels.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SMLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;

struct DeviceState {
  int num_sms = 0;
  void* ws = nullptr;
  size_t ws_bytes = 0;
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(SMLA_ERR_UNSUPPORTED, "device ordinal %d out of range", *dev);
  return SMLA_OK;
}

int num_sms(int* out) {
  int dev;
  int rc = current_device(&dev);
  if (rc != SMLA_OK) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev[dev].num_sms == 0) {
    int n = 0;
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_dev[dev].num_sms = n;
  }
  *out = g_dev[dev].num_sms;
  return SMLA_OK;
}

// Library-cached workspace of the current device, grown on demand.  Growing
// frees the old buffer after a device synchronize, so callers must not have
// other work using it in flight on other streams.
int cached_workspace(size_t need, void** out) {
  int dev;
  int rc = current_device(&dev);
  if (rc != SMLA_OK) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.ws_bytes < need) {
    if (d.ws) {
      cudaDeviceSynchronize();
      cudaFree(d.ws);
      d.ws = nullptr;
      d.ws_bytes = 0;
    }
    size_t sz = need < (size_t(1) << 20) ? (size_t(1) << 20) : need;
    cudaError_t e = cudaMalloc(&d.ws, sz);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    e = cudaMemset(d.ws, 0, sz);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace)");
    d.ws_bytes = sz;
  }
  *out = d.ws;
  return SMLA_OK;
}

int check_heads(int H) {
  if (H <= 0 || H % 16 != 0 || H > 128)
    return fail(SMLA_ERR_UNSUPPORTED, "H=%d unsupported: must be a positive multiple of 16, at most 128", H);
  return SMLA_OK;
}

// qfp8: the FP8-query variant of the decode (its own kernel at 128 heads).
smla::AttnPlan plan_for(bool fp8, bool qfp8, int T, int H, int K, int num_splits, int sms) {
  if (fp8 && qfp8 && smla::wide_supported(H)) return smla::plan_decode_wide8(T, K, num_splits, sms);
  return smla::plan_attention(fp8, T, H, K, num_splits, sms);
}

int run_attention(bool fp8, smla::AttnArgs& a, int num_splits, void* workspace, size_t workspace_bytes,
                  void* stream, bool qfp8 = false) {
  int sms = 0;
  int rc = num_sms(&sms);
  if (rc != SMLA_OK) return rc;
  const smla::AttnPlan plan = plan_for(fp8, qfp8, a.T, a.H, a.K, num_splits, sms);
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < plan.ws_bytes)
      return fail(SMLA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, plan.ws_bytes);
  } else {
    rc = cached_workspace(plan.ws_bytes, &workspace);
    if (rc != SMLA_OK) return rc;
  }
  a.workspace = workspace;
  cudaError_t e = fp8 && qfp8 && plan.HG == 128
                      ? smla::launch_decode_wide8(a, plan, static_cast<cudaStream_t>(stream))
                      : smla::launch_attention(fp8, a, plan, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fp8 ? "sparse_mla_decode_fp8 launch" : "sparse_mla_prefill_bf16 launch");
  return SMLA_OK;
}

size_t workspace_bytes_for(bool fp8, int T, int H, int K, int num_splits) {
  if (T <= 0 || check_heads(H) != SMLA_OK || K < 0) return 0;
  int sms = 0;
  if (num_sms(&sms) != SMLA_OK) return 0;
  const size_t ws = smla::plan_attention(fp8, T, H, K, num_splits, sms).ws_bytes;
  // the decode's size covers its FP8-query variant too
  const size_t ws8 = fp8 ? plan_for(true, true, T, H, K, num_splits, sms).ws_bytes : 0;
  return ws > ws8 ? ws : ws8;
}

// ---- fixed scratch for sparse_mla_decode_fp8_noalloc: part of the module
// image, so no call ever allocates.  Its device address is looked up once per
// device, with that device current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SMLA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(void** out) {
  int dev;
  int rc = current_device(&dev);
  if (rc != SMLA_OK) return rc;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return SMLA_OK;
}

// Bytes of the translated index rows of sparse_mla_prefill_fp8 (256-byte aligned).
size_t fp8_prefill_index_bytes(int T, int K) { return (((size_t)T * (size_t)K * 4 + 255) / 256) * 256; }

int decode_entry(bool qfp8, const void* q, const uint8_t* kv_cache, const int32_t* indices,
                 const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale, int num_splits,
                 void* out, float* lse, int T, int H, int K, int R, int MB, int NB, void* workspace,
                 size_t workspace_bytes, void* stream) {
  if (T < 0 || K < 0 || R <= 0 || MB <= 0 || NB <= 0 || num_splits < 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d R=%d MB=%d NB=%d num_splits=%d", T, K, R, MB, NB,
                num_splits);
  int rc = check_heads(H);
  if (rc != SMLA_OK) return rc;
  if (T == 0) return SMLA_OK;
  if (!q || !kv_cache || (!indices && K > 0) || !block_table || !req_id_per_token || !out || !lse)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return fail(SMLA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  smla::AttnArgs a{};
  a.q = q;
  a.cache = kv_cache;
  a.kv = nullptr;
  a.indices = indices;
  a.block_table = block_table;
  a.req_id = req_id_per_token;
  a.out = out;
  a.lse = lse;
  a.sm_scale = sm_scale;
  a.T = T;
  a.H = H;
  a.K = K;
  a.R = R;
  a.MB = MB;
  a.NB = NB;
  return run_attention(true, a, num_splits, workspace, workspace_bytes, stream, qfp8);
}

}  // namespace

extern "C" {

int sparse_mla_decode_fp8(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                          const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                          int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB, int NB,
                          void* workspace, size_t workspace_bytes, void* stream) {
  return decode_entry(false, q, kv_cache, indices, block_table, req_id_per_token, sm_scale, num_splits, out, lse,
                      T, H, K, R, MB, NB, workspace, workspace_bytes, stream);
}

int sparse_mla_decode_fp8_qfp8(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                               const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                               int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB, int NB,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return decode_entry(true, q, kv_cache, indices, block_table, req_id_per_token, sm_scale, num_splits, out, lse,
                      T, H, K, R, MB, NB, workspace, workspace_bytes, stream);
}

int sparse_mla_decode_fp8_noalloc(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                                  const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                                  int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB,
                                  int NB, void* stream) {
  if (T < 0 || K < 0 || R <= 0 || MB <= 0 || NB <= 0 || num_splits < 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d R=%d MB=%d NB=%d num_splits=%d", T, K, R, MB, NB,
                num_splits);
  int rc = check_heads(H);
  if (rc != SMLA_OK) return rc;
  if (T == 0) return SMLA_OK;
  if (!q || !kv_cache || (!indices && K > 0) || !block_table || !req_id_per_token || !out || !lse)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return fail(SMLA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  int sms = 0;
  rc = num_sms(&sms);
  if (rc != SMLA_OK) return rc;
  const smla::AttnPlan plan = smla::plan_decode_fp8(T, H, K, num_splits, sms);
  if (plan.ws_bytes > SMLA_NOALLOC_SCRATCH_BYTES)
    return fail(SMLA_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch; the fixed scratch holds %zu (use num_splits=1, fewer "
                "tokens per call, or sparse_mla_decode_fp8 with a workspace)",
                plan.ws_bytes, (size_t)SMLA_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != SMLA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word starts at zero (the array is zero-initialised when the
  // module loads) and only a kernel wait that runs out sets it, so nothing
  // needs clearing per call: smla_read_noalloc_status reads and clears it.
  // Partial results are written before they are read.
  smla::AttnArgs a{};
  a.q = q;
  a.cache = kv_cache;
  a.kv = nullptr;
  a.indices = indices;
  a.block_table = block_table;
  a.req_id = req_id_per_token;
  a.out = out;
  a.lse = lse;
  a.sm_scale = sm_scale;
  a.T = T;
  a.H = H;
  a.K = K;
  a.R = R;
  a.MB = MB;
  a.NB = NB;
  a.workspace = scratch;
  cudaError_t e = smla::launch_decode_fp8(a, plan, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_decode_fp8_noalloc launch");
  return SMLA_OK;
}

size_t sparse_mla_decode_workspace_bytes(int T, int H, int K, int num_splits) {
  return workspace_bytes_for(true, T, H, K, num_splits);
}

int sparse_mla_prefill_bf16(const void* q, const void* kv, const int32_t* indices, float sm_scale,
                            int num_splits, void* out, float* lse, int T, int H, int N, int K, void* workspace,
                            size_t workspace_bytes, void* stream) {
  if (T < 0 || K < 0 || N <= 0 || num_splits < 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d N=%d K=%d num_splits=%d", T, N, K, num_splits);
  int rc = check_heads(H);
  if (rc != SMLA_OK) return rc;
  if (T == 0) return SMLA_OK;
  if (!q || !kv || (!indices && K > 0) || !out || !lse) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(kv) || !aligned16(out))
    return fail(SMLA_ERR_INVALID_ARG, "q, kv and out must be 16-byte aligned");
  smla::AttnArgs a{};
  a.q = q;
  a.cache = nullptr;
  a.kv = kv;
  a.indices = indices;
  a.block_table = nullptr;
  a.req_id = nullptr;
  a.out = out;
  a.lse = lse;
  a.sm_scale = sm_scale;
  a.T = T;
  a.H = H;
  a.K = K;
  a.R = 1;
  a.MB = 1;
  a.NB = N;
  return run_attention(false, a, num_splits, workspace, workspace_bytes, stream);
}

size_t sparse_mla_prefill_workspace_bytes(int T, int H, int K, int num_splits) {
  return workspace_bytes_for(false, T, H, K, num_splits);
}

// ---- separate-mode FP8 prefill

size_t sparse_mla_prefill_fp8_workspace_bytes(int T, int H, int K, int num_splits) {
  const size_t attn = workspace_bytes_for(false, T, H, K, num_splits);
  if (attn == 0) return 0;
  return ((attn + 255) / 256) * 256 + fp8_prefill_index_bytes(T, K);
}

int sparse_mla_gather_upconvert_fp8(const uint8_t* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                                    const int32_t* workspace_starts, int R, int MB, int NB, void* kv_workspace, int N,
                                    void* stream) {
  if (R < 0 || MB <= 0 || NB <= 0 || N < 0) return fail(SMLA_ERR_INVALID_ARG, "bad sizes R=%d MB=%d NB=%d N=%d", R, MB, NB, N);
  if (R == 0 || N == 0) return SMLA_OK;
  if (!kv_cache || !block_table || !seq_lens || !workspace_starts || !kv_workspace)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(kv_cache) || !aligned16(kv_workspace))
    return fail(SMLA_ERR_INVALID_ARG, "kv_cache and kv_workspace must be 16-byte aligned");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  int sms = 0;
  int rc = num_sms(&sms);
  if (rc != SMLA_OK) return rc;
  cudaError_t e = smla::launch_gather_upconvert(kv_cache, NB, block_table, R, MB, seq_lens, workspace_starts,
                                                kv_workspace, N, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_gather_upconvert_fp8 launch");
  return SMLA_OK;
}

int sparse_mla_translate_indices_workspace(const int32_t* indices, const int32_t* block_table,
                                           const int32_t* req_id_per_token, const int32_t* prefill_request_id,
                                           const int32_t* workspace_starts, int P, int32_t* out, int T, int K, int R,
                                           int MB, int NB, void* stream) {
  if (T < 0 || K < 0 || R <= 0 || MB <= 0 || NB <= 0 || P < 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d R=%d MB=%d NB=%d P=%d", T, K, R, MB, NB, P);
  if (T == 0 || K == 0) return SMLA_OK;
  if (!indices || !block_table || !req_id_per_token || !prefill_request_id || (!workspace_starts && P > 0) || !out)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  cudaError_t e = smla::launch_translate_ws(indices, block_table, req_id_per_token, prefill_request_id,
                                            workspace_starts, P, out, T, K, R, MB, NB, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_translate_indices_workspace launch");
  return SMLA_OK;
}

int sparse_mla_prefill_fp8(const void* q, const uint8_t* kv_cache, const int32_t* indices, const int32_t* block_table,
                           const int32_t* req_id_per_token, const int32_t* seq_lens, const int32_t* workspace_starts,
                           float sm_scale, int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB,
                           int NB, void* kv_workspace, int N, void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || K < 0 || R <= 0 || MB <= 0 || NB <= 0 || N <= 0 || num_splits < 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d R=%d MB=%d NB=%d N=%d num_splits=%d", T, K, R, MB, NB, N,
                num_splits);
  int rc = check_heads(H);
  if (rc != SMLA_OK) return rc;
  if (T == 0) return SMLA_OK;
  if (!q || !kv_cache || (!indices && K > 0) || !block_table || !req_id_per_token || !seq_lens || !workspace_starts ||
      !out || !lse || !kv_workspace)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out) || !aligned16(kv_workspace))
    return fail(SMLA_ERR_INVALID_ARG, "q, kv_cache, out and kv_workspace must be 16-byte aligned");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  int sms = 0;
  rc = num_sms(&sms);
  if (rc != SMLA_OK) return rc;
  const smla::AttnPlan plan = smla::plan_attention(false, T, H, K, num_splits, sms);
  const size_t need = ((plan.ws_bytes + 255) / 256) * 256 + fp8_prefill_index_bytes(T, K);
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < need) return fail(SMLA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
  } else {
    rc = cached_workspace(need, &workspace);
    if (rc != SMLA_OK) return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // 1. the chunk's requests' rows, up-converted to bf16 into kv_workspace
  cudaError_t e = smla::launch_gather_upconvert(kv_cache, NB, block_table, R, MB, seq_lens, workspace_starts,
                                                kv_workspace, N, sms, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_prefill_fp8 gather launch");
  // 2. the tokens' logical indices -> rows of kv_workspace (every token is a prefill token of request req_id[t]);
  // the workspace holds the prefill's own workspace first (its status word leads), then these rows
  const size_t attn_bytes = ((plan.ws_bytes + 255) / 256) * 256;
  int32_t* rows = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + attn_bytes);
  if (K > 0) {
    e = smla::launch_translate_ws(indices, block_table, req_id_per_token, req_id_per_token, workspace_starts, R, rows,
                                  T, K, R, MB, NB, s);
    if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_prefill_fp8 translate launch");
  }
  // 3. the bf16 prefill over kv_workspace; its own workspace follows the rows
  smla::AttnArgs a{};
  a.q = q;
  a.cache = nullptr;
  a.kv = kv_workspace;
  a.indices = rows;
  a.block_table = nullptr;
  a.req_id = nullptr;
  a.out = out;
  a.lse = lse;
  a.sm_scale = sm_scale;
  a.T = T;
  a.H = H;
  a.K = K;
  a.R = 1;
  a.MB = 1;
  a.NB = N;
  a.workspace = workspace;
  e = smla::launch_attention(false, a, plan, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_prefill_fp8 attention launch");
  return SMLA_OK;
}

int sparse_mla_prefill_chunks(const int32_t* seq_lens, int R, int64_t workspace_rows, int32_t* chunk_ends,
                              int32_t* workspace_starts, int* n_chunks) {
  if (R < 0 || workspace_rows <= 0) return fail(SMLA_ERR_INVALID_ARG, "bad sizes R=%d workspace_rows=%lld", R,
                                                (long long)workspace_rows);
  if (!n_chunks || (R > 0 && (!seq_lens || !chunk_ends || !workspace_starts)))
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  int n = 0;
  int64_t used = 0;
  for (int r = 0; r < R; ++r) {
    const int64_t len = seq_lens[r];
    if (len < 0) return fail(SMLA_ERR_INVALID_ARG, "seq_lens[%d] = %lld is negative", r, (long long)len);
    if (len > workspace_rows)
      return fail(SMLA_ERR_WORKSPACE, "request %d has %lld rows, the workspace holds %lld", r, (long long)len,
                  (long long)workspace_rows);
    if (r > 0 && used + len > workspace_rows) {  // close the chunk before this request
      chunk_ends[n++] = r;
      used = 0;
    }
    workspace_starts[r] = (int32_t)used;
    used += len;
  }
  if (R > 0) chunk_ends[n++] = R;
  *n_chunks = n;
  return SMLA_OK;
}

int sparse_mla_attention_plan(int fp8, int T, int H, int K, int num_splits, int* launches, int* ctas) {
  if (!launches || !ctas) return fail(SMLA_ERR_INVALID_ARG, "null output pointer");
  if (T <= 0 || K < 0 || num_splits < 0) return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d num_splits=%d", T, K, num_splits);
  int rc = check_heads(H);
  if (rc != SMLA_OK) return rc;
  int sms = 0;
  rc = num_sms(&sms);
  if (rc != SMLA_OK) return rc;
  const smla::AttnPlan plan = smla::plan_attention(fp8 != 0, T, H, K, num_splits, sms);
  // the 128-head FP8 path prepares Q in a launch of its own
  *launches = (plan.need_combine ? 2 : 1) + (fp8 != 0 && plan.HG == 128 ? 1 : 0);
  *ctas = plan.HG == 128 ? 2 * plan.G : plan.G;  // the 128-head kernels run CTA pairs
  return SMLA_OK;
}

int mla_cache_store_fp8(const void* kv_new, const int64_t* slot_mapping, uint8_t* kv_cache, int T, int NB,
                        void* stream) {
  if (T < 0 || NB <= 0) return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d NB=%d", T, NB);
  if (T == 0) return SMLA_OK;
  if (!kv_new || !slot_mapping || !kv_cache) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(kv_new) || !aligned16(kv_cache))
    return fail(SMLA_ERR_INVALID_ARG, "kv_new and kv_cache must be 16-byte aligned");
  cudaError_t e = smla::launch_quantize_store(kv_new, slot_mapping, kv_cache, T, NB, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_cache_store_fp8 launch");
  return SMLA_OK;
}

int mla_cache_store_nvfp4(const void* kv_new, const int64_t* slot_mapping, uint8_t* kv_cache, int T, int NB,
                          void* stream) {
  if (T < 0 || NB <= 0) return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d NB=%d", T, NB);
  if (T == 0) return SMLA_OK;
  if (!kv_new || !slot_mapping || !kv_cache) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(kv_new) || !aligned16(kv_cache))
    return fail(SMLA_ERR_INVALID_ARG, "kv_new and kv_cache must be 16-byte aligned");
  cudaError_t e = smla::launch_nvfp4_store(kv_new, slot_mapping, kv_cache, T, NB, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_cache_store_nvfp4 launch");
  return SMLA_OK;
}

size_t sparse_mla_decode_nvfp4_workspace_bytes(int T, int H, int K, int num_splits) {
  if (T <= 0 || K < 0 || (int64_t)T * K > INT32_MAX) return 0;
  if (check_heads(H) != SMLA_OK) return 0;
  int sms = 0;
  if (num_sms(&sms) != SMLA_OK) return 0;
  if (smla::nvfp4_native_supported(H)) return smla::plan_decode_nvfp4(T, H, K, num_splits, sms).ws_bytes;
  const size_t attn = smla::plan_attention(false, T, H, K, num_splits, sms).ws_bytes;
  return ((attn + 255) / 256) * 256 + smla::nvfp4_stage_bytes(T, K);
}

int sparse_mla_decode_nvfp4(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                            const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                            int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB, int NB,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || K < 0 || R <= 0 || MB <= 0 || NB <= 0 || num_splits < 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d R=%d MB=%d NB=%d num_splits=%d", T, K, R, MB, NB,
                num_splits);
  int rc = check_heads(H);
  if (rc != SMLA_OK) return rc;
  if (T == 0) return SMLA_OK;
  if (!q || !kv_cache || (!indices && K > 0) || !block_table || !req_id_per_token || !out || !lse)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return fail(SMLA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  if ((int64_t)T * K > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "T*K must fit in int32");
  int sms = 0;
  rc = num_sms(&sms);
  if (rc != SMLA_OK) return rc;
  // the bf16 attention's own workspace (its status word leads), then, at 128
  // heads, the staged rows
  const bool native = smla::nvfp4_native_supported(H);
  const smla::AttnPlan plan = native ? smla::plan_decode_nvfp4(T, H, K, num_splits, sms)
                                     : smla::plan_attention(false, T, H, K, num_splits, sms);
  const size_t attn_bytes = ((plan.ws_bytes + 255) / 256) * 256;
  const size_t need = native ? plan.ws_bytes : attn_bytes + smla::nvfp4_stage_bytes(T, K);
  if (workspace) {
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < need) return fail(SMLA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
  } else {
    rc = cached_workspace(need, &workspace);
    if (rc != SMLA_OK) return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (native) {
    // the rows are read as stored and dequantized inside the attention kernel
    smla::AttnArgs a{};
    a.q = q;
    a.cache = kv_cache;
    a.indices = indices;
    a.block_table = block_table;
    a.req_id = req_id_per_token;
    a.out = out;
    a.lse = lse;
    a.sm_scale = sm_scale;
    a.T = T;
    a.H = H;
    a.K = K;
    a.R = R;
    a.MB = MB;
    a.NB = NB;
    a.workspace = workspace;
    cudaError_t e = smla::launch_decode_nvfp4(a, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_decode_nvfp4 launch");
    return SMLA_OK;
  }
  uint8_t* stage = static_cast<uint8_t*>(workspace) + attn_bytes;
  cudaError_t e = smla::launch_nvfp4_stage(kv_cache, NB, indices, block_table, req_id_per_token, T, K, R, MB, stage, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_decode_nvfp4 staging launch");
  const int64_t n = (int64_t)T * K;
  smla::AttnArgs a{};
  a.q = q;
  a.cache = nullptr;
  a.kv = stage + ((n * 4 + 255) / 256) * 256;
  a.indices = reinterpret_cast<const int32_t*>(stage);
  a.out = out;
  a.lse = lse;
  a.sm_scale = sm_scale;
  a.T = T;
  a.H = H;
  a.K = K;
  a.NB = n > 0 ? n : 1;  // rows of the staged buffer
  a.workspace = workspace;
  e = smla::launch_attention(false, a, plan, s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_decode_nvfp4 launch");
  return SMLA_OK;
}

int sparse_mla_translate_indices(const int32_t* indices, const int32_t* block_table,
                                 const int32_t* req_id_per_token, int32_t* slots_out, int T, int K, int R,
                                 int MB, int NB, void* stream) {
  if (T < 0 || K < 0 || R <= 0 || MB <= 0 || NB <= 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d K=%d R=%d MB=%d NB=%d", T, K, R, MB, NB);
  if (T == 0 || K == 0) return SMLA_OK;
  if (!indices || !block_table || !req_id_per_token || !slots_out)
    return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if ((int64_t)NB * 64 > INT32_MAX) return fail(SMLA_ERR_UNSUPPORTED, "NB*64 must fit in int32");
  cudaError_t e = smla::launch_translate(indices, block_table, req_id_per_token, slots_out, T, K, R, MB, NB,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_translate_indices launch");
  return SMLA_OK;
}

int smla_read_device_status(void* workspace, int* status_out, void* stream) {
  if (!status_out) return fail(SMLA_ERR_INVALID_ARG, "null status_out");
  if (!workspace) {
    int dev;
    int rc = current_device(&dev);
    if (rc != SMLA_OK) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    workspace = g_dev[dev].ws;
  }
  if (!workspace) {
    *status_out = 0;
    return SMLA_OK;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if (v != 0) {
    e = cudaMemset(workspace, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  }
  *status_out = v;
  return SMLA_OK;
}

// ---- MLA weight absorption

namespace {
// The status word of a call that takes only a status workspace: the caller's
// (>= 256 bytes, 256-byte aligned) or the library-cached workspace.
int status_workspace(void** workspace, size_t workspace_bytes) {
  if (*workspace) {
    if ((reinterpret_cast<uintptr_t>(*workspace) & 255u) != 0)
      return fail(SMLA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < smla::kWsStatusBytes)
      return fail(SMLA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, smla::kWsStatusBytes);
    return SMLA_OK;
  }
  return cached_workspace(smla::kWsStatusBytes, workspace);
}
}  // namespace

int mla_absorb_q(const void* q, const void* w_uk_t, void* q_out, int T, int H, int P, void* workspace,
                 size_t workspace_bytes, void* stream) {
  if (T < 0 || H <= 0 || P <= 0 || P % 64 != 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d H=%d P=%d (P must be a positive multiple of 64)", T, H, P);
  if (T == 0) return SMLA_OK;
  if (!q || !w_uk_t || !q_out) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(w_uk_t) || !aligned16(q_out))
    return fail(SMLA_ERR_INVALID_ARG, "q, w_uk_t and q_out must be 16-byte aligned");
  int rc = status_workspace(&workspace, workspace_bytes);
  if (rc != SMLA_OK) return rc;
  cudaError_t e = smla::launch_absorb_q(q, w_uk_t, q_out, T, H, P, static_cast<int*>(workspace),
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_absorb_q launch");
  return SMLA_OK;
}

int mla_v_up_proj(const void* attn_out, const void* w_uv, void* out, int T, int H, int V, void* workspace,
                  size_t workspace_bytes, void* stream) {
  if (T < 0 || H <= 0 || V <= 0 || V % 128 != 0)
    return fail(SMLA_ERR_INVALID_ARG, "bad sizes T=%d H=%d V=%d (V must be a positive multiple of 128)", T, H, V);
  if (T == 0) return SMLA_OK;
  if (!attn_out || !w_uv || !out) return fail(SMLA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(attn_out) || !aligned16(w_uv) || !aligned16(out))
    return fail(SMLA_ERR_INVALID_ARG, "attn_out, w_uv and out must be 16-byte aligned");
  int rc = status_workspace(&workspace, workspace_bytes);
  if (rc != SMLA_OK) return rc;
  cudaError_t e = smla::launch_v_up_proj(attn_out, w_uv, out, T, H, V, static_cast<int*>(workspace),
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "mla_v_up_proj launch");
  return SMLA_OK;
}

int smla_read_noalloc_status(int* status_out, void* stream) {
  if (!status_out) return fail(SMLA_ERR_INVALID_ARG, "null status_out");
  void* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc != SMLA_OK) return rc;
  return smla_read_device_status(scratch, status_out, stream);
}

const char* smla_last_error(void) { return g_err; }

int smla_version(void) { return 100; }

}  // extern "C"
