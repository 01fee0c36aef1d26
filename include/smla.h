/*
 * smla.h -- C ABI of the sparse MLA attention library for GB300 (sm_103a).
 *
 * The operations follow vLLM "vllm/v1/attention/backends/mla/flashmla_sparse.py"
 * (cited below as [flashmla_sparse.py]):
 *   - the "FP8 with scale" cache row (module docstring): 656 bytes per token =
 *     512 float8_e4m3 NoPE values, 4 float32 scales (one per 128 values),
 *     64 bfloat16 RoPE values;
 *   - the paged cache [num_blocks, 64, 656] (FlashMLASparseBackend.get_kv_cache_shape);
 *   - triton_convert_req_index_to_global_index (logical top-k index -> slot);
 *   - FlashMLASparseImpl.forward: the cache write through slot_mapping
 *     (concat_and_cache_mla), MQA 576/512 sparse attention with softmax_scale
 *     through flash_mla_with_kvcache (FP8 decode) and flash_mla_sparse_prefill
 *     (BF16 prefill).
 *
 * Conventions for every entry point:
 *   - all tensor arguments are DEVICE pointers owned by the caller, contiguous,
 *     row-major, on the current CUDA device; the library keeps no reference
 *     after the call returns (the work itself is asynchronous on `stream`);
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream);
 *   - calls enqueue work and return without synchronizing the host; they do not
 *     allocate when the caller supplies the workspace;
 *   - bf16 tensors are passed as void* holding IEEE bfloat16 values;
 *   - return value: SMLA_OK, or a negative status; smla_last_error() returns a
 *     thread-local description of the last failure on the calling thread.
 *   - invalid DEVICE data (index -1, a block id out of range, a negative slot)
 *     is never an error: it is masked (attention) or skipped (store).
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMLA_OK 0
#define SMLA_ERR_INVALID_ARG -1   /* null pointer, bad size, misaligned pointer */
#define SMLA_ERR_UNSUPPORTED -2   /* e.g. H not a multiple of 16, or H > 128 */
#define SMLA_ERR_CUDA -3          /* a CUDA call or kernel launch failed */
#define SMLA_ERR_WORKSPACE -4     /* caller workspace smaller than required */

/* Sparse MLA decode over the FP8 paged cache (FP8 path of
 * FlashMLASparseImpl.forward in [flashmla_sparse.py]; indices are translated
 * inside, as triton_convert_req_index_to_global_index does).
 *   q                bf16  [T, H, 576]   query (512 absorbed NoPE + 64 RoPE), 16-byte aligned
 *   kv_cache         uint8 [NB, 64, 656] "FP8 with scale" rows, 16-byte aligned
 *   indices          int32 [T, K]        logical positions within the token's request; <0 = none
 *   block_table      int32 [R, MB]       physical block of each logical block of a request
 *   req_id_per_token int32 [T]           request of each query token
 *   sm_scale         softmax scale applied to q.k
 *   num_splits       0 = automatic work split over all SMs; s > 0 = about s CTAs per (token, head group)
 *   out              bf16  [T, H, 512]   attention output (written)
 *   lse              fp32  [T, H]        natural-log sum of exp of the scaled logits (written);
 *                                        a token with no valid index gets out = 0 and lse = -inf
 *   T, H, K, R, MB, NB  sizes; H must be a multiple of 16 and at most 128
 *   workspace        device scratch of at least sparse_mla_decode_workspace_bytes(T, H, K, num_splits)
 *                    bytes, 256-byte aligned; NULL = a buffer cached by the library per device
 *                    (allocated on first use, so that call is not graph-capturable)
 * A slot is invalid (masked) when the index is negative, its block id is >= MB, the request id is
 * outside [0, R) or the physical block is outside [0, NB).
 * Launch order: for H < 128 the decode kernel is a programmatic dependent of the preceding kernel on
 * `stream`.  If that kernel signals its dependents early (this library's mla_cache_store_fp8 and
 * attention kernels do; ordinary kernels do not), the decode's index translation and Q split may read
 * q, indices, block_table and req_id_per_token before it has finished.  Everything that reads kv_cache
 * or writes out, lse or the workspace waits for it.  So write those four inputs with other kernels,
 * not with a kernel of this library launched directly before the call. */
int sparse_mla_decode_fp8(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                          const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                          int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB, int NB,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes sparse_mla_decode_fp8 (and sparse_mla_decode_fp8_qfp8) needs on the current device. */
size_t sparse_mla_decode_workspace_bytes(int T, int H, int K, int num_splits);

/* sparse_mla_decode_fp8 with the query quantized to FP8 and both products on
 * the FP8 tensor path at every head count: the query-precision variant of
 * [vLLM PR #59342] (its tests quantize the query to fp8 for every quantized
 * cache).  Same arguments, layouts, error codes, workspace and launch order
 * as sparse_mla_decode_fp8.  Each (token, head, 128-column group) of q is
 * scaled by a power of two and split into two e4m3 terms, |q - (hi + lo)| <=
 * 2^-8 |q| + 2^-17 of the group's largest; the cache codes enter QK^T and P.V
 * as stored (tcgen05 kind::f8f6f4), the row scales folded into the logits and
 * into P, which is itself split into two e4m3 terms.  For H < 128 this is
 * what sparse_mla_decode_fp8 computes already, and the call is the same.  For
 * H = 128 it runs a CTA-pair kernel of its own, slower on GB300 than
 * sparse_mla_decode_fp8's (which converts the codes to f16 on chip) and less
 * exact in P (about 8 significant bits against f16's 11). */
int sparse_mla_decode_fp8_qfp8(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                               const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                               int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB, int NB,
                               void* workspace, size_t workspace_bytes, void* stream);

/* sparse_mla_decode_fp8 without any allocation: the same computation and
 * arguments, minus the workspace, whose role a fixed scratch array compiled
 * into the library (SMLA_NOALLOC_SCRATCH_BYTES, 32 MiB of device memory per
 * device the library is loaded on) takes.  The pages have no counterpart of
 * this call: it exists for callers that cannot allocate device memory at
 * call time, e.g. code being captured into a CUDA graph (cudaMalloc is not
 * allowed during stream capture), serving loops that must never block in an
 * allocator (cudaMalloc/cudaFree can synchronize the device), or processes
 * whose memory is already fully handed to a caching allocator.
 *   - No cudaMalloc, cudaFree or other allocating routine is called.
 *   - The first call on a device looks up the scratch array's address
 *     (cudaGetSymbolAddress, which may load the library's device module);
 *     make that first call outside any stream capture.
 *   - A call whose work split needs more than SMLA_NOALLOC_SCRATCH_BYTES of
 *     scratch (sparse_mla_decode_workspace_bytes(T, H, K, num_splits)) is
 *     rejected with SMLA_ERR_WORKSPACE; num_splits = 1, or fewer tokens per
 *     call, needs less.
 *   - Every call shares the one scratch array per device and leaves its
 *     contents behind; a call overwrites everything it reads before reading
 *     it.  Calls whose execution overlaps on the GPU (other streams, other
 *     host threads) race on the scratch and give wrong results: serialize
 *     them, or use sparse_mla_decode_fp8 with one workspace per stream.
 *   - The scratch's device status word records a kernel wait that ran past
 *     its time limit (the kernel still ends); smla_read_noalloc_status reads
 *     and clears it. */
#define SMLA_NOALLOC_SCRATCH_BYTES (32u << 20)
int sparse_mla_decode_fp8_noalloc(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                                  const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                                  int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB,
                                  int NB, void* stream);

/* The NVFP4 cache (the nvfp4_ds_mla dtype of [vLLM PR #59342], "Purpose":
 * 352 bytes per token).  The pages give the size, not the layout; this
 * library's row is
 *   bytes   0..255  the 512 NoPE values as OCP MX FP4 E2M1 codes, value 2i in the
 *                   low nibble of byte i and 2i + 1 in the high nibble;
 *   bytes 256..287  one E4M3 scale per block of 16 NoPE values (byte 256 + b for
 *                   values 16b .. 16b + 15);
 *   bytes 288..351  the 64 RoPE values as E4M3.
 * A row dequantizes alone, exactly in bf16: NoPE c = e2m1(code c) * e4m3(scale
 * c / 16), RoPE r = e4m3(byte 288 + r).  The cache is [NB, 64, 352] uint8,
 * 16-byte aligned, paged through the same block tables as the FP8 cache. */

/* Quantize-and-store into the NVFP4 cache: per block of 16, s = e4m3(amax / 6)
 * and code = e2m1(x / s) (float32 divisions, nearest-even, saturating to 448
 * and 6; a block whose scale is 0 stores code 0); RoPE = e4m3(x).  Arguments
 * as for mla_cache_store_fp8 (a slot < 0 or >= NB * 64 skips the token). */
int mla_cache_store_nvfp4(const void* kv_new, const int64_t* slot_mapping, uint8_t* kv_cache, int T, int NB,
                          void* stream);

/* Sparse MLA decode over the NVFP4 cache: the arguments, masking rules and
 * results of sparse_mla_decode_fp8, kv_cache being [NB, 64, 352]; T * K must
 * fit in int32.  The rows are read as stored and dequantized exactly into
 * bf16: for H < 128 inside the attention kernel (the workspace holds only its
 * status word and split partials); for H = 128 into bf16 rows of the
 * workspace (T * K rows of 1152 bytes), over which the 128-head bf16 kernel
 * runs.  No kernel of this call starts before the preceding work on `stream`
 * has completed. */
int sparse_mla_decode_nvfp4(const void* q, const uint8_t* kv_cache, const int32_t* indices,
                            const int32_t* block_table, const int32_t* req_id_per_token, float sm_scale,
                            int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB, int NB,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes sparse_mla_decode_nvfp4 needs on the current device. */
size_t sparse_mla_decode_nvfp4_workspace_bytes(int T, int H, int K, int num_splits);

/* Sparse MLA prefill over a dense bf16 latent buffer (flash_mla_sparse_prefill
 * as called by FlashMLASparseImpl._bf16_flash_mla_kernel in
 * [flashmla_sparse.py]; heads need no padding here).
 *   q        bf16 [T, H, 576]; kv bf16 [N, 576] (row i = latent row i); indices int32 [T, K] rows of
 *   kv, an index < 0 or >= N is masked; out bf16 [T, H, 512]; lse fp32 [T, H].
 *   num_splits / workspace as for decode (sparse_mla_prefill_workspace_bytes). */
int sparse_mla_prefill_bf16(const void* q, const void* kv, const int32_t* indices, float sm_scale,
                            int num_splits, void* out, float* lse, int T, int H, int N, int K, void* workspace,
                            size_t workspace_bytes, void* stream);

size_t sparse_mla_prefill_workspace_bytes(int T, int H, int K, int num_splits);

/* Separate-mode FP8 prefill of one chunk of prefill requests
 * (FlashMLASparseImpl._forward_fp8_kv_separate_prefill_decode in
 * [flashmla_sparse.py], the path taken for prefill tokens over the FP8 cache):
 *   1. positions 0 .. seq_lens[r] - 1 of each request r of the chunk are
 *      gathered from the cache and up-converted into kv_workspace rows
 *      workspace_starts[r] + p (as sparse_mla_gather_upconvert_fp8);
 *   2. each token's logical top-k indices become kv_workspace rows
 *      workspace_starts[req_id_per_token[t]] + idx (as
 *      sparse_mla_translate_indices_workspace with every token a prefill token);
 *   3. the bf16 sparse prefill (sparse_mla_prefill_bf16) runs over kv_workspace.
 *   q bf16 [T, H, 576]; kv_cache uint8 [NB, 64, 656]; indices int32 [T, K] logical positions within the
 *   token's request (< 0 = none); block_table int32 [R, MB] of the chunk's requests; req_id_per_token int32 [T]
 *   in [0, R); seq_lens, workspace_starts int32 [R] (chunk-local rows, e.g. from sparse_mla_prefill_chunks);
 *   out bf16 [T, H, 512], lse fp32 [T, H] as for sparse_mla_prefill_bf16.
 *   kv_workspace  bf16 [N, 576], caller-owned, 16-byte aligned; rows the chunk does not cover are not read
 *                 unless an index points there (then they are read as they are).
 *   workspace     at least sparse_mla_prefill_fp8_workspace_bytes(T, H, K, num_splits) bytes, 256-byte
 *                 aligned (the prefill's status word and partial results, then the translated indices;
 *                 smla_read_device_status reads it); NULL = library-cached.
 * An index whose block id is outside [0, MB) is masked, as is a row outside [0, N). */
int sparse_mla_prefill_fp8(const void* q, const uint8_t* kv_cache, const int32_t* indices, const int32_t* block_table,
                           const int32_t* req_id_per_token, const int32_t* seq_lens, const int32_t* workspace_starts,
                           float sm_scale, int num_splits, void* out, float* lse, int T, int H, int K, int R, int MB,
                           int NB, void* kv_workspace, int N, void* workspace, size_t workspace_bytes, void* stream);

size_t sparse_mla_prefill_fp8_workspace_bytes(int T, int H, int K, int num_splits);

/* Gather and up-convert of the FP8 prefill (ops.cp_gather_and_upconvert_fp8_kv_cache as called by
 * _forward_fp8_kv_separate_prefill_decode in [flashmla_sparse.py]): for each request r < R and position
 * p < seq_lens[r], the cache row at block_table[r, p // 64] * 64 + p % 64 becomes bf16 row
 * workspace_starts[r] + p of kv_workspace [N, 576]: value c < 512 is the float32 product
 * e4m3(code c) * scale[c / 128] rounded to bf16 (nearest, ties to even), the 64 RoPE values are copied.
 * A position whose physical block is outside [0, NB) gives a zero row; a destination row outside
 * [0, N) is not written.  seq_lens, workspace_starts int32 [R] device arrays. */
int sparse_mla_gather_upconvert_fp8(const uint8_t* kv_cache, const int32_t* block_table, const int32_t* seq_lens,
                                    const int32_t* workspace_starts, int R, int MB, int NB, void* kv_workspace, int N,
                                    void* stream);

/* Index translation with a prefill workspace (triton_convert_req_index_to_global_index with
 * HAS_PREFILL_WORKSPACE in [flashmla_sparse.py]): for a token with prefill_request_id[t] < 0 (a
 * decode token) out = the cache slot of sparse_mla_translate_indices; for a prefill token
 * out = workspace_starts[prefill_request_id[t]] + idx; -1 when idx < 0, idx // 64 >= MB, or
 * prefill_request_id[t] >= P.  prefill_request_id int32 [T]; workspace_starts int32 [P]; out int32 [T, K]. */
int sparse_mla_translate_indices_workspace(const int32_t* indices, const int32_t* block_table,
                                           const int32_t* req_id_per_token, const int32_t* prefill_request_id,
                                           const int32_t* workspace_starts, int P, int32_t* out, int T, int K, int R,
                                           int MB, int NB, void* stream);

/* Host-side chunking of prefill requests into workspaces of workspace_rows rows (split_prefill_chunks
 * and the per-chunk workspace starts of FlashMLASparseMetadataBuilder in [flashmla_sparse.py]): requests
 * are taken in order and a chunk is closed before the request that would overflow it.  HOST arrays:
 * seq_lens [R] in; chunk_ends [R] out (exclusive end request of each chunk, *n_chunks of them);
 * workspace_starts [R] out (chunk-local first row of each request).  SMLA_ERR_WORKSPACE if one
 * request alone exceeds workspace_rows.  No device work. */
int sparse_mla_prefill_chunks(const int32_t* seq_lens, int R, int64_t workspace_rows, int32_t* chunk_ends,
                              int32_t* workspace_starts, int* n_chunks);

/* Work split of one attention call on the current device, for callers that
 * count kernel launches or size grids (no work is done):
 *   fp8      nonzero for sparse_mla_decode_fp8, zero for sparse_mla_prefill_bf16
 *   T, H, K, num_splits as for those calls
 *   launches out: kernels the call launches (the attention kernel, plus the
 *            LSE combine when a unit is split across CTAs, plus the Q
 *            preparation of the 128-head FP8 decode)
 *   ctas     out: CTAs of the attention kernel's grid
 * Returns SMLA_OK, or SMLA_ERR_INVALID_ARG / SMLA_ERR_UNSUPPORTED for sizes
 * the call itself would reject, or SMLA_ERR_CUDA without a device. */
int sparse_mla_attention_plan(int fp8, int T, int H, int K, int num_splits, int* launches, int* ctas);

/* Quantize-and-store of new tokens into the FP8 cache (cache write of
 * FlashMLASparseImpl.forward, concat_and_cache_mla with "fp8_ds_mla", in
 * [flashmla_sparse.py]).
 *   kv_new       bf16 [T, 576]: 512 latent (NoPE) values followed by 64 RoPE values, 16-byte aligned
 *   slot_mapping int64 [T]: destination row (block * 64 + offset); < 0 or >= NB*64 skips the token
 *   kv_cache     uint8 [NB, 64, 656], 16-byte aligned
 * Per group of 128 NoPE values: scale = amax / 448 in IEEE float32, code = the float32 quotient
 * value / scale rounded to nearest-even e4m3 with saturation (a group with scale 0 stores zeros);
 * the 4 scales and the RoPE values are stored verbatim.  Two tokens with the same slot race.
 * Launch order: the kernel is a programmatic dependent of the preceding kernel on `stream` (its
 * launch may overlap that kernel's tail).  It writes kv_cache only after that kernel has
 * completed, so a decode running before it still reads the old rows.  If that kernel signals its
 * dependents early (this library's decode and attention kernels do; ordinary kernels do not),
 * kv_new and slot_mapping may be read before it has finished: write those two with other kernels,
 * not with a kernel of this library launched directly before the call. */
int mla_cache_store_fp8(const void* kv_new, const int64_t* slot_mapping, uint8_t* kv_cache, int T, int NB,
                        void* stream);

/* Logical -> physical slot translation on its own (the step the decode
 * kernel fuses), as triton_convert_req_index_to_global_index in
 * [flashmla_sparse.py]: slots_out[t, k] = block_table[req[t], idx // 64] * 64 + idx % 64, or -1
 * under the invalid conditions listed for sparse_mla_decode_fp8.  slots_out int32 [T, K]. */
int sparse_mla_translate_indices(const int32_t* indices, const int32_t* block_table,
                                 const int32_t* req_id_per_token, int32_t* slots_out, int T, int K, int R,
                                 int MB, int NB, void* stream);

/* MLA weight absorption before the attention (FlashMLASparseImpl.forward in [flashmla_sparse.py]: q is
 * split into q_nope and q_pe, ql_nope = bmm(q_nope, W_UK_T) per head, and the attention input is
 * cat(ql_nope, q_pe)), as one tensor-core kernel whose epilogue writes the attention-ready query:
 *   q       bf16 [T, H, P + 64]   P NoPE features (a positive multiple of 64) then 64 RoPE features
 *   w_uk_t  bf16 [H, P, 512]      per head, row p = the 512 latent weights of NoPE feature p
 *   q_out   bf16 [T, H, 576]      q_out[t, h, 0:512] = q[t, h, 0:P] x w_uk_t[h] (fp32 accumulation, rounded
 *                                 to bf16), q_out[t, h, 512:576] = q[t, h, P:P+64]
 *   workspace  >= 256 bytes, 256-byte aligned (the status word); NULL = library-cached. */
int mla_absorb_q(const void* q, const void* w_uk_t, void* q_out, int T, int H, int P, void* workspace,
                 size_t workspace_bytes, void* stream);

/* MLA value up-projection after the attention (FlashMLASparseImpl._v_up_proj in [flashmla_sparse.py]):
 *   attn_out bf16 [T, H, 512]; w_uv bf16 [H, 512, V] (V a positive multiple of 128);
 *   out bf16 [T, H, V] = attn_out[t, h, :] x w_uv[h] per head (fp32 accumulation, rounded to bf16).
 *   workspace as for mla_absorb_q. */
int mla_v_up_proj(const void* attn_out, const void* w_uv, void* out, int T, int H, int V, void* workspace,
                  size_t workspace_bytes, void* stream);

/* Reads (and clears) the device status word of a workspace after
 * synchronizing `stream`: 0 = no fault; 1 = a kernel wait ran past its time
 * limit and the kernel unwound (its outputs are not valid).  workspace NULL =
 * the library-cached workspace of the current device. */
int smla_read_device_status(void* workspace, int* status_out, void* stream);

/* smla_read_device_status for the fixed scratch of
 * sparse_mla_decode_fp8_noalloc on the current device: synchronizes
 * `stream`, then reads and clears the status word (0 = no fault; 1 = a kernel
 * wait ran past its time limit and the kernel unwound, so the outputs of the
 * calls since the last read are not valid). */
int smla_read_noalloc_status(int* status_out, void* stream);

/* Thread-local description of the last failing call on this thread. */
const char* smla_last_error(void);

/* Library ABI version (major * 100 + minor). */
int smla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H_ */
