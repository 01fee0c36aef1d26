/*
 * smla_oracle.c -- plain, slow, float64 CPU reference for sparse MLA attention
 * over the 656-byte "FP8 with scale" paged cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test-suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library; the two meet only through the seeded synthetic inputs.
 *
 * Sources (the pages this follows):
 *  [P2] vLLM, "vllm/v1/attention/backends/mla/flashmla_sparse.py":
 *       - module docstring, "FP8 with scale" format (656 bytes per token:
 *         512 float8_e4m3 NoPE values, 4 float32 scales one per 128 values,
 *         64 bfloat16 RoPE values, not quantized);
 *       - triton_convert_req_index_to_global_index, its docstring formula
 *         out = block_table[req, idx // BLOCK_SIZE] * BLOCK_SIZE + idx % BLOCK_SIZE,
 *         -1 for idx == -1 or an out-of-range block id;
 *       - FlashMLASparseImpl.forward: MQA 576/512 (head_dim_v = 512),
 *         softmax_scale, the write of k_c_normed (512) and k_pe (64) into the
 *         cache through slot_mapping (concat_and_cache_mla).
 *  [OCP] OCP 8-bit floating point specification, E4M3: 1 sign, 4 exponent
 *        (bias 7), 3 mantissa bits; subnormals; no infinities; S.1111.111 NaN.
 *  [OCP-MX] OCP Microscaling Formats (MX) specification, FP4 E2M1 element:
 *        1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
 *        0, 0.5, 1, 1.5, 2, 3, 4, 6; no infinities or NaN.
 *  [P3] vLLM PR #59342, "Purpose": the nvfp4_ds_mla cache holds 352 bytes
 *        per token against the FP8 one's 576; the native decode reads the
 *        rows as stored and sees the exact dequantized values.
 *
 * Readings where the pages are silent:
 *  R1 translate also rejects a physical block id outside [0, NB) and a request
 *     id outside [0, R) (the page would emit a slot from garbage);
 *  R2 the quantizer scale is amax/448 in float32, codes are the float32
 *     quotient x/scale rounded to nearest-even e4m3, saturating to +-448; a
 *     group whose scale is 0 stores code 0 everywhere and scale 0.0f;
 *  R3 V is the NoPE part, columns 0..511 of the 576-wide latent row;
 *  R4 LSE is the natural log of the sum of exp of the scaled logits; a token
 *     with no valid index has output 0 and LSE -infinity;
 *  R5 slot_mapping < 0 (or >= NB*64) skips the token;
 *  R9 separate-mode FP8 prefill: a row is up-converted to bf16 from the float32
 *     product code * scale (ties to even), an invalid slot gives a zero row,
 *     and a prefill request id outside [0, P) gives -1.
 *  R13 the NVFP4 row (the pages give its size, 352 bytes, not its layout):
 *     bytes 0..255 the 512 NoPE values as E2M1 codes, value 2i in the low
 *     nibble of byte i and 2i + 1 in the high nibble; bytes 256..287 one E4M3
 *     scale per block of 16 values (byte 256 + b for values 16b .. 16b + 15);
 *     bytes 288..351 the 64 RoPE values as E4M3.  No per-tensor scale: a row
 *     dequantizes alone.  Quantizer: block scale = e4m3(amax / 6) (float32
 *     division, nearest-even, saturating); code = e2m1(x / s) with s the
 *     scale's value (float32 division, nearest-even, saturating to 6); a
 *     block whose scale is 0 stores code 0; RoPE = e4m3(value).
 *
 * Every floating-point step of attention is in double.  The quantizer decides
 * integer codes, so it runs in float32, the precision the CUDA kernel uses.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ROW_BYTES 656
#define NVFP4_ROW_BYTES 352
#define NVFP4_BLOCK 16
#define D_QK 576
#define D_V 512
#define D_NOPE 512
#define GROUP 128
#define BLOCK 64

/* ---------------------------------------------------------------- formats */

/* [OCP] E4M3 decode: value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
 * (-1)^s * 2^-6 * (m/8) for e == 0; e == 15 && m == 7 is NaN. */
double oracle_e4m3_to_double(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* [OCP] encode a float to E4M3 with round-to-nearest, ties to even, and
 * saturation to the largest finite magnitude (448).  Written from the format:
 * find the exponent bucket, scale the magnitude to an integer grid of 8 steps
 * per binade (or per 2^-9 in the subnormal range) and round on that grid. */
uint8_t oracle_e4m3_from_float(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid: multiples of 2^-9, mantissa 0..8 (8 == smallest normal) */
    double q = nearbyint(a * 512.0); /* default rounding mode: ties to even */
    int m = (int)q;
    if (m >= 8) return sign | 0x08;
    return sign | (uint8_t)m;
  }
  int ex;
  double fr = frexp(a, &ex); /* a = fr * 2^ex, fr in [0.5, 1) */
  int e = ex - 1;            /* a = (2*fr) * 2^e, 2*fr in [1, 2) */
  double q = nearbyint(fr * 2.0 * 8.0); /* 8..16 */
  int m8 = (int)q;
  if (m8 == 16) {
    m8 = 8;
    e += 1;
  }
  int biased = e + 7;
  if (biased > 15 || (biased == 15 && m8 - 8 == 7)) return sign | 0x7E; /* saturate */
  return sign | (uint8_t)((biased << 3) | (m8 - 8));
}

/* [OCP-MX] E2M1 decode: value = (-1)^s * 2^(e-1) * (1 + m/2) for e > 0,
 * (-1)^s * m/2 for e == 0 (code bits: s e1 e0 m). */
double oracle_e2m1_to_double(uint8_t code) {
  int s = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double v = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
  return s ? -v : v;
}

/* [OCP-MX] encode a float to E2M1, round to nearest with ties to even and
 * saturation to 6 (reading R13).  Each binade of the format is an evenly
 * spaced grid: [0, 2) in steps of 1/2 (codes 0..4, the subnormal 0.5 and the
 * binade [1, 2)), [2, 4) in steps of 1 (codes 4..6), [4, 6] in steps of 2
 * (codes 6, 7); every grid starts at an even code, so ties to an even grid
 * index are ties to an even code. */
uint8_t oracle_e2m1_from_float(float y) {
  if (isnan(y)) return 0;
  uint8_t sign = signbit(y) ? 0x8 : 0x0;
  double a = fabs((double)y);
  if (a >= 6.0) return sign | 0x7;
  double base = 0.0, step = 0.5;
  int code0 = 0;
  if (a >= 4.0) {
    base = 4.0;
    step = 2.0;
    code0 = 6;
  } else if (a >= 2.0) {
    base = 2.0;
    step = 1.0;
    code0 = 4;
  }
  int k = (int)nearbyint((a - base) / step); /* default rounding mode: ties to even */
  return sign | (uint8_t)(code0 + k);
}

double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float bf16_to_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* [P2 docstring] Dequantize one 656-byte row as stored:
 * K[c] = e4m3(byte c) * scale[c / 128] for c < 512 (scales are little-endian
 * float32 at bytes 512 + 4g); K[512 + r] = bf16 at bytes 528 + 2r. */
void oracle_dequant_row(const uint8_t* row, double* out) {
  for (int c = 0; c < D_NOPE; ++c) {
    float sc;
    memcpy(&sc, row + D_NOPE + 4 * (c / GROUP), 4);
    out[c] = oracle_e4m3_to_double(row[c]) * (double)sc;
  }
  for (int r = 0; r < D_QK - D_NOPE; ++r) {
    uint16_t b;
    memcpy(&b, row + D_NOPE + 16 + 2 * r, 2);
    out[D_NOPE + r] = oracle_bf16_to_double(b);
  }
}

/* Reading R13: one 352-byte NVFP4 row as stored: K[c] = e2m1(nibble c) *
 * e4m3(byte 256 + c / 16) for c < 512, K[512 + r] = e4m3(byte 288 + r). */
void oracle_nvfp4_dequant_row(const uint8_t* row, double* out) {
  for (int c = 0; c < D_NOPE; ++c) {
    uint8_t code = (uint8_t)((row[c / 2] >> (4 * (c & 1))) & 0xF);
    out[c] = oracle_e2m1_to_double(code) * oracle_e4m3_to_double(row[D_NOPE / 2 + c / NVFP4_BLOCK]);
  }
  for (int r = 0; r < D_QK - D_NOPE; ++r)
    out[D_NOPE + r] = oracle_e4m3_to_double(row[D_NOPE / 2 + D_NOPE / NVFP4_BLOCK + r]);
}

/* ---------------------------------------------------------------- translate */

/* [P2 triton_convert_req_index_to_global_index] plus reading R1. */
int32_t oracle_translate_one(int32_t idx, int32_t req, const int32_t* block_table, int R, int MB, int64_t NB) {
  if (idx < 0) return -1;
  if (req < 0 || req >= R) return -1;
  int32_t b = idx / BLOCK;
  int32_t o = idx % BLOCK;
  if (b >= MB) return -1;
  int32_t p = block_table[(int64_t)req * MB + b];
  if (p < 0 || (int64_t)p >= NB) return -1;
  return p * BLOCK + o;
}

void oracle_translate(const int32_t* indices, const int32_t* block_table, const int32_t* req_id, int T, int K, int R,
                      int MB, int64_t NB, int32_t* slots) {
  for (int t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k)
      slots[(int64_t)t * K + k] =
          oracle_translate_one(indices[(int64_t)t * K + k], req_id[t], block_table, R, MB, NB);
}

/* ---------------------------------------------------------------- quantize */

/* [P2 forward / concat_and_cache_mla] + reading R2: write each new token's
 * latent (512 NoPE, quantized per 128-group) and RoPE (64 bf16, copied) into
 * its cache row at slot_mapping[t]. */
void oracle_quantize_store(const uint16_t* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T, int64_t NB) {
  for (int t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= NB * BLOCK) continue;
    const uint16_t* x = kv_new + (int64_t)t * D_QK;
    uint8_t* row = cache + slot * ROW_BYTES;
    for (int g = 0; g < D_NOPE / GROUP; ++g) {
      float amax = 0.0f;
      for (int c = g * GROUP; c < (g + 1) * GROUP; ++c) {
        float v = fabsf(bf16_to_float(x[c]));
        if (v > amax) amax = v;
      }
      float scale = amax / 448.0f;
      for (int c = g * GROUP; c < (g + 1) * GROUP; ++c) {
        if (scale == 0.0f) {
          row[c] = 0;
        } else {
          float y = bf16_to_float(x[c]) / scale;
          row[c] = oracle_e4m3_from_float(y);
        }
      }
      memcpy(row + D_NOPE + 4 * g, &scale, 4);
    }
    memcpy(row + D_NOPE + 16, x + D_NOPE, 2 * (D_QK - D_NOPE));
  }
}

/* [P3 "Purpose": nvfp4_ds_mla, 352 bytes per token] + reading R13: write each
 * new token's latent into its NVFP4 cache row at slot_mapping[t] (the skip
 * rule R5 as for the FP8 cache). */
void oracle_nvfp4_quantize_store(const uint16_t* kv_new, const int64_t* slot_mapping, uint8_t* cache, int T,
                                 int64_t NB) {
  for (int t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= NB * BLOCK) continue;
    const uint16_t* x = kv_new + (int64_t)t * D_QK;
    uint8_t* row = cache + slot * NVFP4_ROW_BYTES;
    memset(row, 0, D_NOPE / 2);
    for (int b = 0; b < D_NOPE / NVFP4_BLOCK; ++b) {
      float amax = 0.0f;
      for (int c = b * NVFP4_BLOCK; c < (b + 1) * NVFP4_BLOCK; ++c) {
        float v = fabsf(bf16_to_float(x[c]));
        if (v > amax) amax = v;
      }
      uint8_t sb = oracle_e4m3_from_float(amax / 6.0f);
      float s = (float)oracle_e4m3_to_double(sb);
      row[D_NOPE / 2 + b] = sb;
      for (int c = b * NVFP4_BLOCK; c < (b + 1) * NVFP4_BLOCK; ++c) {
        uint8_t code = s == 0.0f ? 0 : oracle_e2m1_from_float(bf16_to_float(x[c]) / s);
        row[c / 2] |= (uint8_t)(code << (4 * (c & 1)));
      }
    }
    for (int r = 0; r < D_QK - D_NOPE; ++r)
      row[D_NOPE / 2 + D_NOPE / NVFP4_BLOCK + r] = oracle_e4m3_from_float(bf16_to_float(x[D_NOPE + r]));
  }
}

/* ---------------------------------------------------------------- attention */

/* Attention of one query head over n dequantized rows (n x 576), [P2]
 * MQA 576/512 with softmax_scale, and readings R3, R4. */
static void attend_head(const double* qh, const double* rows, int n, double sm_scale, double* s_buf, double* out,
                        double* lse) {
  if (n == 0) {
    for (int c = 0; c < D_V; ++c) out[c] = 0.0;
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int c = 0; c < D_QK; ++c) acc += qh[c] * rows[(int64_t)j * D_QK + c];
    s_buf[j] = sm_scale * acc;
    if (s_buf[j] > m) m = s_buf[j];
  }
  double l = 0.0;
  for (int c = 0; c < D_V; ++c) out[c] = 0.0;
  for (int j = 0; j < n; ++j) {
    double w = exp(s_buf[j] - m);
    l += w;
    for (int c = 0; c < D_V; ++c) out[c] += w * rows[(int64_t)j * D_QK + c];
  }
  for (int c = 0; c < D_V; ++c) out[c] /= l;
  *lse = m + log(l);
}

/* FP8 sparse decode.  For each requested token (tokens[i], or i when tokens is
 * NULL): translate its K logical indices, dequantize every valid row as
 * stored, and attend with each of its H heads.
 * q: bf16 bits [T, H, 576]; cache: [NB, 64, 656] bytes; out: [n, H, 512];
 * lse: [n, H].  Workspace is allocated by the caller: rows [K * 576] and
 * s [K] doubles per thread (nthreads copies). */
static void decode_rows(const uint16_t* q, const uint8_t* cache, int row_bytes,
                        void (*dequant)(const uint8_t*, double*), const int32_t* indices,
                        const int32_t* block_table, const int32_t* req_id, double sm_scale, int H, int K, int R,
                        int MB, int64_t NB, const int32_t* tokens, int n_tokens, double* ws_rows, double* ws_s,
                        int nthreads, double* out, double* lse);

void oracle_sparse_mla_decode(const uint16_t* q, const uint8_t* cache, const int32_t* indices,
                              const int32_t* block_table, const int32_t* req_id, double sm_scale, int T, int H, int K,
                              int R, int MB, int64_t NB, const int32_t* tokens, int n_tokens, double* ws_rows,
                              double* ws_s, int nthreads, double* out, double* lse) {
  (void)T;
  decode_rows(q, cache, ROW_BYTES, oracle_dequant_row, indices, block_table, req_id, sm_scale, H, K, R, MB, NB,
              tokens, n_tokens, ws_rows, ws_s, nthreads, out, lse);
}

/* The same decode over the NVFP4 cache [NB, 64, 352] (reading R13): rows
 * dequantized as stored, then the same attention. */
void oracle_sparse_mla_decode_nvfp4(const uint16_t* q, const uint8_t* cache, const int32_t* indices,
                                    const int32_t* block_table, const int32_t* req_id, double sm_scale, int T, int H,
                                    int K, int R, int MB, int64_t NB, const int32_t* tokens, int n_tokens,
                                    double* ws_rows, double* ws_s, int nthreads, double* out, double* lse) {
  (void)T;
  decode_rows(q, cache, NVFP4_ROW_BYTES, oracle_nvfp4_dequant_row, indices, block_table, req_id, sm_scale, H, K, R,
              MB, NB, tokens, n_tokens, ws_rows, ws_s, nthreads, out, lse);
}

static void decode_rows(const uint16_t* q, const uint8_t* cache, int row_bytes,
                        void (*dequant)(const uint8_t*, double*), const int32_t* indices,
                        const int32_t* block_table, const int32_t* req_id, double sm_scale, int H, int K, int R,
                        int MB, int64_t NB, const int32_t* tokens, int n_tokens, double* ws_rows, double* ws_s,
                        int nthreads, double* out, double* lse) {
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int i = 0; i < n_tokens; ++i) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double* rows = ws_rows + (int64_t)tid * K * D_QK;
    double* s_buf = ws_s + (int64_t)tid * K;
    double qh[D_QK];
    int t = tokens ? tokens[i] : i;
    int n = 0;
    for (int k = 0; k < K; ++k) {
      int32_t slot = oracle_translate_one(indices[(int64_t)t * K + k], req_id[t], block_table, R, MB, NB);
      if (slot < 0) continue;
      dequant(cache + (int64_t)slot * row_bytes, rows + (int64_t)n * D_QK);
      ++n;
    }
    for (int h = 0; h < H; ++h) {
      for (int c = 0; c < D_QK; ++c) qh[c] = oracle_bf16_to_double(q[((int64_t)t * H + h) * D_QK + c]);
      attend_head(qh, rows, n, sm_scale, s_buf, out + ((int64_t)i * H + h) * D_V, lse + (int64_t)i * H + h);
    }
  }
}

/* BF16 sparse prefill over a dense latent buffer kv [N, 576]: index i is a row
 * of kv; i < 0 or i >= N is invalid (the prefill analogue of R1). */
void oracle_sparse_mla_prefill(const uint16_t* q, const uint16_t* kv, const int32_t* indices, double sm_scale, int T,
                               int H, int64_t N, int K, const int32_t* tokens, int n_tokens, double* ws_rows,
                               double* ws_s, int nthreads, double* out, double* lse) {
  (void)T;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int i = 0; i < n_tokens; ++i) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    double* rows = ws_rows + (int64_t)tid * K * D_QK;
    double* s_buf = ws_s + (int64_t)tid * K;
    double qh[D_QK];
    int t = tokens ? tokens[i] : i;
    int n = 0;
    for (int k = 0; k < K; ++k) {
      int32_t idx = indices[(int64_t)t * K + k];
      if (idx < 0 || (int64_t)idx >= N) continue;
      for (int c = 0; c < D_QK; ++c) rows[(int64_t)n * D_QK + c] = oracle_bf16_to_double(kv[(int64_t)idx * D_QK + c]);
      ++n;
    }
    for (int h = 0; h < H; ++h) {
      for (int c = 0; c < D_QK; ++c) qh[c] = oracle_bf16_to_double(q[((int64_t)t * H + h) * D_QK + c]);
      attend_head(qh, rows, n, sm_scale, s_buf, out + ((int64_t)i * H + h) * D_V, lse + (int64_t)i * H + h);
    }
  }
}

/* ---------------------------------------------------------------- separate-mode FP8 prefill */

/* float32 -> bfloat16 bits, round to nearest, ties to even (finite inputs;
 * an infinity or NaN keeps its class). */
static uint16_t float_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* [P2 _forward_fp8_kv_separate_prefill_decode: cp_gather_and_upconvert_fp8_kv_cache]
 * + reading R9: one cache row up-converted for the bf16 prefill kernel.  NoPE
 * value c is e4m3(byte c) * scale[c / 128] formed in float32 (the precision
 * of the stored scales; the e4m3 value is exact in float32) and rounded to
 * bf16, nearest with ties to even; the 64 RoPE values are copied as stored. */
void oracle_upconvert_row(const uint8_t* row, uint16_t* out) {
  for (int c = 0; c < D_NOPE; ++c) {
    float sc;
    memcpy(&sc, row + D_NOPE + 4 * (c / GROUP), 4);
    const float v = (float)oracle_e4m3_to_double(row[c]);
    const float prod = v * sc;
    out[c] = float_to_bf16_rne(prod);
  }
  memcpy(out + D_NOPE, row + D_NOPE + 16, 2 * (D_QK - D_NOPE));
}

/* [P2 cp_gather_and_upconvert_fp8_kv_cache(cache, workspace, block_table,
 * seq_lens, workspace_starts, num_reqs)]: positions 0 .. seq_lens[r] - 1 of
 * request r, in order, become workspace rows starts[r] .. starts[r] +
 * seq_lens[r] - 1.  A position whose slot is invalid under R1 gives a row of
 * zeros (reading R9); a destination outside [0, N) is not written. */
void oracle_gather_upconvert(const uint8_t* cache, int64_t NB, const int32_t* block_table, int R, int MB,
                             const int32_t* seq_lens, const int32_t* starts, uint16_t* ws, int64_t N) {
  for (int r = 0; r < R; ++r) {
    for (int32_t pos = 0; pos < seq_lens[r]; ++pos) {
      const int64_t dst = (int64_t)starts[r] + pos;
      if (dst < 0 || dst >= N) continue;
      const int32_t slot = oracle_translate_one(pos, r, block_table, R, MB, NB);
      if (slot < 0)
        memset(ws + dst * D_QK, 0, 2 * D_QK);
      else
        oracle_upconvert_row(cache + (int64_t)slot * ROW_BYTES, ws + dst * D_QK);
    }
  }
}

/* [P2 _convert_req_index_to_global_index_kernel with HAS_PREFILL and its
 * docstring]: a decode token (prefill_req_id < 0) is translated as above; a
 * prefill token's index becomes workspace_starts[prefill_req_id] + index,
 * -1 when the index is negative or its block id is outside [0, MB) (the
 * kernel's own guard), or (reading R9) when prefill_req_id >= P. */
void oracle_translate_workspace(const int32_t* indices, const int32_t* block_table, const int32_t* req_id,
                                const int32_t* prefill_req_id, const int32_t* starts, int T, int K, int R, int MB,
                                int64_t NB, int P, int32_t* out) {
  for (int t = 0; t < T; ++t) {
    const int32_t pr = prefill_req_id[t];
    for (int k = 0; k < K; ++k) {
      const int32_t idx = indices[(int64_t)t * K + k];
      int32_t v;
      if (pr < 0) {
        v = oracle_translate_one(idx, req_id[t], block_table, R, MB, NB);
      } else if (idx < 0 || idx / BLOCK >= MB || pr >= P) {
        v = -1;
      } else {
        v = starts[pr] + idx;
      }
      out[(int64_t)t * K + k] = v;
    }
  }
}
