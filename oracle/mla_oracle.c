/*
 * Plain CPU oracle for MLA decode over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * statement of what the GPU path computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or helper with the CUDA library, and it never imports it.
 *
 * Sources (web pages; cited by page title and section):
 *   [diff]  "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs" ("fix TP"),
 *           a unified diff of vLLM; cited by the file section it falls in.
 *   [note]  "Triton and MLA: portable attention and multi-head latent
 *           attention" (vLLM v0.25.1 architecture note), cited by section.
 *   [api]   "vllm.v1.attention.backends.mla.triton_mla" API reference page,
 *           TritonMLAMetadataBuilder.
 *   [OCP]   OCP 8-bit Floating Point Specification (OFP8), E4M3 format:
 *           bias 7, no infinities, NaN = S.1111.111, max normal 448,
 *           min normal 2^-6, min subnormal 2^-9; E5M2 format: bias 15,
 *           IEEE-like infinities (S.11111.00) and NaNs (S.11111.{01,10,11}),
 *           max normal 57344, min normal 2^-14, min subnormal 2^-16.
 *
 * All floating-point work is fp64 except the one place where the pages fix
 * fp32: the fp8 quantisation step divides the fp32 input by the fp32 scale
 * in IEEE single precision before rounding to E4M3.
 *
 * Compiled with -ffp-contract=off so that x86-64 and aarch64 produce the same
 * bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Scalar codecs                                                        */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> its exact value.  bf16 is the upper half of an IEEE
 * binary32, so the value is the float with those 16 bits on top. */
double oracle_bf16_value(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* E4M3 (OCP "e4m3fn") code -> exact value, from the format definition [OCP]:
 *   S.EEEE.MMM, bias 7; E == 0 is subnormal m * 2^-9; S.1111.111 is NaN. */
double oracle_e4m3_value(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* fp32 value -> E4M3 code, round to nearest with ties to even, saturating
 * finite overflow (and infinities) to +-448, NaN -> the positive NaN code.
 *
 * Written as a nearest-value search over the 127 non-negative finite codes,
 * whose values increase with the code: find the largest code whose value is
 * <= |y|, then pick between it and the next code by distance, ties going to
 * the code with an even mantissa (its low bit clear). */
uint8_t oracle_e4m3_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E; /* saturate (covers +-inf) */
  int lo = 0, hi = 0x7E;              /* v(lo) <= a < v(hi) holds after loop */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e4m3_value((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double dlo = a - oracle_e4m3_value((uint8_t)lo);
  double dhi = oracle_e4m3_value((uint8_t)hi) - a;
  int code;
  if (dlo < dhi)
    code = lo;
  else if (dhi < dlo)
    code = hi;
  else
    code = (lo & 1) ? hi : lo;
  return sign | (uint8_t)code;
}

/* E5M2 code -> exact value, from the format definition [OCP]:
 *   S.EEEEE.MM, bias 15; E == 0 is subnormal m * 2^-16; E == 31 is
 *   infinity (M == 0) or NaN. */
double oracle_e5m2_value(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 2) & 31;
  int m = code & 3;
  double v;
  if (e == 31) {
    if (m != 0) return NAN;
    v = INFINITY;
  } else if (e == 0) {
    v = ldexp((double)m, -16);
  } else {
    v = ldexp(1.0 + m / 4.0, e - 15);
  }
  return s ? -v : v;
}

/* fp32 value -> E5M2 code, round to nearest with ties to even, finite
 * overflow and infinities saturated to +-57344 (the "satfinite" reading, as
 * for E4M3), NaN -> the positive NaN code 0x7F.  Same nearest-value search
 * as oracle_e4m3_encode, over the 124 non-negative finite codes. */
uint8_t oracle_e5m2_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 57344.0) return sign | 0x7B;
  int lo = 0, hi = 0x7B;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e5m2_value((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid;
  }
  double dlo = a - oracle_e5m2_value((uint8_t)lo);
  double dhi = oracle_e5m2_value((uint8_t)hi) - a;
  int code;
  if (dlo < dhi)
    code = lo;
  else if (dhi < dlo)
    code = hi;
  else
    code = (lo & 1) ? hi : lo;
  return sign | (uint8_t)code;
}

/* ------------------------------------------------------------------ */
/* Cache write: [diff] csrc/cache_kernels.cu, concat_and_cache_mla_kernel */
/* and its host wrapper concat_and_cache_mla.                             */
/* ------------------------------------------------------------------ */

/* For every token t < num_tokens in order: slot = slot_mapping[t];
 * slot < 0 is a padded token and is skipped; otherwise block = slot / bs,
 * offset = slot % bs, and row `offset` of block `block` receives
 * kv_c[t, 0:R] in elements [0, R) and k_pe[t, 0:P] in [R, R+P).
 * Elements are stored as bf16 bits unchanged, or (fp8 cache) as
 * E4M3(x / scale) with x / scale an IEEE fp32 division (the "divide on
 * store" reading of scaled_convert, whose body the pages do not print).
 * A slot >= num_blocks * bs is skipped and counted (the pages leave it
 * unchecked).  Returns the number of such skipped slots. */
int64_t oracle_cache_write(const uint16_t *kv_c, int64_t kv_c_row_stride,
                           const uint16_t *k_pe, int64_t k_pe_row_stride,
                           const int64_t *slot_mapping, int64_t num_tokens,
                           int kv_lora_rank, int rope_dim, void *kv_cache,
                           int64_t num_blocks, int block_size,
                           int64_t block_stride, int kv_is_fp8, float scale) {
  const int R = kv_lora_rank, P = rope_dim, D = R + P;
  int64_t bad = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * (int64_t)block_size) {
      ++bad;
      continue;
    }
    int64_t blk = slot / block_size;
    int64_t off = slot % block_size;
    int64_t row = blk * block_stride + off * D; /* element index of row */
    for (int i = 0; i < D; ++i) {
      uint16_t x = (i < R) ? kv_c[t * kv_c_row_stride + i]
                           : k_pe[t * k_pe_row_stride + (i - R)];
      if (kv_is_fp8) {
        float xf = (float)oracle_bf16_value(x);
        float yq = xf / scale; /* IEEE binary32 division */
        ((uint8_t *)kv_cache)[row + i] =
            kv_is_fp8 == 2 ? oracle_e5m2_encode(yq) : oracle_e4m3_encode(yq);
      } else {
        ((uint16_t *)kv_cache)[row + i] = x;
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ */
/* Upstream of the cache write: kv_a_layernorm and the rotary embedding */
/* ------------------------------------------------------------------ */

/* fp64 value -> bf16 bits, one rounding: to nearest, ties to even.  bf16 is
 * binary32 cut to 8 significant bits (same exponent range, subnormals down
 * to 2^-133).  The quantum at |x| is 2^(E-7) for |x| in [2^E, 2^(E+1)),
 * E >= -126, and 2^-133 below 2^-126; |x| / quantum is exact in fp64, is
 * rounded to the nearest integer with ties to even, and multiplied back.  A
 * result of 2^128 or more is infinity.  NaN -> 0x7FC0. */
uint16_t oracle_bf16_round(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int k;
  (void)frexp(a, &k); /* a = m 2^k, m in [0.5, 1): a in [2^(k-1), 2^k) */
  int E = k - 1;
  double quantum = ldexp(1.0, (E < -126 ? -126 : E) - 7);
  double n = a / quantum;
  double fl = floor(n);
  double frac = n - fl;
  double r = fl;
  if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;
  double v = r * quantum;
  if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)v; /* exact: at most 8 significant bits, in range */
  uint32_t w;
  memcpy(&w, &f, sizeof w);
  return sign | (uint16_t)(w >> 16);
}

/* RMSNorm of each latent row before it is cached ([diff]
 * vllm/model_executor/models/deepseek_v2.py: kv_a_layernorm =
 * RMSNorm(kv_lora_rank, eps=rms_norm_eps), applied to kv_c in forward).  The
 * pages print no body; the plain reading of RMSNorm:
 *   out[d] = x[d] / sqrt(mean_d x[d]^2 + eps) * gamma[d],
 * evaluated in fp64 and rounded once to bf16.  x rows at x_row_stride; out
 * dense [n_rows][R]. */
void oracle_rms_norm(const uint16_t *x, int64_t x_row_stride, int64_t n_rows, int R,
                     const uint16_t *gamma, double eps, uint16_t *out) {
  for (int64_t t = 0; t < n_rows; ++t) {
    const uint16_t *xr = x + t * x_row_stride;
    double ss = 0.0;
    for (int d = 0; d < R; ++d) {
      double v = oracle_bf16_value(xr[d]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / R + eps);
    for (int d = 0; d < R; ++d)
      out[t * R + d] =
          oracle_bf16_round(oracle_bf16_value(xr[d]) * inv * oracle_bf16_value(gamma[d]));
  }
}

/* Rotary embedding, non-NeoX ("GPT-J") style, in place ([diff]
 * deepseek_v2.py: rotary_emb = get_rope(qk_rope_head_dim, ...,
 * rope_type 'deepseek_yarn', is_neox_style=False); applied to q_pe and k_pe
 * by input position before concat_and_cache_mla, MLA common forward).  The
 * pages print neither the rotation nor the table.  Readings: non-NeoX
 * rotates the interleaved pairs (x[2i], x[2i+1]), i < P/2, by the angle of
 * pair i:
 *   x'[2i]   = x[2i] cos_i - x[2i+1] sin_i
 *   x'[2i+1] = x[2i+1] cos_i + x[2i] sin_i,
 * with cos_i = table[pos][i] and sin_i = table[pos][P/2 + i] (the DeepSeek
 * YaRN frequencies and magnitude scale are whatever the fp32 table holds);
 * fp64 arithmetic, one rounding to bf16.  x is [n_rows][n_heads][P] bf16 at
 * the given strides; every head of row t uses positions[t].  A row whose
 * position is outside [0, max_position) is left as it is.  Returns the
 * number of such rows. */
int64_t oracle_rope_interleaved(uint16_t *x, int64_t row_stride, int64_t head_stride,
                                int64_t n_rows, int n_heads, int P, const int64_t *positions,
                                const float *table, int64_t max_position) {
  int64_t bad = 0;
  for (int64_t t = 0; t < n_rows; ++t) {
    int64_t pos = positions[t];
    if (pos < 0 || pos >= max_position) {
      ++bad;
      continue;
    }
    const float *cs = table + pos * P;
    for (int h = 0; h < n_heads; ++h) {
      uint16_t *v = x + t * row_stride + h * head_stride;
      for (int i = 0; i < P / 2; ++i) {
        double a = oracle_bf16_value(v[2 * i]), b = oracle_bf16_value(v[2 * i + 1]);
        double c = cs[i], s = cs[P / 2 + i];
        v[2 * i] = oracle_bf16_round(a * c - b * s);
        v[2 * i + 1] = oracle_bf16_round(b * c + a * s);
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------ */
/* Decode                                                              */
/* ------------------------------------------------------------------ */

typedef struct {
  const uint16_t *q;
  int64_t q_row_stride, q_head_stride;
  int num_rows, num_heads;
  const void *kv_cache;
  int kv_is_fp8;
  int64_t num_blocks;
  int block_size;
  int64_t block_stride;
  int R, P;
  const int32_t *block_table;
  int64_t block_table_stride;
  const int32_t *seq_lens;
  int num_seqs;
  double sm_scale, kv_scale;
} dec_args;

/* Value of element d of the latent row of token j of sequence b, fp64.
 * The page of token j is block_table[b][j / bs]; inside it the row is
 * j % bs ([diff] triton_decode_attention.py, _fwd_grouped_kernel_stage1:
 * kv_page_number / kv_loc).  The fp8 cache dequantises with the same scale
 * for K and V ([note] Data flow: k_scale = v_scale = layer._k_scale).  A
 * block id outside [0, num_blocks) reads as zeros (reading of an unchecked
 * case; the GPU's tensor-map loads fill out-of-range boxes with zeros). */
static double kv_elem(const dec_args *A, int b, int64_t j, int d) {
  int32_t blk = A->block_table[(int64_t)b * A->block_table_stride +
                               j / A->block_size];
  if (blk < 0 || (int64_t)blk >= A->num_blocks) return 0.0;
  int64_t idx = (int64_t)blk * A->block_stride +
                (j % A->block_size) * (int64_t)(A->R + A->P) + d;
  if (A->kv_is_fp8 == 2)
    return oracle_e5m2_value(((const uint8_t *)A->kv_cache)[idx]) *
           A->kv_scale;
  if (A->kv_is_fp8)
    return oracle_e4m3_value(((const uint8_t *)A->kv_cache)[idx]) *
           A->kv_scale;
  return oracle_bf16_value(((const uint16_t *)A->kv_cache)[idx]);
}

/* score s_j = sm_scale * sum_{d < R+P} q[r,h,d] * K_j[d]: the dot over the
 * latent and rope parts, then the scale ([diff] _fwd_grouped_kernel_stage1:
 * qk = dot(q, k) + dot(qpe, kpe); qk *= sm_scale). */
static double score(const dec_args *A, int r, int h, int b, int64_t j) {
  const int D = A->R + A->P;
  double acc = 0.0;
  const uint16_t *qr = A->q + (int64_t)r * A->q_row_stride +
                       (int64_t)h * A->q_head_stride;
  for (int d = 0; d < D; ++d)
    acc += oracle_bf16_value(qr[d]) * kv_elem(A, b, j, d);
  return A->sm_scale * acc;
}

/* Softmax attention of (r, h) over tokens [j0, j1) of its sequence, by the
 * plain definition: m = max s_j, Z = sum exp(s_j - m),
 * o = sum exp(s_j - m) V_j / Z with V_j = K_j[0:R] (MLA: V is the latent
 * part of the same cached row, [note] Data flow), lse = m + ln Z.
 * s[] is scratch of length >= j1 - j0.  Requires j1 > j0. */
static void attend_range(const dec_args *A, int r, int h, int b, int64_t j0,
                         int64_t j1, double *s, double *o, double *lse) {
  const int R = A->R;
  double m = -INFINITY;
  for (int64_t j = j0; j < j1; ++j) {
    s[j - j0] = score(A, r, h, b, j);
    if (s[j - j0] > m) m = s[j - j0];
  }
  double Z = 0.0;
  for (int64_t j = j0; j < j1; ++j) Z += exp(s[j - j0] - m);
  for (int d = 0; d < R; ++d) o[d] = 0.0;
  for (int64_t j = j0; j < j1; ++j) {
    double w = exp(s[j - j0] - m);
    for (int d = 0; d < R; ++d) o[d] += w * kv_elem(A, b, j, d);
  }
  for (int d = 0; d < R; ++d) o[d] /= Z;
  *lse = m + log(Z);
}

/* One (row, head) pair.  Row r belongs to sequence r / rows_per_seq, with
 * rows_per_seq = num_rows / num_seqs (consecutive rows of one sequence are
 * the flattened non-causal query rows of [api] TritonMLAMetadataBuilder;
 * they all attend to the whole sequence, no causal mask).  A sequence of
 * length 0 gives o = 0 and lse = -inf (reading; the pages' stage 2 would
 * divide 0 by 0).
 *
 * num_kv_splits == 0: the direct definition over all tokens.
 * num_kv_splits >= 1: the split-KV route of [diff] triton_decode_attention.py
 *   (_fwd_grouped_kernel_stage1 then _fwd_kernel_stage2): per = ceil(L/S),
 *   split s covers [s*per, min(s*per + per, L)), empty splits are skipped;
 *   each non-empty split yields its normalised o_s and lse_s; the merge is
 *   M = max lse_s, o = sum e^{lse_s - M} o_s / sum e^{lse_s - M},
 *   lse = M + ln sum e^{lse_s - M}, splits visited in index order. */
static void decode_pair(const dec_args *A, int r, int h, int num_kv_splits,
                        double *o, double *lse, double *s, double *tmp) {
  const int R = A->R;
  int rows_per_seq = A->num_rows / A->num_seqs;
  int b = r / rows_per_seq;
  int64_t L = A->seq_lens[b];
  if (L <= 0) {
    for (int d = 0; d < R; ++d) o[d] = 0.0;
    *lse = -INFINITY;
    return;
  }
  if (num_kv_splits <= 0) {
    attend_range(A, r, h, b, 0, L, s, o, lse);
    return;
  }
  int64_t S = num_kv_splits;
  int64_t per = (L + S - 1) / S;
  /* first pass: the maximum of the split lse values */
  double M = -INFINITY;
  for (int64_t sp = 0; sp < S; ++sp) {
    int64_t st = sp * per, en = st + per < L ? st + per : L;
    if (en <= st) continue;
    double ls;
    attend_range(A, r, h, b, st, en, s, tmp, &ls);
    if (ls > M) M = ls;
  }
  double den = 0.0;
  for (int d = 0; d < R; ++d) o[d] = 0.0;
  for (int64_t sp = 0; sp < S; ++sp) {
    int64_t st = sp * per, en = st + per < L ? st + per : L;
    if (en <= st) continue;
    double ls;
    attend_range(A, r, h, b, st, en, s, tmp, &ls);
    double w = exp(ls - M);
    for (int d = 0; d < R; ++d) o[d] += w * tmp[d];
    den += w;
  }
  for (int d = 0; d < R; ++d) o[d] /= den;
  *lse = M + log(den);
}

/* Decode for a list of (row, head) pairs (pairs[2k], pairs[2k+1]); pairs ==
 * NULL means every (row, head) in row-major order.  o_out is
 * [num_pairs, R] fp64, lse_out [num_pairs] fp64.  scratch_s must hold
 * num_threads * max_seq_len doubles and scratch_o num_threads * R doubles.
 * Pairs are independent, so they are spread over threads; each pair's
 * arithmetic is sequential and identical whatever the thread count. */
void oracle_decode(const uint16_t *q, int64_t q_row_stride,
                   int64_t q_head_stride, int num_rows, int num_heads,
                   const void *kv_cache, int kv_is_fp8, int64_t num_blocks,
                   int block_size, int64_t block_stride, int kv_lora_rank,
                   int rope_dim, const int32_t *block_table,
                   int64_t block_table_stride, const int32_t *seq_lens,
                   int num_seqs, float sm_scale, float kv_scale,
                   int num_kv_splits, const int64_t *pairs, int64_t num_pairs,
                   double *o_out, double *lse_out, double *scratch_s,
                   int64_t max_seq_len, double *scratch_o, int num_threads) {
  dec_args A = {q,          q_row_stride,   q_head_stride, num_rows,
                num_heads,  kv_cache,       kv_is_fp8,     num_blocks,
                block_size, block_stride,   kv_lora_rank,  rope_dim,
                block_table, block_table_stride, seq_lens, num_seqs,
                (double)sm_scale, (double)kv_scale};
  int64_t n = pairs ? num_pairs : (int64_t)num_rows * num_heads;
  if (num_threads < 1) num_threads = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int64_t k = 0; k < n; ++k) {
    int tid = 0;
#ifdef _OPENMP
    tid = omp_get_thread_num();
#endif
    int r = pairs ? (int)pairs[2 * k] : (int)(k / num_heads);
    int h = pairs ? (int)pairs[2 * k + 1] : (int)(k % num_heads);
    decode_pair(&A, r, h, num_kv_splits, o_out + k * kv_lora_rank,
                lse_out + k, scratch_s + (int64_t)tid * max_seq_len,
                scratch_o + (int64_t)tid * kv_lora_rank);
  }
}

/* Split-count rule ([note] Key files: _compute_num_kv_splits picks the KV
 * split count from max_seq_len / 512, capped at sm_count * 2; [note] Data
 * flow: VLLM_BATCH_INVARIANT forces 1 split).  The body is not printed; the
 * plainest reading is min(ceil(max_seq_len / 512), 2 * sm_count), at least 1. */
/* Cross-shard merge ([note] Design motivation: decode returns lse because
 * decode context parallelism merges the per-shard (o, lse) pairs with
 * cp_lse_ag_out_rs; [api] decode with DCP all-gathers q heads first).  The
 * same LSE algebra as the split merge above: for each of n (row, head)
 * records, M = max over the G parts of lse_g (parts with lse = -inf hold no
 * tokens and are skipped), o = sum e^{lse_g - M} o_g / sum e^{lse_g - M},
 * lse = M + ln sum e^{lse_g - M}, parts visited in index order; when every
 * part is empty, o = 0 and lse = -inf.  o_parts is [G][n][R], lse_parts
 * [G][n], both fp64. */
void oracle_lse_merge(const double *o_parts, const double *lse_parts, int G, int64_t n,
                      int R, double *o, double *lse) {
  for (int64_t i = 0; i < n; ++i) {
    double M = -INFINITY;
    for (int g = 0; g < G; ++g)
      if (lse_parts[(int64_t)g * n + i] > M) M = lse_parts[(int64_t)g * n + i];
    double *oi = o + i * R;
    for (int d = 0; d < R; ++d) oi[d] = 0.0;
    if (M == -INFINITY) {
      lse[i] = -INFINITY;
      continue;
    }
    double den = 0.0;
    for (int g = 0; g < G; ++g) {
      double lg = lse_parts[(int64_t)g * n + i];
      if (lg == -INFINITY) continue;
      double w = exp(lg - M);
      const double *og = o_parts + ((int64_t)g * n + i) * R;
      for (int d = 0; d < R; ++d) oi[d] += w * og[d];
      den += w;
    }
    for (int d = 0; d < R; ++d) oi[d] /= den;
    lse[i] = M + log(den);
  }
}

int oracle_num_kv_splits(int64_t max_seq_len, int sm_count, int deterministic) {
  if (deterministic) return 1;
  int64_t s = (max_seq_len + 511) / 512;
  int64_t cap = 2 * (int64_t)sm_count;
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  return (int)s;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Array forms of the scalar codecs, for the tests' exhaustive sweeps. */
void oracle_e4m3_encode_n(const float *y, uint8_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(y[i]);
}
void oracle_e4m3_value_n(const uint8_t *codes, double *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]);
}
void oracle_bf16_value_n(const uint16_t *bits, double *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_value(bits[i]);
}
void oracle_e5m2_encode_n(const float *y, uint8_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_encode(y[i]);
}
void oracle_e5m2_value_n(const uint8_t *codes, double *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_value(codes[i]);
}
void oracle_bf16_round_n(const double *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_round(x[i]);
}
