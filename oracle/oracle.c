/*
 * oracle.c -- plain, slow, fp64 CPU implementation of the hybrid-attention hot path.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this library. It shares no code, header, table or helper
 * with the CUDA path; it re-derives every index from the written layout below.
 *
 * Pages followed:
 *   [KV] "推理框架适配Hybrid Model：KV Cache管理与算子调度实战" (icman.com.cn/news/43047)
 *   [VL] "Hybrid Model推理适配：vLLM与SGLang的工程实践指南"   (gsyq.cn/news/436086)
 *
 * Layouts (element indices; every product is formed in int64):
 *   paged K or V cache  [num_blocks][H][bs][D]: element (blk,h,s,d) at ((blk*H+h)*bs+s)*D+d
 *   block table         int32 [B][MB]: logical block -> physical block
 *   slot                blk*bs + offset inside the block; -1 means "write nothing"
 *   packed rows q/k/v   [T][H][D]; decode batches use T = B
 *   linear state        fp32 [num_slots][H][D][D]; row i = key dim, column j = value dim
 *   element types       dtype 0 = fp32, dtype 1 = bf16 (raw 16-bit patterns)
 *
 * All arithmetic is fp64 and follows the definitions in the order the pages give
 * them; no blocking, no online softmax, no reassociation beyond plain loops.
 * Built with -ffp-contract=off so results do not depend on the host's FMA use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ helpers */
static double ld(const void *p, int64_t i, int dtype) {
  if (dtype == 1) {
    uint32_t w = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
  }
  return (double)((const float *)p)[i];
}

int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}

/* ------------------------------------------------------ A1: slot mapping
 * [KV §2.1]: the KV of every token is kept; it is cut into blocks holding a fixed
 * number of tokens (16) and blocks are reached through a page table. The token at
 * absolute position p of request b therefore sits at offset p % bs of logical
 * block p / bs, whose physical block is block_tables[b][p / bs].
 * Token j of request b in a call sits at absolute position ctx_lens[b] + j.
 * Returns 0, or -1 if a position needs a logical block beyond MB. */
int oracle_slot_mapping(const int32_t *block_tables, int MB, const int32_t *cu_q_lens,
                        const int32_t *ctx_lens, int B, int bs, int64_t *slot_out) {
  for (int b = 0; b < B; ++b) {
    for (int t = cu_q_lens[b]; t < cu_q_lens[b + 1]; ++t) {
      int64_t p = (int64_t)(ctx_lens ? ctx_lens[b] : 0) + (t - cu_q_lens[b]);
      int64_t logical = p / bs;
      if (logical >= MB) return -1;
      int32_t blk = block_tables[(int64_t)b * MB + logical];
      slot_out[t] = blk < 0 ? -1 : (int64_t)blk * bs + p % bs;
    }
  }
  return 0;
}

/* ------------------------------------------------------ A2: KV append
 * [KV §2.1]: each token's key and value vectors are saved. Bytewise copy of row
 * (t, h) into (slot / bs, h, slot % bs); slot -1 is skipped. */
void oracle_kv_append(const void *k, const void *v, const int64_t *slot_mapping, int T,
                      int H, int D, int bs, int esize, void *k_cache, void *v_cache) {
  for (int t = 0; t < T; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    int64_t blk = s / bs, off = s % bs;
    for (int h = 0; h < H; ++h) {
      int64_t dst = ((blk * H + h) * bs + off) * (int64_t)D * esize;
      int64_t src = ((int64_t)t * H + h) * (int64_t)D * esize;
      memcpy((char *)k_cache + dst, (const char *)k + src, (size_t)D * esize);
      memcpy((char *)v_cache + dst, (const char *)v + src, (size_t)D * esize);
    }
  }
}

/* element d of the key (or value) at absolute position p of request b, head h,
 * found by walking the block table [KV §2.1] */
static double paged(const void *cache, const int32_t *bt, int MB, int b, int h, int64_t p,
                    int d, int H, int D, int bs, int dtype) {
  int64_t blk = bt[(int64_t)b * MB + p / bs];
  return ld(cache, ((blk * H + h) * bs + p % bs) * (int64_t)D + d, dtype);
}

/* softmax(scale * q.K_p) V_p over p in [lo, n), q given as doubles; two plain passes */
static void attend(const double *q, const void *kc, const void *vc, const int32_t *bt, int MB,
                   int b, int h, int64_t lo, int64_t n, int H, int D, int bs, int dtype,
                   double scale, double *s, double *o) {
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (n <= lo) return;
  double m = -INFINITY;
  for (int64_t p = lo; p < n; ++p) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * paged(kc, bt, MB, b, h, p, d, H, D, bs, dtype);
    s[p] = scale * dot;
    if (s[p] > m) m = s[p];
  }
  double den = 0.0;
  for (int64_t p = lo; p < n; ++p) {
    double w = exp(s[p] - m);
    den += w;
    for (int d = 0; d < D; ++d) o[d] += w * paged(vc, bt, MB, b, h, p, d, H, D, bs, dtype);
  }
  for (int d = 0; d < D; ++d) o[d] /= den;
}

/* ------------------------------------------------------ A3: Full paged decode
 * [KV §2.3]: decode uses a PagedAttention-type kernel whose inputs are Q, K, V and
 * the block table. Per (b, h): o = sum_p softmax_p(scale * q.K_p) V_p over the
 * seq_lens[b] cached positions (the token of this step has already been appended).
 * seq_len 0 gives a zero row. window > 0 keeps only the last `window` positions
 * (sliding-window attention, the model-side alternative of [KV §1.3]). out: fp64 [B][H][D]. */
void oracle_full_decode(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, int MB, const int32_t *seq_lens, int B,
                        int H, int D, int bs, int dtype, double scale, int window, double *out) {
  int64_t nmax = 1;
  for (int b = 0; b < B; ++b) if (seq_lens[b] > nmax) nmax = seq_lens[b];
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * nmax);
    double *qd = (double *)malloc(sizeof(double) * D);
#pragma omp for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; ++b)
      for (int h = 0; h < H; ++h) {
        for (int d = 0; d < D; ++d) qd[d] = ld(q, ((int64_t)b * H + h) * D + d, dtype);
        const int64_t n = seq_lens[b];
        const int64_t lo = (window > 0 && n > window) ? n - window : 0;
        attend(qd, k_cache, v_cache, block_tables, MB, b, h, lo, n, H, D, bs, dtype, scale, s,
               out + ((int64_t)b * H + h) * D);
      }
    free(s);
    free(qd);
  }
}

/* ------------------------------------------------------ A4: Full causal prefill
 * [KV §2.3]: prefill runs a FlashAttention-type kernel; the result it must equal is
 * causal softmax attention. Token j of request b (packed row t = cu_q_lens[b] + j)
 * sits at absolute position i = ctx_lens[b] + j and attends to cached positions
 * p <= i (the call's own keys were appended to the cache first).
 * window > 0 keeps only the positions p > i - window (sliding window).
 * rows == NULL: out fp64 [T][H][D]. Otherwise only the packed rows listed are
 * computed and out is [nrows][H][D]. */
void oracle_full_prefill(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int MB, const int32_t *cu_q_lens,
                         const int32_t *ctx_lens, int B, int H, int D, int bs, int dtype,
                         double scale, int window, const int32_t *rows, int nrows,
                         double *out) {
  int T = cu_q_lens[B];
  int n_out = rows ? nrows : T;
  int64_t nmax = 1;
  for (int b = 0; b < B; ++b) {
    int64_t e = (int64_t)(ctx_lens ? ctx_lens[b] : 0) + cu_q_lens[b + 1] - cu_q_lens[b];
    if (e > nmax) nmax = e;
  }
#pragma omp parallel
  {
    double *s = (double *)malloc(sizeof(double) * nmax);
    double *qd = (double *)malloc(sizeof(double) * D);
#pragma omp for collapse(2) schedule(dynamic, 1)
    for (int r = 0; r < n_out; ++r)
      for (int h = 0; h < H; ++h) {
        int t = rows ? rows[r] : r;
        int b = 0;
        while (b + 1 < B && cu_q_lens[b + 1] <= t) ++b;
        int64_t i = (int64_t)(ctx_lens ? ctx_lens[b] : 0) + (t - cu_q_lens[b]);
        for (int d = 0; d < D; ++d) qd[d] = ld(q, ((int64_t)t * H + h) * D + d, dtype);
        const int64_t lo = (window > 0 && i + 1 > window) ? i + 1 - window : 0;
        attend(qd, k_cache, v_cache, block_tables, MB, b, h, lo, i + 1, H, D, bs, dtype, scale,
               s, out + ((int64_t)r * H + h) * D);
      }
    free(s);
    free(qd);
  }
}

/* ------------------------------------------------------ A5: Linear recurrence
 * [KV §2.1]: the linear layer keeps a state matrix (D x D per head, H x D x D per
 * request); each new token updates it as S <- S + k (outer) v and the output is q.S.
 * [KV §2.3]: the state is zeroed when the request starts, accumulated through
 * prefill and carried into decode.
 * Readings: k (outer) v = k v^T (row i = key dim, column j = value dim); the output
 * uses the state after this token's update; q.S = sum_i q_i S_ij; no feature map,
 * normaliser, decay or scale.
 * Request b covers packed rows [cu[b], cu[b+1]). Its starting state is zero when
 * reset[b] != 0 or state_pool is NULL, else state_pool[state_slots[b]] (fp32).
 * out fp64 [T][H][D]; state_out fp64 [B][H][D][D] (the state after the last row). */
void oracle_linear_recurrence(const void *q, const void *k, const void *v, const int32_t *cu,
                              int B, int H, int D, int dtype, const float *state_pool,
                              const int32_t *state_slots, const uint8_t *reset, double *out,
                              double *state_out) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      double *S = state_out + ((int64_t)b * H + h) * D * D;
      int zero = (state_pool == NULL) || (reset && reset[b]);
      for (int64_t e = 0; e < (int64_t)D * D; ++e)
        S[e] = zero ? 0.0
                    : (double)state_pool[((int64_t)state_slots[b] * H + h) * D * D + e];
      for (int t = cu[b]; t < cu[b + 1]; ++t) {
        int64_t row = ((int64_t)t * H + h) * D;
        for (int i = 0; i < D; ++i) {
          double ki = ld(k, row + i, dtype);
          for (int j = 0; j < D; ++j) S[(int64_t)i * D + j] += ki * ld(v, row + j, dtype);
        }
        for (int j = 0; j < D; ++j) {
          double o = 0.0;
          for (int i = 0; i < D; ++i) o += ld(q, row + i, dtype) * S[(int64_t)i * D + j];
          out[row + j] = o;
        }
      }
    }
}

/* ------------------------------------------------------ Linear recurrence, 16-bit state
 * The state-precision comparison: the vLLM/SGLang page keeps the linear state in fp16,
 * [KV §2.3] keeps it in fp32 so that it does not drift. Here the state is held as 16-bit
 * values and each token updates every element as
 *     S_ij <- round16(fmaf(k_i, v_j, S_ij))
 * (one fp32 fused multiply-add, then one rounding to the 16-bit format, nearest with ties
 * to even), and the output reads the rounded state: o_j = sum_i q_i S_ij, summed in fp64.
 * state_dtype 1 = bf16, 2 = fp16. state_pool (may be NULL) and state_out hold raw 16-bit
 * patterns, [slots][H][D][D] and [B][H][D][D]. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x40u);   /* NaN */
  x += 0x7fffu + ((x >> 16) & 1u);
  return (uint16_t)(x >> 16);
}
static float bf16_to_f32(uint16_t u) {
  uint32_t x = (uint32_t)u << 16;
  float f;
  memcpy(&f, &x, 4);
  return f;
}
static uint16_t f32_to_f16_rne(float f) {   /* C's conversion to _Float16 rounds to nearest even */
  _Float16 h = (_Float16)f;
  uint16_t u;
  memcpy(&u, &h, 2);
  return u;
}
static float f16_to_f32(uint16_t u) {
  _Float16 h;
  memcpy(&h, &u, 2);
  return (float)h;
}

void oracle_linear_recurrence_lowp(const void *q, const void *k, const void *v,
                                   const int32_t *cu, int B, int H, int D, int dtype,
                                   int state_dtype, const uint16_t *state_pool,
                                   const int32_t *state_slots, const uint8_t *reset, double *out,
                                   uint16_t *state_out) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      uint16_t *S = state_out + ((int64_t)b * H + h) * D * D;
      int zero = (state_pool == NULL) || (reset && reset[b]);
      for (int64_t e = 0; e < (int64_t)D * D; ++e)
        S[e] = zero ? 0 : state_pool[((int64_t)state_slots[b] * H + h) * D * D + e];
      for (int t = cu[b]; t < cu[b + 1]; ++t) {
        int64_t row = ((int64_t)t * H + h) * D;
        for (int i = 0; i < D; ++i) {
          float ki = (float)ld(k, row + i, dtype);
          for (int j = 0; j < D; ++j) {
            uint16_t *e = &S[(int64_t)i * D + j];
            float vj = (float)ld(v, row + j, dtype);
            float sf = state_dtype == 1 ? bf16_to_f32(*e) : f16_to_f32(*e);
            float nf = fmaf(ki, vj, sf);
            *e = state_dtype == 1 ? f32_to_bf16_rne(nf) : f32_to_f16_rne(nf);
          }
        }
        for (int j = 0; j < D; ++j) {
          double o = 0.0;
          for (int i = 0; i < D; ++i) {
            uint16_t e = S[(int64_t)i * D + j];
            o += ld(q, row + i, dtype) * (double)(state_dtype == 1 ? bf16_to_f32(e) : f16_to_f32(e));
          }
          out[row + j] = o;
        }
      }
    }
}

/* ------------------------------------------------------ A6: Linear chunk form
 * [KV §2.4]: long prompts are prefilled in chunks; a linear layer carries its state
 * from chunk to chunk and chunk boundaries sit at the same positions in every layer.
 * Chunks are the position ranges [c*C, (c+1)*C) counted from the request start
 * (absolute position = ctx_lens[b] + row offset), so a call that starts at an
 * unaligned position begins with a short chunk. Per chunk, with S the state at the
 * chunk start:
 *   o_t = q_t S + sum_{t' in chunk, t' <= t} (q_t . k_t') v_t'
 *   S  <- S + sum_{t' in chunk} k_t' v_t'^T
 * This is the same quantity as the recurrence, associated differently; it exists so
 * the two can pin each other. Arguments as in oracle_linear_recurrence. */
void oracle_linear_chunked(const void *q, const void *k, const void *v, const int32_t *cu,
                           const int32_t *ctx_lens, int B, int H, int D, int C, int dtype,
                           const float *state_pool, const int32_t *state_slots,
                           const uint8_t *reset, double *out, double *state_out) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      double *S = state_out + ((int64_t)b * H + h) * D * D;
      int zero = (state_pool == NULL) || (reset && reset[b]);
      for (int64_t e = 0; e < (int64_t)D * D; ++e)
        S[e] = zero ? 0.0
                    : (double)state_pool[((int64_t)state_slots[b] * H + h) * D * D + e];
      int64_t pos0 = ctx_lens ? ctx_lens[b] : 0;
      int t = cu[b];
      while (t < cu[b + 1]) {
        int64_t p = pos0 + (t - cu[b]);
        int64_t chunk_end_pos = (p / C + 1) * C;
        int e = t + (int)(chunk_end_pos - p);
        if (e > cu[b + 1]) e = cu[b + 1];
        for (int a = t; a < e; ++a) {
          int64_t ra = ((int64_t)a * H + h) * D;
          for (int j = 0; j < D; ++j) {
            double o = 0.0;
            for (int i = 0; i < D; ++i) o += ld(q, ra + i, dtype) * S[(int64_t)i * D + j];
            out[ra + j] = o;
          }
          for (int c = t; c <= a; ++c) {
            int64_t rc = ((int64_t)c * H + h) * D;
            double qk = 0.0;
            for (int i = 0; i < D; ++i) qk += ld(q, ra + i, dtype) * ld(k, rc + i, dtype);
            for (int j = 0; j < D; ++j) out[ra + j] += qk * ld(v, rc + j, dtype);
          }
        }
        for (int i = 0; i < D; ++i)
          for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int c = t; c < e; ++c) {
              int64_t rc = ((int64_t)c * H + h) * D;
              acc += ld(k, rc + i, dtype) * ld(v, rc + j, dtype);
            }
            S[(int64_t)i * D + j] += acc;
          }
        t = e;
      }
    }
}

/* ------------------------------------------------------ memory accounting
 * [KV §2.1]: Full-attention KV bytes = 2 x L x H x D x S x sizeof(dtype).
 * [KV §3.3]: with batch, Full part = 2 x L_full x H x D x S x batch x bytes and
 * Linear part = L_linear x H x D x D x batch x bytes. Returns full + linear. */
uint64_t oracle_cache_bytes(int L_full, int L_linear, int H, int D, int64_t tokens, int batch,
                            int kv_elem_bytes, int state_elem_bytes, uint64_t *full_out,
                            uint64_t *linear_out) {
  uint64_t full = 2ull * (uint64_t)L_full * (uint64_t)H * (uint64_t)D * (uint64_t)tokens *
                  (uint64_t)batch * (uint64_t)kv_elem_bytes;
  uint64_t lin = (uint64_t)L_linear * (uint64_t)H * (uint64_t)D * (uint64_t)D *
                 (uint64_t)batch * (uint64_t)state_elem_bytes;
  if (full_out) *full_out = full;
  if (linear_out) *linear_out = lin;
  return full + lin;
}
