/*
 * pa_oracle.c -- plain, slow fp64 CPU oracle of the paged-attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * loads this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code with the CUDA path (only the seeded
 * input generator, which holds no attention arithmetic, serves both).
 *
 * Sources (page title -- section):
 *  [ATT]  "Configuring vLLM and PagedAttention for High Throughput Enterprise
 *         LLM Serving" -- "Architectural Foundations: PagedAttention & Virtual
 *         Memory": the attention-weight equation
 *         A_ij = exp(q_i.k_j/sqrt(d)) / sum_m exp(q_i.k_m/sqrt(d)), and the
 *         address translation P_physical = BlockTable[j / B] with B tokens per
 *         block (B = 16 in the example).
 *  [MAP]  "vLLM Guide: High-Throughput Multi-GPU LLM Serving with
 *         PagedAttention" -- "What Is PagedAttention?": the logical->physical
 *         figure (tokens 0..15 -> block 9, 16..31 -> block 2, 32..47 -> block
 *         14), i.e. tokens fill a block in order; blocks shared with
 *         copy-on-write semantics.
 *  [PHASE] same page as [ATT] -- "Memory Bottlenecks in Autoregressive LLM
 *         Inference": prefill computes K/V for every token position; decode
 *         reads every previous K/V vector for each new token.
 *  [CHUNK] same page as [ATT] -- "High-Throughput Batching: Continuous
 *         Batching & Chunked Prefill": prompts split into chunks (512/1024).
 *  [SIZE] same page as [ATT] -- "Tuning Checklist for Production / KV Cache
 *         Memory Sizing Formula": bytes per token = 2 * layers * kv_heads *
 *         head_dim * bytes_per_element.
 *  [SWAP] same page as [ATT] -- "Quick Answers" (KV cache offloading when VRAM
 *         is full): a paused request's KV blocks move from GPU memory to host
 *         memory and, once blocks are free again, back to the GPU, so that
 *         generation resumes where it stopped.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes):
 *  - the attention output is sum_j A_ij v_j;
 *  - offset within a block is j mod B; "j / B" is floor division;
 *  - GQA maps query head h to kv head floor(h / G), G = Hq / Hkv;
 *  - the softmax is evaluated as exp(x_j - max x) / sum exp(x_m - max x),
 *    which equals [ATT] exactly in real arithmetic;
 *  - a decode step attends keys 0..ctx-1 (ctx includes the new token);
 *  - a prefill chunk of C rows over context ctx: row i sits at position
 *    ctx - C + i and attends keys 0..pos (causal);
 *  - ctx <= 0 or ctx > max_blocks * B, or a page id outside the pool, is an
 *    error: the result is zeros and a status bit is returned;
 *  - a negative slot in reshape_and_cache means "no write".
 *
 * Layouts (shared convention): pools bf16 [N_blk][H_kv][B][D] carried as
 * uint16 bit patterns; block tables int32 [S][max_blocks]; q bf16
 * [S][H_q][D]; outputs fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_CTX 1      /* ctx <= 0 or ctx > max_blocks * B */
#define ORA_ERR_PAGE 2     /* block id outside [0, num_blocks) */
#define ORA_ERR_SLOT 4     /* slot >= num_blocks * B */
#define ORA_ERR_ARGS 8

/* bf16 bit pattern -> double (exact: a bf16 is the top half of an fp32). */
double ora_bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* [SIZE]: KV-cache bytes per token over all layers. */
int64_t ora_kv_bytes_per_token(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t elem_bytes) {
  return 2 * layers * kv_heads * head_dim * elem_bytes;
}

/* [ATT] address translation for logical token j of a sequence:
 * page = table[j / B], offset = j mod B.  Returns the page id. */
static int32_t translate(const int32_t *table_row, int B, int j, int *offset) {
  *offset = j % B;
  return table_row[j / B];
}

/* Gather keys/values 0..n-1 of kv head g of one sequence into contiguous fp64
 * arrays K[n][D], V[n][D].  Returns ORA_ERR_PAGE if a page id is out of range. */
static int gather(const uint16_t *k_pool, const uint16_t *v_pool, int num_blocks, int Hkv, int B,
                  int D, const int32_t *table_row, int g, int n, double *K, double *V) {
  for (int j = 0; j < n; ++j) {
    int o;
    int32_t p = translate(table_row, B, j, &o);
    if (p < 0 || p >= num_blocks) return ORA_ERR_PAGE;
    size_t base = (((size_t)p * Hkv + g) * B + o) * (size_t)D;
    for (int d = 0; d < D; ++d) {
      K[(size_t)j * D + d] = ora_bf16_to_f64(k_pool[base + d]);
      V[(size_t)j * D + d] = ora_bf16_to_f64(v_pool[base + d]);
    }
  }
  return ORA_OK;
}

/* [ATT]: out = sum_j A_j v_j with A_j = exp(x_j) / sum_m exp(x_m),
 * x_j = scale * q.k_j, over n contiguous keys (n >= 1). */
static void attend(const double *q, const double *K, const double *V, int n, int D, double scale,
                   double *out) {
  double *x = (double *)malloc(sizeof(double) * (size_t)n);
  double m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += q[d] * K[(size_t)j * D + d];
    x[j] = scale * dot;
    if (x[j] > m) m = x[j];
  }
  double denom = 0.0;
  for (int j = 0; j < n; ++j) {
    x[j] = exp(x[j] - m);
    denom += x[j];
  }
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += x[j] * V[(size_t)j * D + d];
    out[d] = acc / denom;
  }
  free(x);
}

/* Decode attention for one (sequence s, query head h): out[D] in fp64.
 * Returns a status bit set (0 = ok); on error out is zero. */
int ora_decode_head(int S, int Hq, int Hkv, int D, int B, int num_blocks, int max_blocks,
                    const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                    const int32_t *block_tables, const int32_t *context_lens, double scale, int s,
                    int h, double *out) {
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (S <= 0 || Hkv <= 0 || Hq % Hkv != 0 || s < 0 || s >= S || h < 0 || h >= Hq) return ORA_ERR_ARGS;
  int G = Hq / Hkv;
  int g = h / G;
  int ctx = context_lens[s];
  if (ctx <= 0 || ctx > max_blocks * B) return ORA_ERR_CTX;
  double *K = (double *)malloc(sizeof(double) * (size_t)ctx * D);
  double *V = (double *)malloc(sizeof(double) * (size_t)ctx * D);
  double *qd = (double *)malloc(sizeof(double) * (size_t)D);
  int st = gather(k_pool, v_pool, num_blocks, Hkv, B, D, block_tables + (size_t)s * max_blocks, g,
                  ctx, K, V);
  if (st == ORA_OK) {
    for (int d = 0; d < D; ++d) qd[d] = ora_bf16_to_f64(q[((size_t)s * Hq + h) * D + d]);
    attend(qd, K, V, ctx, D, scale, out);
  }
  free(K);
  free(V);
  free(qd);
  return st;
}

/* Decode attention for every (s, h): out [S][Hq][D]; status [S] (or-ed bits). */
int ora_decode(int S, int Hq, int Hkv, int D, int B, int num_blocks, int max_blocks,
               const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
               const int32_t *block_tables, const int32_t *context_lens, double scale, double *out,
               int32_t *status) {
  int all = 0;
  for (int s = 0; s < S; ++s) {
    status[s] = 0;
    for (int h = 0; h < Hq; ++h) {
      int st = ora_decode_head(S, Hq, Hkv, D, B, num_blocks, max_blocks, q, k_pool, v_pool,
                               block_tables, context_lens, scale, s, h,
                               out + ((size_t)s * Hq + h) * D);
      status[s] |= st;
    }
    all |= status[s];
  }
  return all;
}

/* [PHASE]+[CHUNK]: causal attention for row i of chunk r and query head h.
 * Chunk r has C = cu_q[r+1] - cu_q[r] query rows over context ctx = context_lens[r]
 * (the chunk's own tokens included); row i sits at position ctx - C + i and sees
 * keys 0..pos.  q is [sum C][Hq][D]; out[D]. */
int ora_prefill_row(int R, int Hq, int Hkv, int D, int B, int num_blocks, int max_blocks,
                    const uint16_t *q, const int32_t *cu_q, const uint16_t *k_pool,
                    const uint16_t *v_pool, const int32_t *block_tables,
                    const int32_t *context_lens, double scale, int r, int i, int h, double *out) {
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (r < 0 || r >= R || Hkv <= 0 || Hq % Hkv != 0 || h < 0 || h >= Hq) return ORA_ERR_ARGS;
  int C = cu_q[r + 1] - cu_q[r];
  int ctx = context_lens[r];
  if (i < 0 || i >= C) return ORA_ERR_ARGS;
  if (ctx <= 0 || C > ctx || ctx > max_blocks * B) return ORA_ERR_CTX;
  int pos = ctx - C + i;
  int n = pos + 1;
  int G = Hq / Hkv;
  int g = h / G;
  double *K = (double *)malloc(sizeof(double) * (size_t)n * D);
  double *V = (double *)malloc(sizeof(double) * (size_t)n * D);
  double *qd = (double *)malloc(sizeof(double) * (size_t)D);
  int st = gather(k_pool, v_pool, num_blocks, Hkv, B, D, block_tables + (size_t)r * max_blocks, g,
                  n, K, V);
  if (st == ORA_OK) {
    size_t row = (size_t)cu_q[r] + (size_t)i;
    for (int d = 0; d < D; ++d) qd[d] = ora_bf16_to_f64(q[(row * Hq + h) * D + d]);
    attend(qd, K, V, n, D, scale, out);
  }
  free(K);
  free(V);
  free(qd);
  return st;
}

/* Partial attention of one (s, h) over the key range [j0, j1): the running
 * quantities m = max x_j, l = sum exp(x_j - m), o = sum exp(x_j - m) v_j / l.
 * An empty range gives m = -inf, l = 0, o = 0.  (Split-K state; the pages do
 * not describe a split, this is the plain definition of its pieces.) */
int ora_partial(int S, int Hq, int Hkv, int D, int B, int num_blocks, int max_blocks,
                const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                const int32_t *block_tables, const int32_t *context_lens, double scale, int s,
                int h, int j0, int j1, double *m_out, double *l_out, double *o_out) {
  for (int d = 0; d < D; ++d) o_out[d] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (s < 0 || s >= S || h < 0 || h >= Hq || Hkv <= 0 || Hq % Hkv != 0) return ORA_ERR_ARGS;
  int ctx = context_lens[s];
  if (ctx <= 0 || ctx > max_blocks * B) return ORA_ERR_CTX;
  if (j0 < 0) j0 = 0;
  if (j1 > ctx) j1 = ctx;
  if (j1 <= j0) return ORA_OK;
  int G = Hq / Hkv, g = h / G;
  double *K = (double *)malloc(sizeof(double) * (size_t)ctx * D);
  double *V = (double *)malloc(sizeof(double) * (size_t)ctx * D);
  int st = gather(k_pool, v_pool, num_blocks, Hkv, B, D, block_tables + (size_t)s * max_blocks, g,
                  ctx, K, V);
  if (st == ORA_OK) {
    double *x = (double *)malloc(sizeof(double) * (size_t)(j1 - j0));
    double m = -INFINITY;
    for (int j = j0; j < j1; ++j) {
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += ora_bf16_to_f64(q[((size_t)s * Hq + h) * D + d]) * K[(size_t)j * D + d];
      x[j - j0] = scale * dot;
      if (x[j - j0] > m) m = x[j - j0];
    }
    double l = 0.0;
    for (int j = j0; j < j1; ++j) {
      x[j - j0] = exp(x[j - j0] - m);
      l += x[j - j0];
    }
    for (int d = 0; d < D; ++d) {
      double acc = 0.0;
      for (int j = j0; j < j1; ++j) acc += x[j - j0] * V[(size_t)j * D + d];
      o_out[d] = acc / l;
    }
    *m_out = m;
    *l_out = l;
    free(x);
  }
  free(K);
  free(V);
  return st;
}

/* Combine P partial states (m_p, l_p, o_p) of disjoint key ranges into the
 * attention output: m = max m_p, w_p = l_p exp(m_p - m),
 * out = sum_p w_p o_p / sum_p w_p.  Parts with l_p = 0 contribute nothing. */
void ora_combine(int P, int D, const double *m, const double *l, const double *o, double *out) {
  double mx = -INFINITY;
  for (int p = 0; p < P; ++p)
    if (l[p] > 0.0 && m[p] > mx) mx = m[p];
  double den = 0.0;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int p = 0; p < P; ++p) {
    if (!(l[p] > 0.0)) continue;
    double w = l[p] * exp(m[p] - mx);
    den += w;
    for (int d = 0; d < D; ++d) out[d] += w * o[(size_t)p * D + d];
  }
  if (den > 0.0)
    for (int d = 0; d < D; ++d) out[d] /= den;
}

/* [PHASE]/[ATT]: write the K/V of T new tokens into their slots, in array
 * order: slot -> block slot / B, offset slot mod B.  Negative slot: no write.
 * k, v are bf16 [T][Hkv][D]; pools bf16 [N_blk][Hkv][B][D] (modified in place).
 * Returns ORA_ERR_SLOT if some slot is past the pool (that token is skipped). */
int ora_reshape_and_cache(int T, int Hkv, int D, int B, int num_blocks, const uint16_t *k,
                          const uint16_t *v, uint16_t *k_pool, uint16_t *v_pool,
                          const int64_t *slot_mapping) {
  int st = ORA_OK;
  for (int t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= (int64_t)num_blocks * B) {
      st |= ORA_ERR_SLOT;
      continue;
    }
    int64_t p = slot / B, o = slot % B;
    for (int h = 0; h < Hkv; ++h)
      for (int d = 0; d < D; ++d) {
        size_t dst = (((size_t)p * Hkv + h) * B + (size_t)o) * D + d;
        size_t src = ((size_t)t * Hkv + h) * D + d;
        k_pool[dst] = k[src];
        v_pool[dst] = v[src];
      }
  }
  return st;
}

/* [MAP] copy-on-write: for each layer and each (src, dst) pair in order, the
 * whole dst block (all kv heads, K and V) becomes a copy of the src block.
 * k_pools/v_pools: arrays of L pool pointers; block_elems = Hkv * B * D. */
int ora_copy_blocks(int L, uint16_t *const *k_pools, uint16_t *const *v_pools, int num_blocks,
                    int64_t block_elems, const int64_t *pairs, int num_pairs) {
  int st = ORA_OK;
  for (int l = 0; l < L; ++l)
    for (int i = 0; i < num_pairs; ++i) {
      int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
      if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
        st |= ORA_ERR_PAGE;
        continue;
      }
      memcpy(k_pools[l] + dst * block_elems, k_pools[l] + src * block_elems,
             sizeof(uint16_t) * (size_t)block_elems);
      memcpy(v_pools[l] + dst * block_elems, v_pools[l] + src * block_elems,
             sizeof(uint16_t) * (size_t)block_elems);
    }
  return st;
}

/* [SWAP] preemptive swapping: for each layer l and each (src, dst) pair in
 * order, block dst of the destination pools (dst_k[l], dst_v[l]) becomes a
 * copy of block src of the source pools (src_k[l], src_v[l]) -- K and V, every
 * kv head, token and element.  Source and destination are different pools
 * (device and host) with their own block counts; block_elems = Hkv * B * D.
 * A pair outside either pool is skipped and ORA_ERR_PAGE returned. */
int ora_swap_blocks(int L, const uint16_t *const *src_k, const uint16_t *const *src_v, uint16_t *const *dst_k,
                    uint16_t *const *dst_v, int src_blocks, int dst_blocks, int64_t block_elems,
                    const int64_t *pairs, int num_pairs) {
  int st = ORA_OK;
  for (int l = 0; l < L; ++l)
    for (int i = 0; i < num_pairs; ++i) {
      int64_t from = pairs[2 * i], to = pairs[2 * i + 1];
      if (from < 0 || from >= src_blocks || to < 0 || to >= dst_blocks) {
        st |= ORA_ERR_PAGE;
        continue;
      }
      for (int64_t e = 0; e < block_elems; ++e) {
        dst_k[l][to * block_elems + e] = src_k[l][from * block_elems + e];
        dst_v[l][to * block_elems + e] = src_v[l][from * block_elems + e];
      }
    }
  return st;
}
