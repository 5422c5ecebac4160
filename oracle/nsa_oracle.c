/*
 * nsa_oracle.c -- plain CPU oracle for the native-sparse-attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference arm may load this library.  It shares
 * no code, header, table or helper with the CUDA library; neither includes the
 * other.  It is deliberately slow: plain loops, fp64 accumulation, one row at a
 * time, OpenMP only across independent rows.
 *
 * Sources (web pages; cited by title and section):
 *   [NOSA-Triton]  "NOSA-1B source walk-through #3: how the Triton kernel speeds up
 *                   attention" (kwkr.cn/news/198629)
 *   [NOSA-Parts]   "NOSA-1B core components: how KV-cache offload gives 5.04x decode
 *                   throughput" (kwkr.cn/news/199670)
 *   [NSA-Triton]   "DeepSeek NSA sparse attention in practice: optimising training
 *                   with Triton" (mcp.csdn.net)
 *   [TileLang-NSA] "TileLang operator development: Native Sparse Attention
 *                   implementation and optimisation" (devpress.csdn.net)
 *
 * Notation (per sequence of length L, positions t = 0..L-1 relative to its start):
 *   H query heads, Hkv kv-heads, group size r = H/Hkv, head h reads kv-head h / r
 *   ([TileLang-NSA] sec. 2, "head_kv = heads // groups").
 *   compression kernel l and stride s ([NOSA-Parts] core component 1: 32 and 16);
 *   n_c(L) = floor((L-l)/s)+1 compressed keys when L >= l, else 0 (full windows only).
 *   selection block size B ([NOSA-Parts] core component 1; [TileLang-NSA] sec. 2: 64).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - compressed key c is causal for query t iff its window ends at or before t:
 *     c*s + l - 1 <= t.  Rows with no causal compressed key get probability 0.
 *   - the pooled block score of block j is the mean of the group probabilities of
 *     the compressed windows lying inside block j, {c : c*s >= jB, c*s+l <= (j+1)B},
 *     counting only windows that exist (c < n_c(L)); causally masked windows count
 *     as zeros; an empty set gives 0.
 *   - top-k keeps the forced blocks (n_init initial, n_local local ending at the
 *     query's own block), excludes blocks starting after t, breaks ties toward the
 *     lower block index, pads with -1 and returns ascending order.
 *
 * dtype codes: 0 = fp32, 1 = bf16 (raw 16-bit patterns).  Element values are
 * widened exactly to double.  All arrays are dense row-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_BF16 = 1 };

static double ld(const void* p, int dtype, size_t i) {
  if (dtype == OR_BF16) {
    uint32_t u = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
  }
  return (double)((const float*)p)[i];
}

/* Correctly rounded (nearest, ties to even) conversion of a double to bf16 bits,
 * done in one step so that no intermediate float rounding intervenes. */
static uint16_t to_bf16_bits(double x) {
  if (isnan(x)) return 0x7fc0;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int e;
  frexp(x, &e);             /* |x| = m * 2^e with 0.5 <= m < 1 */
  int q = e - 8;            /* bf16 carries 8 significant bits */
  if (q < -133) q = -133;   /* smallest bf16 subnormal is 2^-133 */
  double y = ldexp(nearbyint(ldexp(x, -q)), q);
  if (fabs(y) >= 0x1p128) return signbit(x) ? 0xff80 : 0x7f80;
  float f = (float)y;       /* exact: y has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static void st_rounded(void* p, int dtype, size_t i, double x) {
  if (dtype == OR_BF16)
    ((uint16_t*)p)[i] = to_bf16_bits(x);
  else
    ((float*)p)[i] = (float)x; /* C conversion rounds to nearest even */
}

int nsa_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Number of full compression windows in a sequence of length L. */
int nsa_oracle_num_cmp(int L, int kernel, int stride) {
  if (kernel <= 0 || stride <= 0 || L < kernel) return 0;
  return (L - kernel) / stride + 1;
}

/* Number of compressed keys that are causal for position t: c*s + l - 1 <= t. */
static int num_causal_cmp(int t, int n_c, int kernel, int stride) {
  if (t < kernel - 1) return 0;
  int n = (t - (kernel - 1)) / stride + 1;
  return n < n_c ? n : n_c;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Map a packed token index to its sequence by scanning cu_seqlens. */
static int seq_of(const int32_t* cu, int n_seqs, int64_t tok) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/* First compressed row of every sequence when compressed keys are packed
 * sequence after sequence (n_seqs+1 entries). */
static int64_t* cmp_offsets(const int32_t* cu, int n_seqs, int kernel, int stride) {
  int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_seqs + 1));
  off[0] = 0;
  for (int i = 0; i < n_seqs; ++i)
    off[i + 1] = off[i] + nsa_oracle_num_cmp(cu[i + 1] - cu[i], kernel, stride);
  return off;
}

/* ------------------------------------------------------------------------ */
/* S1: key compression.  [NOSA-Parts] core component 1 ("Key compressor"): cut the
 * keys into windows of `kernel` tokens at step `stride` and mean-pool each window;
 * [NOSA-Triton] "beyond the kernel" (kernel 32, stride 16, 50% overlap).  Windows
 * stay inside their sequence.  out_exact gets the fp64 mean, out_rounded the mean
 * rounded to the input dtype (the stored compressed key). */
int nsa_oracle_compress(const void* k, int dtype, const int32_t* cu, int n_seqs, int hkv, int d,
                        int kernel, int stride, double* out_exact, void* out_rounded) {
  if (kernel <= 0 || stride <= 0) return 1;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  for (int sq = 0; sq < n_seqs; ++sq) {
    int L = cu[sq + 1] - cu[sq];
    int n_c = nsa_oracle_num_cmp(L, kernel, stride);
#pragma omp parallel for schedule(static)
    for (int c = 0; c < n_c; ++c) {
      for (int g = 0; g < hkv; ++g) {
        for (int i = 0; i < d; ++i) {
          double acc = 0.0;
          for (int w = 0; w < kernel; ++w) {
            size_t tok = (size_t)cu[sq] + (size_t)c * stride + w;
            acc += ld(k, dtype, (tok * hkv + g) * d + i);
          }
          double mean = acc / kernel;
          size_t o = ((size_t)(off[sq] + c) * hkv + g) * d + i;
          if (out_exact) out_exact[o] = mean;
          if (out_rounded) st_rounded(out_rounded, dtype, o, mean);
        }
      }
    }
  }
  free(off);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* S2 for one query row and one kv-group: per head h of group g, the scores
 * z[h,c] = scale * q[t,h] . kc[c,g] over the causal compressed keys, a softmax
 * over them, and the group sum P_g[c] = sum_h p[h,c]  ([NSA-Triton] sec. 1.1:
 * selection reuses the compressed-attention scores; [NOSA-Parts] core component 3,
 * stage 1: a light attention of q against the compressed keys gives block scores).
 * pg receives n_c entries (zeros past the causal ones).  If o_cmp is non-NULL the
 * same probabilities also give the compressed-attention output of each head of
 * the group, o_cmp[(h - g*r)*d + i] = sum_c p[h,c] vc[c,g,i], and lse[h - g*r]. */
static void row_group_probs(const void* q, const void* kc, const void* vc, int dtype, int64_t tok,
                            int64_t kc_base, int n_c, int t, int h, int hkv, int d, int g,
                            int kernel, int stride, double scale, double* pg, double* z,
                            double* o_cmp, double* lse) {
  int r = h / hkv;
  int nca = num_causal_cmp(t, n_c, kernel, stride);
  for (int c = 0; c < n_c; ++c) pg[c] = 0.0;
  for (int hh = g * r; hh < (g + 1) * r; ++hh) {
    double* oc = o_cmp ? o_cmp + (size_t)(hh - g * r) * d : NULL;
    if (oc) for (int i = 0; i < d; ++i) oc[i] = 0.0;
    if (nca == 0) {
      if (lse) lse[hh - g * r] = -INFINITY;
      continue;
    }
    double mx = -INFINITY;
    for (int c = 0; c < nca; ++c) {
      double acc = 0.0;
      for (int i = 0; i < d; ++i)
        acc += ld(q, dtype, ((size_t)tok * h + hh) * d + i) *
               ld(kc, dtype, ((size_t)(kc_base + c) * hkv + g) * d + i);
      z[c] = acc * scale;
      if (z[c] > mx) mx = z[c];
    }
    double sum = 0.0;
    for (int c = 0; c < nca; ++c) sum += exp(z[c] - mx);
    for (int c = 0; c < nca; ++c) {
      double p = exp(z[c] - mx) / sum;
      pg[c] += p;
      if (oc)
        for (int i = 0; i < d; ++i) oc[i] += p * ld(vc, dtype, ((size_t)(kc_base + c) * hkv + g) * d + i);
    }
    if (lse) lse[hh - g * r] = mx + log(sum);
  }
}

/* S3 for one row: pooled block scores.  [NOSA-Triton] mechanisms 2 and 3: the
 * pooling kernel sums the scores of a window and divides by the number of valid
 * entries, the validity mask coming from the sequence length.  Block j pools the
 * compressed windows that lie inside it: {c : c*s >= jB and c*s + l <= (j+1)B},
 * restricted to existing windows c < n_c; empty -> 0. */
int nsa_oracle_pool_row(const double* pg, int n_c, int n_b, int block_size, int kernel, int stride,
                        double* out) {
  if (block_size <= 0 || kernel <= 0 || stride <= 0) return 1;
  for (int j = 0; j < n_b; ++j) {
    long first_tok = (long)j * block_size;           /* window must start here or later */
    long last_start = (long)(j + 1) * block_size - kernel; /* ... and start no later than this */
    double acc = 0.0;
    int cnt = 0;
    if (last_start >= first_tok) {
      long c_lo = (first_tok + stride - 1) / stride;
      long c_hi = last_start / stride;
      for (long c = c_lo; c <= c_hi; ++c) {
        if (c >= n_c) break;
        acc += pg[c];
        ++cnt;
      }
    }
    out[j] = cnt ? acc / cnt : 0.0;
  }
  return 0;
}

/* P_g for a set of rows: pg[row, g, c] (c < nc_stride; zero past n_c). */
int nsa_oracle_cmp_probs(const void* q, const void* kc, int dtype, const int32_t* cu, int n_seqs,
                         int h, int hkv, int d, int kernel, int stride, double scale,
                         const int64_t* rows, int64_t n_rows, double* pg, int nc_stride) {
  if (h % hkv) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  int err = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(nc_stride + 1));
    double* buf = (double*)malloc(sizeof(double) * (size_t)(nc_stride + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int L = cu[sq + 1] - cu[sq];
      int t = (int)(tok - cu[sq]);
      int n_c = nsa_oracle_num_cmp(L, kernel, stride);
      if (n_c > nc_stride) { err = 1; continue; }
      for (int g = 0; g < hkv; ++g) {
        row_group_probs(q, kc, NULL, dtype, tok, off[sq], n_c, t, h, hkv, d, g, kernel, stride,
                        scale, buf, z, NULL, NULL);
        double* dst = pg + ((size_t)rr * hkv + g) * nc_stride;
        for (int c = 0; c < nc_stride; ++c) dst[c] = c < n_c ? buf[c] : 0.0;
      }
    }
    free(z);
    free(buf);
  }
  free(off);
  return err;
}

/* S2+S3: pooled block scores scores[row, g, j] for j < nb_stride (zero past n_b(L)). */
int nsa_oracle_cmp_scores_pool(const void* q, const void* kc, int dtype, const int32_t* cu, int n_seqs,
                               int h, int hkv, int d, int kernel, int stride, int block_size,
                               double scale, const int64_t* rows, int64_t n_rows, double* scores,
                               int nb_stride) {
  if (h % hkv) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  int maxL = 0;
  for (int i = 0; i < n_seqs; ++i) if (cu[i + 1] - cu[i] > maxL) maxL = cu[i + 1] - cu[i];
  int nc_max = nsa_oracle_num_cmp(maxL, kernel, stride) + 1;
  int err = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* pg = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* sb = (double*)malloc(sizeof(double) * (size_t)(nb_stride + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int L = cu[sq + 1] - cu[sq];
      int t = (int)(tok - cu[sq]);
      int n_c = nsa_oracle_num_cmp(L, kernel, stride);
      int n_b = (L + block_size - 1) / block_size;
      if (n_b > nb_stride) { err = 1; continue; }
      for (int g = 0; g < hkv; ++g) {
        row_group_probs(q, kc, NULL, dtype, tok, off[sq], n_c, t, h, hkv, d, g, kernel, stride,
                        scale, pg, z, NULL, NULL);
        nsa_oracle_pool_row(pg, n_c, n_b, block_size, kernel, stride, sb);
        double* dst = scores + ((size_t)rr * hkv + g) * nb_stride;
        for (int j = 0; j < nb_stride; ++j) dst[j] = j < n_b ? sb[j] : 0.0;
      }
    }
    free(z);
    free(pg);
    free(sb);
  }
  free(off);
  return err;
}

/* ------------------------------------------------------------------------ */
/* S4 for one row.  [NOSA-Triton] "beyond the kernel: how the sliding window and
 * top-k cooperate": keep init_blocks + local_blocks + selected candidates, fill the
 * rest with -inf, take the top-k, and hand the indices on in sorted order.  Forced
 * blocks score +inf; only blocks j with j*B <= t are candidates; order is by score,
 * descending, then by lower block index.  k counts the forced blocks. */
typedef struct { double key; int j; } cand_t;

static int cand_cmp(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->key > y->key) return -1;
  if (x->key < y->key) return 1;
  return (x->j > y->j) - (x->j < y->j);
}

static int int_cmp(const void* a, const void* b) {
  int x = *(const int*)a, y = *(const int*)b;
  return (x > y) - (x < y);
}

static void row_topk(const double* sc, int t, int block_size, int n_init, int n_local, int k,
                     int32_t* out, cand_t* cand, int* pick) {
  int own = t / block_size;
  int ncand = own + 1;
  for (int j = 0; j < ncand; ++j) {
    int forced = (j < n_init) || (j > own - n_local);
    cand[j].key = forced ? INFINITY : sc[j];
    cand[j].j = j;
  }
  qsort(cand, (size_t)ncand, sizeof(cand_t), cand_cmp);
  int take = k < ncand ? k : ncand;
  for (int i = 0; i < take; ++i) pick[i] = cand[i].j;
  qsort(pick, (size_t)take, sizeof(int), int_cmp);
  for (int i = 0; i < k; ++i) out[i] = i < take ? pick[i] : -1;
}

int nsa_oracle_topk(const double* scores, int nb_stride, const int32_t* cu, int n_seqs, int hkv,
                    int block_size, int n_init, int n_local, int k, const int64_t* rows,
                    int64_t n_rows, int32_t* idx) {
  if (k <= 0 || block_size <= 0) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int err = 0;
#pragma omp parallel
  {
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nb_stride + 1));
    int* pick = (int*)malloc(sizeof(int) * (size_t)(nb_stride + k + 1));
#pragma omp for schedule(dynamic, 64)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      if (t / block_size + 1 > nb_stride) { err = 1; continue; }
      for (int g = 0; g < hkv; ++g)
        row_topk(scores + ((size_t)rr * hkv + g) * nb_stride, t, block_size, n_init, n_local, k,
                 idx + ((size_t)rr * hkv + g) * k, cand, pick);
    }
    free(cand);
    free(pick);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Softmax attention of one query head over an explicit key list (two passes:
 * maximum, then normalised sum).  Empty list -> zero output, lse = -inf. */
static void attend_list(const void* q, const void* k, const void* v, int dtype, int64_t tok, int hh,
                        int h, int hkv, int d, int g, int64_t seq_start, const int* keys, int n,
                        double scale, double* s, double* o, double* lse) {
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double mx = -INFINITY;
  for (int e = 0; e < n; ++e) {
    double acc = 0.0;
    size_t kr = ((size_t)(seq_start + keys[e]) * hkv + g) * d;
    for (int i = 0; i < d; ++i) acc += ld(q, dtype, ((size_t)tok * h + hh) * d + i) * ld(k, dtype, kr + i);
    s[e] = acc * scale;
    if (s[e] > mx) mx = s[e];
  }
  double sum = 0.0;
  for (int e = 0; e < n; ++e) sum += exp(s[e] - mx);
  for (int e = 0; e < n; ++e) {
    double p = exp(s[e] - mx) / sum;
    size_t vr = ((size_t)(seq_start + keys[e]) * hkv + g) * d;
    for (int i = 0; i < d; ++i) o[i] += p * ld(v, dtype, vr + i);
  }
  *lse = mx + log(sum);
}

/* Key list of the selected blocks for query t.  [TileLang-NSA] sec. 2: block start
 * i_s = index * block_size, used only when 0 <= i_s <= t; inside a used block keys
 * past t are masked.  Every list entry is walked, so a repeated index counts twice. */
static int selected_keys(const int32_t* idx_row, int S, int block_size, int t, int* keys) {
  int n = 0;
  for (int e = 0; e < S; ++e) {
    long i = idx_row[e];
    if (i < 0 || i * (long)block_size > t) continue;
    for (long tau = i * block_size; tau < (i + 1) * (long)block_size && tau <= t; ++tau) keys[n++] = (int)tau;
  }
  return n;
}

/* S5: selected-block attention.  o[row, h, :], lse[row, h] (lse nullable). */
int nsa_oracle_sparse_attn(const void* q, const void* k, const void* v, int dtype, const int32_t* cu,
                           int n_seqs, int h, int hkv, int d, const int32_t* idx, int S,
                           int block_size, double scale, const int64_t* rows, int64_t n_rows,
                           double* o, double* lse) {
  if (h % hkv || block_size <= 0) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int r = h / hkv;
#pragma omp parallel
  {
    int* keys = (int*)malloc(sizeof(int) * (size_t)(S * block_size + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(S * block_size + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      for (int hh = 0; hh < h; ++hh) {
        int g = hh / r;
        int n = selected_keys(idx + ((size_t)tok * hkv + g) * S, S, block_size, t, keys);
        double l;
        attend_list(q, k, v, dtype, tok, hh, h, hkv, d, g, cu[sq], keys, n, scale, s,
                    o + ((size_t)rr * h + hh) * d, &l);
        if (lse) lse[(size_t)rr * h + hh] = l;
      }
    }
    free(keys);
    free(s);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward of S5: gradients of the selected-block attention with respect to q, k
 * and v for an upstream gradient dO.  The pages give the forward only ([TileLang-NSA]
 * sec. 2; the training claims of [NSA-Triton] sec. 4 need its gradient); this is the
 * derivative of that forward written out.  For one (token, head) with list keys
 * tau_1..tau_n (as in selected_keys, duplicates included):
 *   s_e = scale q . k_e,  p = softmax(s),  o = sum_e p_e v_e,
 *   dp_e = dO . v_e,  D = sum_e p_e dp_e  (= dO . o),  ds_e = p_e (dp_e - D),
 *   dq = scale sum_e ds_e k_e,  dk[tau_e] += scale ds_e q,  dv[tau_e] += p_e dO.
 * A row with no key contributes nothing.  When o_in (the forward output the caller
 * holds, same dtype as q; nullable) is given, D is taken as dO . o_in instead: the
 * gradient step then uses the stored output, as a training step does when it keeps
 * only the rounded forward output (D = dO . o is an identity of the exact forward).
 * dq [n_q_rows, h, d] for q_rows (every token when NULL; n_q_rows < 0 skips dq);
 * dk, dv [n_kv_rows, hkv, d] for the key rows kv_rows (every token when NULL;
 * n_kv_rows < 0 skips them).  Only tokens whose lists reach a requested key row are
 * visited for dk and dv.  Thread-private accumulators are summed in thread order. */
static void row_probs_grads(const void* q, const void* k, const void* v, const void* dout, const void* o_in,
                            int dtype, int64_t tok, int hh, int h, int hkv, int d, int g, int64_t seq_start,
                            const int* keys, int n, double scale, double* p, double* ds) {
  double mx = -INFINITY;
  for (int e = 0; e < n; ++e) {
    double acc = 0.0;
    size_t kr = ((size_t)(seq_start + keys[e]) * hkv + g) * d;
    for (int i = 0; i < d; ++i) acc += ld(q, dtype, ((size_t)tok * h + hh) * d + i) * ld(k, dtype, kr + i);
    p[e] = acc * scale;
    if (p[e] > mx) mx = p[e];
  }
  double sum = 0.0;
  for (int e = 0; e < n; ++e) sum += exp(p[e] - mx);
  for (int e = 0; e < n; ++e) p[e] = exp(p[e] - mx) / sum;
  double D = 0.0;
  for (int e = 0; e < n; ++e) {
    double acc = 0.0;
    size_t vr = ((size_t)(seq_start + keys[e]) * hkv + g) * d;
    for (int i = 0; i < d; ++i) acc += ld(dout, dtype, ((size_t)tok * h + hh) * d + i) * ld(v, dtype, vr + i);
    ds[e] = acc;  /* dp_e for now */
    D += p[e] * acc;
  }
  if (o_in) {
    D = 0.0;
    for (int i = 0; i < d; ++i)
      D += ld(dout, dtype, ((size_t)tok * h + hh) * d + i) * ld(o_in, dtype, ((size_t)tok * h + hh) * d + i);
  }
  for (int e = 0; e < n; ++e) ds[e] = p[e] * (ds[e] - D);
}

int nsa_oracle_sparse_attn_bwd(const void* q, const void* k, const void* v, const void* dout, const void* o_in,
                               int dtype,
                               const int32_t* cu, int n_seqs, int h, int hkv, int d, const int32_t* idx, int S,
                               int block_size, double scale, const int64_t* q_rows, int64_t n_q_rows, double* dq,
                               const int64_t* kv_rows, int64_t n_kv_rows, double* dk, double* dv) {
  if (h % hkv || block_size <= 0) return 1;
  const int64_t total = cu[n_seqs];
  const int r = h / hkv;
  const int max_keys = S * block_size + 1;
  if (n_q_rows >= 0 && !q_rows) n_q_rows = total;
  if (n_q_rows > 0) {
#pragma omp parallel
    {
      int* keys = (int*)malloc(sizeof(int) * (size_t)max_keys);
      double* p = (double*)malloc(sizeof(double) * (size_t)max_keys);
      double* ds = (double*)malloc(sizeof(double) * (size_t)max_keys);
#pragma omp for schedule(dynamic, 8)
      for (int64_t rr = 0; rr < n_q_rows; ++rr) {
        int64_t tok = q_rows ? q_rows[rr] : rr;
        int sq = seq_of(cu, n_seqs, tok);
        int t = (int)(tok - cu[sq]);
        for (int hh = 0; hh < h; ++hh) {
          int g = hh / r;
          double* out = dq + ((size_t)rr * h + hh) * d;
          for (int i = 0; i < d; ++i) out[i] = 0.0;
          int n = selected_keys(idx + ((size_t)tok * hkv + g) * S, S, block_size, t, keys);
          if (n == 0) continue;
          row_probs_grads(q, k, v, dout, o_in, dtype, tok, hh, h, hkv, d, g, cu[sq], keys, n, scale, p, ds);
          for (int e = 0; e < n; ++e) {
            size_t kr = ((size_t)(cu[sq] + keys[e]) * hkv + g) * d;
            for (int i = 0; i < d; ++i) out[i] += scale * ds[e] * ld(k, dtype, kr + i);
          }
        }
      }
      free(keys);
      free(p);
      free(ds);
    }
  }
  if (n_kv_rows >= 0 && !kv_rows) n_kv_rows = total;
  if (n_kv_rows <= 0) return 0;
  /* slot of every token as a requested key row (-1: not requested) */
  int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total + 1));
  if (!slot) return 2;
  for (int64_t i = 0; i < total; ++i) slot[i] = kv_rows ? -1 : i;
  if (kv_rows)
    for (int64_t i = 0; i < n_kv_rows; ++i) slot[kv_rows[i]] = i;
  const size_t acc_len = (size_t)n_kv_rows * hkv * d;
  for (size_t i = 0; i < acc_len; ++i) dk[i] = dv[i] = 0.0;
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  double* acc = (double*)calloc((size_t)nthr * 2 * acc_len, sizeof(double));
  if (!acc) {
    free(slot);
    return 2;
  }
#pragma omp parallel num_threads(nthr)
  {
    int me = 0;
#ifdef _OPENMP
    me = omp_get_thread_num();
#endif
    double* mdk = acc + (size_t)me * 2 * acc_len;
    double* mdv = mdk + acc_len;
    int* keys = (int*)malloc(sizeof(int) * (size_t)max_keys);
    double* p = (double*)malloc(sizeof(double) * (size_t)max_keys);
    double* ds = (double*)malloc(sizeof(double) * (size_t)max_keys);
#pragma omp for schedule(static)
    for (int64_t tok = 0; tok < total; ++tok) {
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      for (int g = 0; g < hkv; ++g) {
        int n = selected_keys(idx + ((size_t)tok * hkv + g) * S, S, block_size, t, keys);
        int hit = 0;
        for (int e = 0; e < n && !hit; ++e) hit = slot[cu[sq] + keys[e]] >= 0;
        if (!hit) continue;
        for (int hh = g * r; hh < (g + 1) * r; ++hh) {
          row_probs_grads(q, k, v, dout, o_in, dtype, tok, hh, h, hkv, d, g, cu[sq], keys, n, scale, p, ds);
          for (int e = 0; e < n; ++e) {
            int64_t sl = slot[cu[sq] + keys[e]];
            if (sl < 0) continue;
            double* ak = mdk + ((size_t)sl * hkv + g) * d;
            double* av = mdv + ((size_t)sl * hkv + g) * d;
            for (int i = 0; i < d; ++i) {
              ak[i] += scale * ds[e] * ld(q, dtype, ((size_t)tok * h + hh) * d + i);
              av[i] += p[e] * ld(dout, dtype, ((size_t)tok * h + hh) * d + i);
            }
          }
        }
      }
    }
    free(keys);
    free(p);
    free(ds);
  }
  for (int th = 0; th < nthr; ++th) {
    const double* mdk = acc + (size_t)th * 2 * acc_len;
    const double* mdv = mdk + acc_len;
    for (size_t i = 0; i < acc_len; ++i) {
      dk[i] += mdk[i];
      dv[i] += mdv[i];
    }
  }
  free(acc);
  free(slot);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* NOSA stage 2.  [NOSA-Parts] core component 2: a scorer gives every key position an
 * importance score (CIS; here an input, since the scorer is learned); [NOSA-Triton]
 * mechanisms 1-3: the scores are mean-pooled over windows of `kernel` positions at step
 * `stride`, aligned with the key compressor; [NOSA-Parts] core component 3: the pooled
 * scores are brought to the block granularity.  Window c of a sequence averages cis over
 * positions c*stride .. c*stride+kernel-1 (full windows only, n_c of them, as for the
 * compressed keys); block j averages the windows inside it exactly as S3 does.
 *   cis [tokens, hkv] (fp64 values); out [n_seqs, hkv, nb_stride], zero past n_b(L). */
int nsa_oracle_cis_block_scores(const double* cis, const int32_t* cu, int n_seqs, int hkv, int kernel, int stride,
                                int block_size, int nb_stride, double* out) {
  if (kernel <= 0 || stride <= 0 || block_size <= 0) return 1;
  int err = 0;
  for (int sq = 0; sq < n_seqs; ++sq) {
    const int L = cu[sq + 1] - cu[sq];
    const int n_c = nsa_oracle_num_cmp(L, kernel, stride);
    const int n_b = (L + block_size - 1) / block_size;
    if (n_b > nb_stride) {
      err = 1;
      continue;
    }
    double* win = (double*)malloc(sizeof(double) * (size_t)(n_c + 1));
    for (int g = 0; g < hkv; ++g) {
      for (int c = 0; c < n_c; ++c) {
        double acc = 0.0;
        for (int i = 0; i < kernel; ++i) acc += cis[((size_t)cu[sq] + (size_t)c * stride + i) * hkv + g];
        win[c] = acc / kernel;
      }
      double* row = out + ((size_t)sq * hkv + g) * nb_stride;
      for (int j = 0; j < nb_stride; ++j) row[j] = 0.0;
      nsa_oracle_pool_row(win, n_c, n_b, block_size, kernel, stride, row);
    }
    free(win);
  }
  return err;
}

/* NOSA two-stage selection ([NOSA-Parts] core component 3).  Stage 1 keeps, for each
 * (token, kv-head), the forced blocks and the best blocks by the attention block score:
 * S4 with k = qk_select.  Stage 2 ranks the kept blocks by the pooled CIS score of the
 * token's sequence and keeps the forced blocks and the best others up to k in total;
 * equal scores go to the lower block index; output ascending, -1 padded.
 *   cis_scores [n_seqs, hkv, nb_stride];  k <= qk_select. */
int nsa_oracle_topk_two_stage(const double* scores, int nb_stride, const double* cis_scores, const int32_t* cu,
                              int n_seqs, int hkv, int block_size, int n_init, int n_local, int qk_select, int k,
                              const int64_t* rows, int64_t n_rows, int32_t* idx) {
  if (k <= 0 || qk_select < k || block_size <= 0) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int err = 0;
#pragma omp parallel
  {
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nb_stride + 1));
    int* pick = (int*)malloc(sizeof(int) * (size_t)(nb_stride + qk_select + 1));
    int32_t* first = (int32_t*)malloc(sizeof(int32_t) * (size_t)qk_select);
#pragma omp for schedule(dynamic, 64)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      int own = t / block_size;
      if (own + 1 > nb_stride) {
        err = 1;
        continue;
      }
      for (int g = 0; g < hkv; ++g) {
        row_topk(scores + ((size_t)rr * hkv + g) * nb_stride, t, block_size, n_init, n_local, qk_select, first,
                 cand, pick);
        const double* cs = cis_scores + ((size_t)sq * hkv + g) * nb_stride;
        int n = 0;
        for (int i = 0; i < qk_select; ++i) {
          int j = first[i];
          if (j < 0) continue;
          int forced = (j < n_init) || (j > own - n_local);
          cand[n].key = forced ? INFINITY : cs[j];
          cand[n].j = j;
          ++n;
        }
        qsort(cand, (size_t)n, sizeof(cand_t), cand_cmp);
        int take = k < n ? k : n;
        for (int i = 0; i < take; ++i) pick[i] = cand[i].j;
        qsort(pick, (size_t)take, sizeof(int), int_cmp);
        int32_t* o = idx + ((size_t)rr * hkv + g) * k;
        for (int i = 0; i < k; ++i) o[i] = i < take ? pick[i] : -1;
      }
    }
    free(cand);
    free(pick);
    free(first);
  }
  return err;
}

/* NOSA sparse_forward ([NOSA-Parts] "decoding over only 64 KV blocks"): the values are
 * scaled by the CIS of their key (scaled_v = v * cis) and the result is divided by the
 * same attention applied to all-ones values scaled alike (the "fake" attention whose
 * output is the denominator).  With p the softmax over the listed keys and c_e the CIS
 * of key e this is o = sum_e p_e c_e v_e / sum_e p_e c_e.  lse (natural log) is
 * log sum_e exp(s_e) c_e.  A row whose weights sum to zero gets o = 0 and lse = -inf.
 *   cis [tokens, hkv] (fp64 values), read at the key's own row. */
int nsa_oracle_sparse_attn_cis(const void* q, const void* k, const void* v, int dtype, const double* cis,
                               const int32_t* cu, int n_seqs, int h, int hkv, int d, const int32_t* idx, int S,
                               int block_size, double scale, const int64_t* rows, int64_t n_rows, double* o,
                               double* lse) {
  if (h % hkv || block_size <= 0) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int r = h / hkv;
#pragma omp parallel
  {
    int* keys = (int*)malloc(sizeof(int) * (size_t)(S * block_size + 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(S * block_size + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      for (int hh = 0; hh < h; ++hh) {
        int g = hh / r;
        int n = selected_keys(idx + ((size_t)tok * hkv + g) * S, S, block_size, t, keys);
        double* out = o + ((size_t)rr * h + hh) * d;
        for (int i = 0; i < d; ++i) out[i] = 0.0;
        double mx = -INFINITY;
        for (int e = 0; e < n; ++e) {
          double acc = 0.0;
          size_t kr = ((size_t)(cu[sq] + keys[e]) * hkv + g) * d;
          for (int i = 0; i < d; ++i) acc += ld(q, dtype, ((size_t)tok * h + hh) * d + i) * ld(k, dtype, kr + i);
          w[e] = acc * scale;
          if (w[e] > mx) mx = w[e];
        }
        double sum = 0.0;
        for (int e = 0; e < n; ++e) {
          w[e] = exp(w[e] - mx) * cis[(size_t)(cu[sq] + keys[e]) * hkv + g];
          sum += w[e];
        }
        if (sum > 0.0) {
          for (int e = 0; e < n; ++e) {
            size_t vr = ((size_t)(cu[sq] + keys[e]) * hkv + g) * d;
            for (int i = 0; i < d; ++i) out[i] += w[e] / sum * ld(v, dtype, vr + i);
          }
        }
        if (lse) lse[(size_t)rr * h + hh] = sum > 0.0 ? mx + log(sum) : -INFINITY;
      }
    }
    free(keys);
    free(w);
  }
  return 0;
}

/* Block-mask sparse attention ([TileLang-NSA] sec. 1, block-sparse attention: the
 * attention matrix is cut into block x block tiles and a mask marks the active ones;
 * only active tiles are computed; is_causal keeps the lower triangle).  Dense layout:
 * B sequences of T tokens.  Query (b, t, head hh) attends the keys of every key block
 * kb with mask[b, hh, t / block, kb] != 0, restricted to keys <= t when causal.  A row
 * without any attended key gets o = 0 and lse = -inf (the pages leave it undefined).
 *   mask  uint8 [B, h, nqb, nkb] with nqb = nkb = ceil(T / block). */
int nsa_oracle_block_sparse_attn(const void* q, const void* k, const void* v, int dtype, int B, int T,
                                 int h, int hkv, int d, const uint8_t* mask, int block, int causal,
                                 double scale, const int64_t* rows, int64_t n_rows, double* o, double* lse) {
  if (h % hkv || block <= 0 || B < 0 || T < 0) return 1;
  const int nb = (T + block - 1) / block;
  if (!rows) n_rows = (int64_t)B * T;
  const int r = h / hkv;
#pragma omp parallel
  {
    int* keys = (int*)malloc(sizeof(int) * (size_t)(T + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(T + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      const int64_t tok = rows ? rows[rr] : rr;
      const int b = (int)(tok / T), t = (int)(tok % T);
      for (int hh = 0; hh < h; ++hh) {
        const uint8_t* mrow = mask + (((size_t)b * h + hh) * nb + t / block) * nb;
        int n = 0;
        for (int kb = 0; kb < nb; ++kb) {
          if (!mrow[kb]) continue;
          for (int tau = kb * block; tau < (kb + 1) * block && tau < T; ++tau)
            if (!causal || tau <= t) keys[n++] = tau;
        }
        double l;
        attend_list(q, k, v, dtype, tok, hh, h, hkv, d, hh / r, (int64_t)b * T, keys, n, scale, s,
                    o + ((size_t)rr * h + hh) * d, &l);
        if (lse) lse[(size_t)rr * h + hh] = l;
      }
    }
    free(keys);
    free(s);
  }
  return 0;
}

/* S8: sliding-window attention over keys max(0, t-window+1) .. t ([NSA-Triton]
 * sec. 1.1: the sliding branch looks at the most recent tokens). */
int nsa_oracle_swa(const void* q, const void* k, const void* v, int dtype, const int32_t* cu,
                   int n_seqs, int h, int hkv, int d, int window, double scale,
                   const int64_t* rows, int64_t n_rows, double* o, double* lse) {
  if (h % hkv || window <= 0) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int r = h / hkv;
#pragma omp parallel
  {
    int* keys = (int*)malloc(sizeof(int) * (size_t)(window + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(window + 1));
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      int lo = t - window + 1 > 0 ? t - window + 1 : 0;
      int n = 0;
      for (int tau = lo; tau <= t; ++tau) keys[n++] = tau;
      for (int hh = 0; hh < h; ++hh) {
        double l;
        attend_list(q, k, v, dtype, tok, hh, h, hkv, d, hh / r, cu[sq], keys, n, scale, s,
                    o + ((size_t)rr * h + hh) * d, &l);
        if (lse) lse[(size_t)rr * h + hh] = l;
      }
    }
    free(keys);
    free(s);
  }
  return 0;
}

/* S7: compressed-attention branch over stored compressed keys/values
 * ([NSA-Triton] sec. 1.1 and 2.2 taken as a definition): per head, softmax of
 * scale * q . kc[c] over the causal compressed keys, weighted sum of vc[c]. */
int nsa_oracle_cmp_attn(const void* q, const void* kc, const void* vc, int dtype, const int32_t* cu,
                        int n_seqs, int h, int hkv, int d, int kernel, int stride, double scale,
                        const int64_t* rows, int64_t n_rows, double* o, double* lse) {
  if (h % hkv) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int r = h / hkv;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  int maxL = 0;
  for (int i = 0; i < n_seqs; ++i) if (cu[i + 1] - cu[i] > maxL) maxL = cu[i + 1] - cu[i];
  int nc_max = nsa_oracle_num_cmp(maxL, kernel, stride) + 1;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* pg = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* oc = (double*)malloc(sizeof(double) * (size_t)r * d);
    double* lg = (double*)malloc(sizeof(double) * (size_t)r);
#pragma omp for schedule(dynamic, 16)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int L = cu[sq + 1] - cu[sq];
      int t = (int)(tok - cu[sq]);
      int n_c = nsa_oracle_num_cmp(L, kernel, stride);
      for (int g = 0; g < hkv; ++g) {
        row_group_probs(q, kc, vc, dtype, tok, off[sq], n_c, t, h, hkv, d, g, kernel, stride, scale,
                        pg, z, oc, lg);
        for (int j = 0; j < r; ++j) {
          memcpy(o + ((size_t)rr * h + g * r + j) * d, oc + (size_t)j * d, sizeof(double) * (size_t)d);
          if (lse) lse[(size_t)rr * h + g * r + j] = lg[j];
        }
      }
    }
    free(z);
    free(pg);
    free(oc);
    free(lg);
  }
  free(off);
  return 0;
}

/* Backward of S7 (the compressed branch), written as the derivative of the forward
 * above.  Per (token, head) row over its causal compressed keys c < n_causal(t):
 *   p_c = softmax_c(scale q . kc_c),  dp_c = dO . vc_c,  D = dO . o (o_in when given,
 *   else sum_c p_c dp_c),  ds_c = p_c (dp_c - D);
 *   dq = scale sum_c ds_c kc_c,  dkc[c] += scale ds_c q,  dvc[c] += p_c dO.
 * A row without causal compressed keys contributes nothing and gets dq = 0.
 * dq [n_q_rows, h, d] for q_rows (all when NULL; n_q_rows < 0 skips); dkc, dvc
 * [n_kv_rows, hkv, d] for the packed compressed rows kv_rows (all when NULL; n_kv_rows
 * < 0 skips).  Thread-private accumulators, summed in thread order. */
static int cmp_row_grads(const void* q, const void* kc, const void* vc, const void* dout, const void* o_in, int dtype,
                         int64_t tok, int hh, int h, int hkv, int d, int g, int64_t c0, int n, double scale,
                         double* p, double* ds) {
  if (n == 0) return 0;
  double mx = -INFINITY;
  for (int c = 0; c < n; ++c) {
    double acc = 0.0;
    size_t kr = ((size_t)(c0 + c) * hkv + g) * d;
    for (int i = 0; i < d; ++i) acc += ld(q, dtype, ((size_t)tok * h + hh) * d + i) * ld(kc, dtype, kr + i);
    p[c] = acc * scale;
    if (p[c] > mx) mx = p[c];
  }
  double sum = 0.0;
  for (int c = 0; c < n; ++c) sum += exp(p[c] - mx);
  double D = 0.0;
  for (int c = 0; c < n; ++c) {
    p[c] = exp(p[c] - mx) / sum;
    double acc = 0.0;
    size_t vr = ((size_t)(c0 + c) * hkv + g) * d;
    for (int i = 0; i < d; ++i) acc += ld(dout, dtype, ((size_t)tok * h + hh) * d + i) * ld(vc, dtype, vr + i);
    ds[c] = acc;
    D += p[c] * acc;
  }
  if (o_in) {
    D = 0.0;
    for (int i = 0; i < d; ++i)
      D += ld(dout, dtype, ((size_t)tok * h + hh) * d + i) * ld(o_in, dtype, ((size_t)tok * h + hh) * d + i);
  }
  for (int c = 0; c < n; ++c) ds[c] = p[c] * (ds[c] - D);
  return n;
}

int nsa_oracle_cmp_attn_bwd(const void* q, const void* kc, const void* vc, const void* dout, const void* o_in,
                            int dtype, const int32_t* cu, int n_seqs, int h, int hkv, int d, int kernel, int stride,
                            double scale, const int64_t* q_rows, int64_t n_q_rows, double* dq,
                            const int64_t* kv_rows, int64_t n_kv_rows, double* dkc, double* dvc) {
  if (h % hkv || kernel <= 0 || stride <= 0) return 1;
  const int64_t total = cu[n_seqs];
  const int r = h / hkv;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  const int64_t n_cmp = off[n_seqs];
  int maxL = 0;
  for (int i = 0; i < n_seqs; ++i) if (cu[i + 1] - cu[i] > maxL) maxL = cu[i + 1] - cu[i];
  const int nc_max = nsa_oracle_num_cmp(maxL, kernel, stride) + 1;
  if (n_q_rows >= 0 && !q_rows) n_q_rows = total;
  if (n_q_rows > 0) {
#pragma omp parallel
    {
      double* p = (double*)malloc(sizeof(double) * (size_t)nc_max);
      double* ds = (double*)malloc(sizeof(double) * (size_t)nc_max);
#pragma omp for schedule(dynamic, 8)
      for (int64_t rr = 0; rr < n_q_rows; ++rr) {
        int64_t tok = q_rows ? q_rows[rr] : rr;
        int sq = seq_of(cu, n_seqs, tok);
        int L = cu[sq + 1] - cu[sq];
        int t = (int)(tok - cu[sq]);
        int n = num_causal_cmp(t, nsa_oracle_num_cmp(L, kernel, stride), kernel, stride);
        for (int hh = 0; hh < h; ++hh) {
          int g = hh / r;
          double* out = dq + ((size_t)rr * h + hh) * d;
          for (int i = 0; i < d; ++i) out[i] = 0.0;
          if (!cmp_row_grads(q, kc, vc, dout, o_in, dtype, tok, hh, h, hkv, d, g, off[sq], n, scale, p, ds)) continue;
          for (int c = 0; c < n; ++c) {
            size_t kr = ((size_t)(off[sq] + c) * hkv + g) * d;
            for (int i = 0; i < d; ++i) out[i] += scale * ds[c] * ld(kc, dtype, kr + i);
          }
        }
      }
      free(p);
      free(ds);
    }
  }
  if (n_kv_rows >= 0 && !kv_rows) n_kv_rows = n_cmp;
  if (n_kv_rows <= 0) {
    free(off);
    return 0;
  }
  int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_cmp + 1));
  for (int64_t i = 0; i < n_cmp; ++i) slot[i] = kv_rows ? -1 : i;
  if (kv_rows)
    for (int64_t i = 0; i < n_kv_rows; ++i) slot[kv_rows[i]] = i;
  const size_t acc_len = (size_t)n_kv_rows * hkv * d;
  for (size_t i = 0; i < acc_len; ++i) dkc[i] = dvc[i] = 0.0;
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  double* acc = (double*)calloc((size_t)nthr * 2 * acc_len, sizeof(double));
#pragma omp parallel num_threads(nthr)
  {
    int me = 0;
#ifdef _OPENMP
    me = omp_get_thread_num();
#endif
    double* mk = acc + (size_t)me * 2 * acc_len;
    double* mv = mk + acc_len;
    double* p = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* ds = (double*)malloc(sizeof(double) * (size_t)nc_max);
#pragma omp for schedule(static)
    for (int64_t tok = 0; tok < total; ++tok) {
      int sq = seq_of(cu, n_seqs, tok);
      int L = cu[sq + 1] - cu[sq];
      int t = (int)(tok - cu[sq]);
      int n = num_causal_cmp(t, nsa_oracle_num_cmp(L, kernel, stride), kernel, stride);
      int hit = 0;
      for (int c = 0; c < n && !hit; ++c) hit = slot[off[sq] + c] >= 0;
      if (!hit) continue;
      for (int hh = 0; hh < h; ++hh) {
        int g = hh / r;
        cmp_row_grads(q, kc, vc, dout, o_in, dtype, tok, hh, h, hkv, d, g, off[sq], n, scale, p, ds);
        for (int c = 0; c < n; ++c) {
          int64_t sl = slot[off[sq] + c];
          if (sl < 0) continue;
          double* ak = mk + ((size_t)sl * hkv + g) * d;
          double* av = mv + ((size_t)sl * hkv + g) * d;
          for (int i = 0; i < d; ++i) {
            ak[i] += scale * ds[c] * ld(q, dtype, ((size_t)tok * h + hh) * d + i);
            av[i] += p[c] * ld(dout, dtype, ((size_t)tok * h + hh) * d + i);
          }
        }
      }
    }
    free(p);
    free(ds);
  }
  for (int th = 0; th < nthr; ++th) {
    const double* mk = acc + (size_t)th * 2 * acc_len;
    const double* mv = mk + acc_len;
    for (size_t i = 0; i < acc_len; ++i) {
      dkc[i] += mk[i];
      dvc[i] += mv[i];
    }
  }
  free(acc);
  free(slot);
  free(off);
  return 0;
}

/* Backward of S1 (the mean pooling): the gradient of every token row is the sum, over
 * the compressed windows that contain it, of the window's gradient divided by the window
 * length.  dkc [n_cmp_total, hkv, d] fp64 in; dk [tokens, hkv, d] fp64 out. */
int nsa_oracle_compress_bwd(const double* dkc, const int32_t* cu, int n_seqs, int hkv, int d, int kernel, int stride,
                            double* dk) {
  if (kernel <= 0 || stride <= 0) return 1;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  const int64_t total = cu[n_seqs];
  for (size_t i = 0; i < (size_t)total * hkv * d; ++i) dk[i] = 0.0;
  for (int sq = 0; sq < n_seqs; ++sq) {
    int L = cu[sq + 1] - cu[sq];
    int n_c = nsa_oracle_num_cmp(L, kernel, stride);
    for (int c = 0; c < n_c; ++c)
      for (int w = 0; w < kernel; ++w) {
        size_t tok = (size_t)cu[sq] + (size_t)c * stride + w;
        for (int g = 0; g < hkv; ++g)
          for (int i = 0; i < d; ++i)
            dk[(tok * hkv + g) * d + i] += dkc[((size_t)(off[sq] + c) * hkv + g) * d + i] / kernel;
      }
  }
  free(off);
  return 0;
}

/* S9: gate combine ([NSA-Triton] sec. 1.1: gates[0]*compressed + gates[1]*selected
 * + gates[2]*local), each gate the logistic sigmoid of its logit;
 * gates is [tokens, h, 3] fp32. */
int nsa_oracle_gate_combine(const double* o_cmp, const double* o_slc, const double* o_swa,
                            const float* gates, int64_t n_rows, int h, int d, double* o) {
#pragma omp parallel for schedule(static)
  for (int64_t rr = 0; rr < n_rows; ++rr)
    for (int hh = 0; hh < h; ++hh) {
      size_t gi = ((size_t)rr * h + hh) * 3;
      double g0 = sigmoid(gates[gi]), g1 = sigmoid(gates[gi + 1]), g2 = sigmoid(gates[gi + 2]);
      for (int i = 0; i < d; ++i) {
        size_t x = ((size_t)rr * h + hh) * d + i;
        o[x] = g0 * o_cmp[x] + g1 * o_slc[x] + g2 * o_swa[x];
      }
    }
  return 0;
}

/* Backward of S8 (the sliding window): the derivative of the forward above; per (token,
 * head) row over keys max(0, t-window+1) .. t, with the formulas of the S5 backward
 * (row_probs_grads; D = dO . o_in when o_in is given).  dq for q_rows (all when NULL;
 * n_q_rows < 0 skips), dk / dv for the token rows kv_rows (all when NULL; n_kv_rows < 0
 * skips); thread-private accumulators summed in thread order. */
int nsa_oracle_swa_bwd(const void* q, const void* k, const void* v, const void* dout, const void* o_in, int dtype,
                       const int32_t* cu, int n_seqs, int h, int hkv, int d, int window, double scale,
                       const int64_t* q_rows, int64_t n_q_rows, double* dq, const int64_t* kv_rows,
                       int64_t n_kv_rows, double* dk, double* dv) {
  if (h % hkv || window <= 0) return 1;
  const int64_t total = cu[n_seqs];
  const int r = h / hkv;
  if (n_q_rows >= 0 && !q_rows) n_q_rows = total;
  if (n_q_rows > 0) {
#pragma omp parallel
    {
      int* keys = (int*)malloc(sizeof(int) * (size_t)(window + 1));
      double* p = (double*)malloc(sizeof(double) * (size_t)(window + 1));
      double* ds = (double*)malloc(sizeof(double) * (size_t)(window + 1));
#pragma omp for schedule(dynamic, 8)
      for (int64_t rr = 0; rr < n_q_rows; ++rr) {
        int64_t tok = q_rows ? q_rows[rr] : rr;
        int sq = seq_of(cu, n_seqs, tok);
        int t = (int)(tok - cu[sq]);
        int lo = t - window + 1 > 0 ? t - window + 1 : 0, n = 0;
        for (int tau = lo; tau <= t; ++tau) keys[n++] = tau;
        for (int hh = 0; hh < h; ++hh) {
          int g = hh / r;
          double* out = dq + ((size_t)rr * h + hh) * d;
          for (int i = 0; i < d; ++i) out[i] = 0.0;
          row_probs_grads(q, k, v, dout, o_in, dtype, tok, hh, h, hkv, d, g, cu[sq], keys, n, scale, p, ds);
          for (int e = 0; e < n; ++e) {
            size_t kr = ((size_t)(cu[sq] + keys[e]) * hkv + g) * d;
            for (int i = 0; i < d; ++i) out[i] += scale * ds[e] * ld(k, dtype, kr + i);
          }
        }
      }
      free(keys);
      free(p);
      free(ds);
    }
  }
  if (n_kv_rows >= 0 && !kv_rows) n_kv_rows = total;
  if (n_kv_rows <= 0) return 0;
  int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(total + 1));
  for (int64_t i = 0; i < total; ++i) slot[i] = kv_rows ? -1 : i;
  if (kv_rows)
    for (int64_t i = 0; i < n_kv_rows; ++i) slot[kv_rows[i]] = i;
  const size_t acc_len = (size_t)n_kv_rows * hkv * d;
  for (size_t i = 0; i < acc_len; ++i) dk[i] = dv[i] = 0.0;
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  double* acc = (double*)calloc((size_t)nthr * 2 * acc_len, sizeof(double));
#pragma omp parallel num_threads(nthr)
  {
    int me = 0;
#ifdef _OPENMP
    me = omp_get_thread_num();
#endif
    double* mk = acc + (size_t)me * 2 * acc_len;
    double* mv = mk + acc_len;
    int* keys = (int*)malloc(sizeof(int) * (size_t)(window + 1));
    double* p = (double*)malloc(sizeof(double) * (size_t)(window + 1));
    double* ds = (double*)malloc(sizeof(double) * (size_t)(window + 1));
#pragma omp for schedule(static)
    for (int64_t tok = 0; tok < total; ++tok) {
      int sq = seq_of(cu, n_seqs, tok);
      int t = (int)(tok - cu[sq]);
      int lo = t - window + 1 > 0 ? t - window + 1 : 0, n = 0, hit = 0;
      for (int tau = lo; tau <= t; ++tau) {
        keys[n++] = tau;
        hit |= slot[cu[sq] + tau] >= 0;
      }
      if (!hit) continue;
      for (int hh = 0; hh < h; ++hh) {
        int g = hh / r;
        row_probs_grads(q, k, v, dout, o_in, dtype, tok, hh, h, hkv, d, g, cu[sq], keys, n, scale, p, ds);
        for (int e = 0; e < n; ++e) {
          int64_t sl = slot[cu[sq] + keys[e]];
          if (sl < 0) continue;
          double* ak = mk + ((size_t)sl * hkv + g) * d;
          double* av = mv + ((size_t)sl * hkv + g) * d;
          for (int i = 0; i < d; ++i) {
            ak[i] += scale * ds[e] * ld(q, dtype, ((size_t)tok * h + hh) * d + i);
            av[i] += p[e] * ld(dout, dtype, ((size_t)tok * h + hh) * d + i);
          }
        }
      }
    }
    free(keys);
    free(p);
    free(ds);
  }
  for (int th = 0; th < nthr; ++th) {
    const double* mk = acc + (size_t)th * 2 * acc_len;
    const double* mv = mk + acc_len;
    for (size_t i = 0; i < acc_len; ++i) {
      dk[i] += mk[i];
      dv[i] += mv[i];
    }
  }
  free(acc);
  free(slot);
  return 0;
}

/* Backward of S9: with g_i = sigmoid(a_i) and o = sum_i g_i o_i, the branch gradients
 * are g_i dO and the logit gradients g_i (1 - g_i) (dO . o_i), per (token, head). */
int nsa_oracle_gate_bwd(const double* o_cmp, const double* o_slc, const double* o_swa, const float* gates,
                        const double* dout, int64_t n_rows, int h, int d, double* d_cmp, double* d_slc,
                        double* d_swa, double* d_gates) {
#pragma omp parallel for schedule(static)
  for (int64_t rr = 0; rr < n_rows; ++rr)
    for (int hh = 0; hh < h; ++hh) {
      size_t gi = ((size_t)rr * h + hh) * 3;
      const double* br[3] = {o_cmp, o_slc, o_swa};
      double* db[3] = {d_cmp, d_slc, d_swa};
      for (int b = 0; b < 3; ++b) {
        double g = sigmoid(gates[gi + b]), dot = 0.0;
        for (int i = 0; i < d; ++i) {
          size_t x = ((size_t)rr * h + hh) * d + i;
          db[b][x] = g * dout[x];
          dot += dout[x] * br[b][x];
        }
        d_gates[gi + b] = g * (1.0 - g) * dot;
      }
    }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* S6: one decode step.  [NOSA-Parts] "how decoding uses only 64 KV blocks": the
 * newest query (position L-1; the cache already holds its key and value) is scored
 * against the compressed keys, the pooled block scores choose k blocks, and
 * attention runs over the chosen blocks only.
 *   q [B, h, d]; k_cache, v_cache [B, max_len, hkv, d]; kc_cache [B, nc_stride, hkv, d]
 *   with the first n_c(L_b) rows valid.  idx [B, hkv, k] out.  idx_in (nullable)
 *   overrides the selection used for attention.  o [B, h, d].  scores (nullable)
 *   [B, hkv, nb_stride] receives the pooled block scores. */
int nsa_oracle_decode(const void* q, const void* k_cache, const void* v_cache, const void* kc_cache,
                      int dtype, int B, const int32_t* seqlens, int max_len, int h, int hkv, int d,
                      int kernel, int stride, int block_size, int n_init, int n_local, int k,
                      double scale, const int32_t* idx_in, int32_t* idx, double* o, double* scores,
                      int nb_stride) {
  if (h % hkv) return 1;
  int r = h / hkv;
  int nc_stride = nsa_oracle_num_cmp(max_len, kernel, stride);
  int nb_max = (max_len + block_size - 1) / block_size;
  if (scores && nb_stride < nb_max) return 1;
  int err = 0;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(nc_stride + 1));
    double* pg = (double*)malloc(sizeof(double) * (size_t)(nc_stride + 1));
    double* sb = (double*)malloc(sizeof(double) * (size_t)(nb_max + 1));
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)(nb_max + 1));
    int* pick = (int*)malloc(sizeof(int) * (size_t)(nb_max + k + 1));
    int* keys = (int*)malloc(sizeof(int) * (size_t)(k * block_size + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(k * block_size + 1));
#pragma omp for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
      int L = seqlens[b];
      if (L < 1 || L > max_len) { err = 1; continue; }
      int t = L - 1;
      int n_c = nsa_oracle_num_cmp(L, kernel, stride);
      int n_b = (L + block_size - 1) / block_size;
      for (int g = 0; g < hkv; ++g) {
        /* the q row of sequence b is token b of a [B, h, d] array; the caches are
         * sequences of stride max_len (compressed: nc_stride) */
        for (int c = 0; c < n_c; ++c) pg[c] = 0.0;
        int nca = num_causal_cmp(t, n_c, kernel, stride);
        for (int hh = g * r; hh < (g + 1) * r && nca > 0; ++hh) {
          double mx = -INFINITY;
          for (int c = 0; c < nca; ++c) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
              acc += ld(q, dtype, ((size_t)b * h + hh) * d + i) *
                     ld(kc_cache, dtype, (((size_t)b * nc_stride + c) * hkv + g) * d + i);
            z[c] = acc * scale;
            if (z[c] > mx) mx = z[c];
          }
          double sum = 0.0;
          for (int c = 0; c < nca; ++c) sum += exp(z[c] - mx);
          for (int c = 0; c < nca; ++c) pg[c] += exp(z[c] - mx) / sum;
        }
        nsa_oracle_pool_row(pg, n_c, n_b, block_size, kernel, stride, sb);
        if (scores)
          for (int j = 0; j < nb_stride; ++j) scores[((size_t)b * hkv + g) * nb_stride + j] = j < n_b ? sb[j] : 0.0;
        int32_t* ir = idx + ((size_t)b * hkv + g) * k;
        row_topk(sb, t, block_size, n_init, n_local, k, ir, cand, pick);
        const int32_t* use = idx_in ? idx_in + ((size_t)b * hkv + g) * k : ir;
        int n = selected_keys(use, k, block_size, t, keys);
        for (int hh = g * r; hh < (g + 1) * r; ++hh) {
          double l;
          /* k/v caches: token tau of sequence b is row b*max_len + tau */
          attend_list(q, k_cache, v_cache, dtype, b, hh, h, hkv, d, g, (int64_t)b * max_len, keys, n,
                      scale, s, o + ((size_t)b * h + hh) * d, &l);
        }
      }
    }
    free(z); free(pg); free(sb); free(cand); free(pick); free(keys); free(s);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Full three-branch layer ([NSA-Triton] sec. 1.1): compressed attention over the
 * mean-pooled keys and values, selected-block attention over the blocks chosen
 * from the same compressed probabilities, sliding-window attention, and the gated
 * sum.  Compressed keys/values are rounded to the input dtype as stored values.
 * idx_in (nullable, [tokens, hkv, S]) overrides the selection for the selected
 * branch.  Outputs are per requested row: idx [n_rows, hkv, S], o and the three
 * branch outputs [n_rows, h, d] (branch outputs nullable). */
int nsa_oracle_layer(const void* q, const void* k, const void* v, const float* gates, int dtype,
                     const int32_t* cu, int n_seqs, int h, int hkv, int d, int kernel, int stride,
                     int block_size, int S, int n_init, int n_local, int window, double scale,
                     const int32_t* idx_in, const int64_t* rows, int64_t n_rows, int32_t* idx,
                     double* o, double* o_cmp_out, double* o_slc_out, double* o_swa_out) {
  if (h % hkv) return 1;
  int64_t total = cu[n_seqs];
  if (!rows) n_rows = total;
  int r = h / hkv;
  int64_t* off = cmp_offsets(cu, n_seqs, kernel, stride);
  size_t ncr = (size_t)off[n_seqs];
  size_t esz = dtype == OR_BF16 ? 2 : 4;
  void* kc = malloc(esz * (ncr * hkv * d + 1));
  void* vc = malloc(esz * (ncr * hkv * d + 1));
  nsa_oracle_compress(k, dtype, cu, n_seqs, hkv, d, kernel, stride, NULL, kc);
  nsa_oracle_compress(v, dtype, cu, n_seqs, hkv, d, kernel, stride, NULL, vc);
  int maxL = 0;
  for (int i = 0; i < n_seqs; ++i) if (cu[i + 1] - cu[i] > maxL) maxL = cu[i + 1] - cu[i];
  int nc_max = nsa_oracle_num_cmp(maxL, kernel, stride) + 1;
  int nb_max = (maxL + block_size - 1) / block_size + 1;
  int nkeys = (S * block_size > window ? S * block_size : window) + 1;
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* pg = (double*)malloc(sizeof(double) * (size_t)nc_max);
    double* sb = (double*)malloc(sizeof(double) * (size_t)nb_max);
    double* oc = (double*)malloc(sizeof(double) * (size_t)r * d);
    double* lg = (double*)malloc(sizeof(double) * (size_t)r);
    double* os = (double*)malloc(sizeof(double) * (size_t)d);
    double* ow = (double*)malloc(sizeof(double) * (size_t)d);
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)nb_max);
    int* pick = (int*)malloc(sizeof(int) * (size_t)(nb_max + S + 1));
    int* keys = (int*)malloc(sizeof(int) * (size_t)nkeys);
    int* wkeys = (int*)malloc(sizeof(int) * (size_t)nkeys);
    double* s = (double*)malloc(sizeof(double) * (size_t)nkeys);
#pragma omp for schedule(dynamic, 4)
    for (int64_t rr = 0; rr < n_rows; ++rr) {
      int64_t tok = rows ? rows[rr] : rr;
      int sq = seq_of(cu, n_seqs, tok);
      int L = cu[sq + 1] - cu[sq];
      int t = (int)(tok - cu[sq]);
      int n_c = nsa_oracle_num_cmp(L, kernel, stride);
      int n_b = (L + block_size - 1) / block_size;
      int lo = t - window + 1 > 0 ? t - window + 1 : 0;
      int nw = 0;
      for (int tau = lo; tau <= t; ++tau) wkeys[nw++] = tau;
      for (int g = 0; g < hkv; ++g) {
        row_group_probs(q, kc, vc, dtype, tok, off[sq], n_c, t, h, hkv, d, g, kernel, stride, scale,
                        pg, z, oc, lg);
        nsa_oracle_pool_row(pg, n_c, n_b, block_size, kernel, stride, sb);
        int32_t* ir = idx + ((size_t)rr * hkv + g) * S;
        row_topk(sb, t, block_size, n_init, n_local, S, ir, cand, pick);
        const int32_t* use = idx_in ? idx_in + ((size_t)tok * hkv + g) * S : ir;
        int n = selected_keys(use, S, block_size, t, keys);
        for (int j = 0; j < r; ++j) {
          int hh = g * r + j;
          double l;
          attend_list(q, k, v, dtype, tok, hh, h, hkv, d, g, cu[sq], keys, n, scale, s, os, &l);
          attend_list(q, k, v, dtype, tok, hh, h, hkv, d, g, cu[sq], wkeys, nw, scale, s, ow, &l);
          size_t gi = ((size_t)tok * h + hh) * 3;
          double g0 = sigmoid(gates[gi]), g1 = sigmoid(gates[gi + 1]), g2 = sigmoid(gates[gi + 2]);
          size_t base = ((size_t)rr * h + hh) * d;
          for (int i = 0; i < d; ++i) {
            double xc = oc[(size_t)j * d + i];
            o[base + i] = g0 * xc + g1 * os[i] + g2 * ow[i];
            if (o_cmp_out) o_cmp_out[base + i] = xc;
            if (o_slc_out) o_slc_out[base + i] = os[i];
            if (o_swa_out) o_swa_out[base + i] = ow[i];
          }
        }
      }
    }
    free(z); free(pg); free(sb); free(oc); free(lg); free(os); free(ow);
    free(cand); free(pick); free(keys); free(wkeys); free(s);
  }
  free(kc);
  free(vc);
  free(off);
  return 0;
}
