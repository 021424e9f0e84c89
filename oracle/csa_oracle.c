/*
 * csa_oracle.c -- plain CPU oracle for the compressed sparse attention
 * forward (DeepSeek-V4 CSA / HCA / window-only layers).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite,
 * the package smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * Every function evaluates the plain definition, in double precision, one
 * query (or one compressed entry) at a time.  Inputs are the exact values the
 * GPU receives (bf16 values widened to float, or float parameters).  Loops
 * over independent queries are spread over OpenMP threads when the compiler
 * supports it; the arithmetic of each query is sequential.
 *
 * Sources (page title, section):
 *   "DeepSeek-V4 Attention Training Systems" (Megatron V4 notes):
 *     §2  phase table: dense mode / sparse warm-up / sparse mode;
 *     §3  indexer KL loss  L_I = sum_t KL(Softmax(a_{t,C_t}) || Softmax(i_{t,C_t}));
 *     §4  THD packing, n_b = floor(L_b / r), reset list at sample boundaries;
 *     §5.1 compression spans D_compress = 8 (overlapping r=4) and 128 (HCA),
 *          local window D_window = 128;
 *     §8.2 kernel map: learned-score compressor reduction, indexer score +
 *          top-k, selected attention returning output and LSE, compressed
 *          ids combined with window ids;
 *     §9  precision table: FP32 compressor positional parameter, FP32
 *          attention sink, FP32 softmax / KL math.
 *
 * Readings taken where the pages leave a step open (each is listed in the
 * design notes and pinned by the CPU tests where a pin exists):
 *   - compressor: per-channel softmax gate over the span, logits z + P[u];
 *     overlapping entry j spans blocks j-1 and j (2r tokens), the
 *     non-overlapping entry spans block j (r tokens); span positions before
 *     the sequence start are left out of the softmax (parity unpinned beyond
 *     "softmax-gated weighted sum" and the span widths);
 *   - indexer logit i_{t,j} = sum_h w[t,h] * ReLU(qI[t,h,:] . kI[j,:]);
 *   - top-k ties go to the smaller entry index; output ascending, -1 padded;
 *   - attention sink is a denominator-only logit; lse includes it;
 *   - teacher a_{t,j} = log of the head-averaged per-head softmax over C_t
 *     (parity unpinned: the pages do not say how heads are combined).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Sequence that owns packed row `row`: the b with cu[b] <= row < cu[b+1],
 * or -1 for capacity padding (row >= cu[B]).  §4: samples are concatenated on
 * one token axis and delimited by cu_seqlens. */
static int owner_sequence(const int32_t* cu, int B, int64_t row) {
  if (B <= 0 || row < cu[0] || row >= cu[B]) return -1;
  for (int b = 0; b < B; ++b)
    if (row >= cu[b] && row < cu[b + 1]) return b;
  return -1;
}

/* Number of compressed entries visible to local query position t:
 * entry j (tokens up to r(j+1)-1) is visible once r(j+1)-1 <= t  (§4 causal
 * visibility of completed compressed groups). */
static int64_t visible_count(int64_t t, int r) {
  if (r <= 0) return 0;
  return (t + 1) / r;
}

/* §4: only complete groups are compressed, n_b = floor(L_b / r).
 * cu_cmp[b] = sum_{b' < b} n_{b'}.  Returns cu_cmp[B]. */
int64_t oracle_compressed_offsets(const int32_t* cu, int B, int r, int32_t* cu_cmp) {
  cu_cmp[0] = 0;
  for (int b = 0; b < B; ++b) {
    int64_t L = (int64_t)cu[b + 1] - cu[b];
    int64_t n = r > 0 ? L / r : 0;
    cu_cmp[b + 1] = (int32_t)(cu_cmp[b] + n);
  }
  return cu_cmp[B];
}

/* Learned-score block compression (§4, §5.1, §8.2 "C4/C128 compression",
 * §9 FP32 positional parameter).
 *   x, z : [T, D] packed rows (values, gate logits)
 *   P    : [S, D] positional logit bias, S = 2r (overlap) or r
 *   out  : [N_c, D] compressed rows, double
 * Entry j of sequence b covers local tokens first .. first+S-1 with
 * first = r*j + r - S; positions before the start of the sequence are not
 * available and are left out of the per-channel softmax. */
void oracle_compress(const float* x, const float* z, const float* P,
                     const int32_t* cu, const int32_t* cu_cmp, int B, int D,
                     int r, int overlap, double* out) {
  const int S = overlap ? 2 * r : r;
  for (int b = 0; b < B; ++b) {
    const int64_t L = (int64_t)cu[b + 1] - cu[b];
    const int64_t n = r > 0 ? L / r : 0;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
      const int64_t first = (int64_t)r * j + r - S;
      for (int c = 0; c < D; ++c) {
        double m = -INFINITY;
        for (int u = 0; u < S; ++u) {
          const int64_t t = first + u;
          if (t < 0) continue;
          const double logit = (double)z[(cu[b] + t) * (int64_t)D + c] + (double)P[(int64_t)u * D + c];
          if (logit > m) m = logit;
        }
        double den = 0.0, num = 0.0;
        for (int u = 0; u < S; ++u) {
          const int64_t t = first + u;
          if (t < 0) continue;
          const double logit = (double)z[(cu[b] + t) * (int64_t)D + c] + (double)P[(int64_t)u * D + c];
          const double e = exp(logit - m);
          den += e;
          num += e * (double)x[(cu[b] + t) * (int64_t)D + c];
        }
        out[((int64_t)cu_cmp[b] + j) * D + c] = num / den;
      }
    }
  }
}

/* Compressor variant with the extras the pages list around the compressor
 * (§10 "compressor softmax and normalization intermediates"; §12 invariant 2
 * "RoPE mode is per layer and per compressed coordinate system"; §9 FP32
 * positional parameter).  Three steps, in this order, per compressed entry:
 *
 *  1. gate: the per-channel softmax-weighted sum of oracle_compress, except
 *     that with x_prev/z_prev given (overlapping spans only) span positions
 *     u < r -- the previous block -- read x_prev/z_prev and positions u >= r
 *     read x/z (two projections of the same tokens, one per half of the span);
 *  2. RMSNorm (when gamma is given): y <- y / sqrt(mean_c y_c^2 + eps) * gamma;
 *  3. RoPE (when rope_dim > 0) on the last rope_dim channels, as rope_dim/2
 *     interleaved pairs (2i, 2i+1) rotated by the angle p * theta^(-2i/rope_dim)
 *     (the rotary embedding of Su et al., "RoFormer", 2021), p = the entry's
 *     position in its sequence's compressed coordinates scaled as
 *     p = j * pos_stride + pos_offset.
 * Arguments as oracle_compress; x_prev, z_prev, gamma may be NULL. */
void oracle_compress_ex(const float* x, const float* z, const float* x_prev, const float* z_prev,
                        const float* P, const float* gamma, float eps, int rope_dim, double theta,
                        int64_t pos_stride, int64_t pos_offset, const int32_t* cu,
                        const int32_t* cu_cmp, int B, int D, int r, int overlap, double* out) {
  const int S = overlap ? 2 * r : r;
  const int two = overlap && x_prev != NULL && z_prev != NULL;
  for (int b = 0; b < B; ++b) {
    const int64_t L = (int64_t)cu[b + 1] - cu[b];
    const int64_t n = r > 0 ? L / r : 0;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) {
      double* y = out + ((int64_t)cu_cmp[b] + j) * D;
      const int64_t first = (int64_t)r * j + r - S;
      /* 1. softmax gate over the span */
      for (int c = 0; c < D; ++c) {
        double m = -INFINITY;
        for (int u = 0; u < S; ++u) {
          const int64_t t = first + u;
          if (t < 0) continue;
          const float* zs = (two && u < r) ? z_prev : z;
          const double logit = (double)zs[(cu[b] + t) * (int64_t)D + c] + (double)P[(int64_t)u * D + c];
          if (logit > m) m = logit;
        }
        double den = 0.0, num = 0.0;
        for (int u = 0; u < S; ++u) {
          const int64_t t = first + u;
          if (t < 0) continue;
          const float* zs = (two && u < r) ? z_prev : z;
          const float* xs = (two && u < r) ? x_prev : x;
          const double logit = (double)zs[(cu[b] + t) * (int64_t)D + c] + (double)P[(int64_t)u * D + c];
          const double e = exp(logit - m);
          den += e;
          num += e * (double)xs[(cu[b] + t) * (int64_t)D + c];
        }
        y[c] = num / den;
      }
      /* 2. RMSNorm over the D channels of the entry */
      if (gamma != NULL) {
        double ss = 0.0;
        for (int c = 0; c < D; ++c) ss += y[c] * y[c];
        const double rms = sqrt(ss / D + (double)eps);
        for (int c = 0; c < D; ++c) y[c] = y[c] / rms * (double)gamma[c];
      }
      /* 3. rotary embedding of the trailing rope_dim channels */
      if (rope_dim > 0) {
        const double p = (double)(j * pos_stride + pos_offset);
        for (int i = 0; i < rope_dim / 2; ++i) {
          const int c = D - rope_dim + 2 * i;
          const double ang = p * pow(theta, -(2.0 * i) / rope_dim);
          const double cs = cos(ang), sn = sin(ang);
          const double a = y[c], bb = y[c + 1];
          y[c] = a * cs - bb * sn;
          y[c + 1] = a * sn + bb * cs;
        }
      }
    }
  }
}

/* Lightning-indexer logits of one query against its visible entries
 * (§3 i_{t,j}; form sum_h w * ReLU(qI . kI)).  logits must hold nvis values. */
static void indexer_logits_one(const float* qI, const float* w, const float* kI,
                               int64_t row, int64_t cmp_base, int64_t nvis,
                               int H_I, int dI, double* logits) {
  for (int64_t j = 0; j < nvis; ++j) {
    double s = 0.0;
    for (int h = 0; h < H_I; ++h) {
      double dot = 0.0;
      for (int c = 0; c < dI; ++c)
        dot += (double)qI[(row * H_I + h) * (int64_t)dI + c] * (double)kI[(cmp_base + j) * dI + c];
      const double relu = dot > 0.0 ? dot : 0.0;
      s += (double)w[row * H_I + h] * relu;
    }
    logits[j] = s;
  }
}

/* Indexer logits for a list of query rows: logits[q*max_vis + j] for
 * j < nvis[q] (the rest left untouched). */
void oracle_indexer_logits(const float* qI, const float* w, const float* kI,
                           const int32_t* cu, const int32_t* cu_cmp, int B,
                           int H_I, int dI, int r, const int64_t* rows, int nq,
                           int64_t max_vis, double* logits, int32_t* nvis_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int q = 0; q < nq; ++q) {
    const int64_t row = rows[q];
    const int b = owner_sequence(cu, B, row);
    if (b < 0) { nvis_out[q] = 0; continue; }
    const int64_t t = row - cu[b];
    int64_t nvis = visible_count(t, r);
    if (nvis > max_vis) nvis = max_vis;
    nvis_out[q] = (int32_t)nvis;
    indexer_logits_one(qI, w, kI, row, cu_cmp[b], nvis, H_I, dI, logits + (int64_t)q * max_vis);
  }
}

typedef struct { double s; int64_t j; } scored_entry;

/* Larger score first; equal scores: smaller entry index first. */
static int by_score_then_index(const void* pa, const void* pb) {
  const scored_entry* a = (const scored_entry*)pa;
  const scored_entry* b = (const scored_entry*)pb;
  if (a->s > b->s) return -1;
  if (a->s < b->s) return 1;
  return (a->j > b->j) - (a->j < b->j);
}

/* Per-query top-k of the indexer logits (§8 "indexer scoring and radix
 * top-k", §8.2 flat global index list, §8.1 top-k padding).
 * idx[q*k_pad + i]: the min(topk, |V_t|) selected entries as global
 * compressed rows cu_cmp[b] + j in ascending j, then -1 up to k_pad.
 * Capacity rows (not in any sequence) get all -1. */
void oracle_indexer_topk(const float* qI, const float* w, const float* kI,
                         const int32_t* cu, const int32_t* cu_cmp, int B,
                         int H_I, int dI, int r, int topk, int k_pad,
                         const int64_t* rows, int nq, int32_t* idx) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int q = 0; q < nq; ++q) {
    int32_t* out = idx + (int64_t)q * k_pad;
    for (int i = 0; i < k_pad; ++i) out[i] = -1;
    const int64_t row = rows[q];
    const int b = owner_sequence(cu, B, row);
    if (b < 0) continue;
    const int64_t t = row - cu[b];
    const int64_t nvis = visible_count(t, r);
    if (nvis == 0) continue;
    double* logits = (double*)malloc(sizeof(double) * nvis);
    scored_entry* order = (scored_entry*)malloc(sizeof(scored_entry) * nvis);
    char* chosen = (char*)calloc((size_t)nvis, 1);
    indexer_logits_one(qI, w, kI, row, cu_cmp[b], nvis, H_I, dI, logits);
    for (int64_t j = 0; j < nvis; ++j) { order[j].s = logits[j]; order[j].j = j; }
    qsort(order, (size_t)nvis, sizeof(scored_entry), by_score_then_index);
    const int64_t m = nvis < topk ? nvis : topk;
    for (int64_t i = 0; i < m; ++i) chosen[order[i].j] = 1;
    int64_t k = 0;
    for (int64_t j = 0; j < nvis; ++j)
      if (chosen[j]) out[k++] = (int32_t)(cu_cmp[b] + j);
    free(chosen); free(order); free(logits);
  }
}

/* Attention kinds: which compressed entries join the candidate list. */
enum { ORACLE_CSA = 0, ORACLE_HCA = 1, ORACLE_WINDOW = 2 };

/* Selected / HCA / window-only attention forward for a list of query rows
 * (§2 phase table: top-k compressed entries + local window; HCA reads every
 * completed compressed entry + the window; window-only has no compressed
 * part; §8.2 FlashMLA returns output and LSE; §9 FP32 attention sink).
 *
 * One shared KV head (MQA): key rows kc (compressed) / kr (raw), value rows
 * vc / vr (pass the key arrays again when K = V).  Candidate list of query t
 * in sequence b: compressed rows (csa: the valid entries of idx row; hca: all
 * visible entries), then the window rows cu[b] + s for s in
 * [max(0, t-W+1), t].  Entries and window rows are distinct keys.
 * For each head h:
 *   s_i   = scale * q[t,h,:] . K_i
 *   m     = max(max_i s_i, sink_h)   (sink only when given)
 *   Z     = sum_i exp(s_i - m) + exp(sink_h - m)
 *   o     = sum_i exp(s_i - m) V_i / Z,   lse = m + log Z
 *   lse_cmp = logsumexp of s_i over the compressed candidates only
 *             (no sink, no window), -inf when there are none.
 * Capacity rows: o = 0, lse = lse_cmp = -inf.
 * err[q] = 1 when an idx entry lies outside the query's visible entries (the
 * entry is then skipped), else 0. */
void oracle_attention(int kind, const float* q, const float* kc, const float* vc,
                      const float* kr, const float* vr, const int32_t* idx,
                      int k_pad, const float* sink, const int32_t* cu,
                      const int32_t* cu_cmp, int B, int H, int d, int r, int W,
                      double scale, const int64_t* rows, int nq, double* o,
                      double* lse, double* lse_cmp, int32_t* err) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int qi = 0; qi < nq; ++qi) {
    const int64_t row = rows[qi];
    double* oq = o + (int64_t)qi * H * d;
    err[qi] = 0;
    const int b = owner_sequence(cu, B, row);
    if (b < 0) {
      for (int64_t e = 0; e < (int64_t)H * d; ++e) oq[e] = 0.0;
      for (int h = 0; h < H; ++h) { lse[(int64_t)qi * H + h] = -INFINITY; lse_cmp[(int64_t)qi * H + h] = -INFINITY; }
      continue;
    }
    const int64_t t = row - cu[b];
    const int64_t nvis = kind == ORACLE_WINDOW ? 0 : visible_count(t, r);
    /* compressed candidate rows */
    int64_t ncmp = 0;
    int64_t cap = kind == ORACLE_CSA ? k_pad : nvis;
    int64_t* crow = (int64_t*)malloc(sizeof(int64_t) * (cap > 0 ? cap : 1));
    if (kind == ORACLE_CSA) {
      for (int i = 0; i < k_pad; ++i) {
        const int64_t g = idx[row * (int64_t)k_pad + i];
        if (g < 0) continue;
        if (g < cu_cmp[b] || g >= cu_cmp[b] + nvis) { err[qi] = 1; continue; }
        crow[ncmp++] = g;
      }
    } else if (kind == ORACLE_HCA) {
      for (int64_t j = 0; j < nvis; ++j) crow[ncmp++] = cu_cmp[b] + j;
    }
    const int64_t w0 = t - W + 1 > 0 ? t - W + 1 : 0;
    const int64_t nwin = t - w0 + 1;
    const int64_t n = ncmp + nwin;
    double* s = (double*)malloc(sizeof(double) * n);
    for (int h = 0; h < H; ++h) {
      const float* qh = q + (row * H + h) * (int64_t)d;
      for (int64_t i = 0; i < n; ++i) {
        const float* kk = i < ncmp ? kc + crow[i] * d : kr + (cu[b] + w0 + (i - ncmp)) * (int64_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += (double)qh[c] * (double)kk[c];
        s[i] = scale * dot;
      }
      double m = -INFINITY;
      for (int64_t i = 0; i < n; ++i) if (s[i] > m) m = s[i];
      if (sink && (double)sink[h] > m) m = (double)sink[h];
      double Z = 0.0;
      for (int64_t i = 0; i < n; ++i) Z += exp(s[i] - m);
      if (sink) Z += exp((double)sink[h] - m);
      double* oh = oq + (int64_t)h * d;
      for (int c = 0; c < d; ++c) oh[c] = 0.0;
      for (int64_t i = 0; i < n; ++i) {
        const double p = exp(s[i] - m) / Z;
        const float* vv = i < ncmp ? vc + crow[i] * d : vr + (cu[b] + w0 + (i - ncmp)) * (int64_t)d;
        for (int c = 0; c < d; ++c) oh[c] += p * (double)vv[c];
      }
      lse[(int64_t)qi * H + h] = m + log(Z);
      if (ncmp == 0) {
        lse_cmp[(int64_t)qi * H + h] = -INFINITY;
      } else {
        double mc = -INFINITY;
        for (int64_t i = 0; i < ncmp; ++i) if (s[i] > mc) mc = s[i];
        double Zc = 0.0;
        for (int64_t i = 0; i < ncmp; ++i) Zc += exp(s[i] - mc);
        lse_cmp[(int64_t)qi * H + h] = mc + log(Zc);
      }
    }
    free(s);
    free(crow);
  }
}

/* Backward of oracle_attention for a list of query rows (§8.2 "main attention
 * backward": consumes saved output/LSE and produces Q, KV and attention-sink
 * gradients).  Given the upstream gradient dout = dL/do, for each query row t
 * and head h, with the candidate list, s_i, lse and o of oracle_attention:
 *   p_i      = exp(s_i - lse)                  (the attention weights)
 *   D        = sum_c dout[c] o[c]
 *   dp_i     = dout . V_i
 *   ds_i     = p_i (dp_i - D)                  (gradient of L w.r.t. s_i / scale)
 *   dq       = scale sum_i ds_i K_i
 *   dK_i    += scale ds_i q                    (accumulated over queries)
 *   dV_i    += p_i dout
 *   dsink_h += -exp(sink_h - lse) D            (the sink is a logit with no value)
 * These are the chain rule through o = sum_i p_i V_i and p = softmax(s, sink).
 * dq is [nq, H, d]; dkc/dvc are [rows of kc, d], dkr/dvr [rows of kr, d] and
 * dsink [H], all accumulated into (the caller zeroes them); any of dkc, dvc,
 * dkr, dvr, dsink may be NULL (not wanted).  Capacity rows contribute nothing
 * (dq = 0).  err[q] as in oracle_attention. */
void oracle_attention_bwd(int kind, const float* q, const float* kc, const float* vc,
                          const float* kr, const float* vr, const int32_t* idx, int k_pad,
                          const float* sink, const int32_t* cu, const int32_t* cu_cmp, int B, int H,
                          int d, int r, int W, double scale, const float* dout,
                          const int64_t* rows, int nq, double* dq, double* dkc, double* dvc,
                          double* dkr, double* dvr, double* dsink, int32_t* err) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int qi = 0; qi < nq; ++qi) {
    const int64_t row = rows[qi];
    double* dqq = dq + (int64_t)qi * H * d;
    for (int64_t e = 0; e < (int64_t)H * d; ++e) dqq[e] = 0.0;
    err[qi] = 0;
    const int b = owner_sequence(cu, B, row);
    if (b < 0) continue;
    const int64_t t = row - cu[b];
    const int64_t nvis = kind == ORACLE_WINDOW ? 0 : visible_count(t, r);
    int64_t ncmp = 0;
    const int64_t cap = kind == ORACLE_CSA ? k_pad : nvis;
    int64_t* crow = (int64_t*)malloc(sizeof(int64_t) * (cap > 0 ? cap : 1));
    if (kind == ORACLE_CSA) {
      for (int i = 0; i < k_pad; ++i) {
        const int64_t g = idx[row * (int64_t)k_pad + i];
        if (g < 0) continue;
        if (g < cu_cmp[b] || g >= cu_cmp[b] + nvis) { err[qi] = 1; continue; }
        crow[ncmp++] = g;
      }
    } else if (kind == ORACLE_HCA) {
      for (int64_t j = 0; j < nvis; ++j) crow[ncmp++] = cu_cmp[b] + j;
    }
    const int64_t w0 = t - W + 1 > 0 ? t - W + 1 : 0;
    const int64_t nwin = t - w0 + 1;
    const int64_t n = ncmp + nwin;
    double* s = (double*)malloc(sizeof(double) * n);
    double* p = (double*)malloc(sizeof(double) * n);
    double* ds = (double*)malloc(sizeof(double) * n);
    double* o = (double*)malloc(sizeof(double) * d);
    /* this row's contributions to the key / value gradients, merged at the end */
    double* gk = (double*)calloc((size_t)n * d, sizeof(double));
    double* gv = (double*)calloc((size_t)n * d, sizeof(double));
    double* gsink = (double*)calloc((size_t)H, sizeof(double));
    for (int h = 0; h < H; ++h) {
      const float* qh = q + (row * H + h) * (int64_t)d;
      const float* gh = dout + (row * H + h) * (int64_t)d;
      for (int64_t i = 0; i < n; ++i) {
        const float* kk = i < ncmp ? kc + crow[i] * d : kr + (cu[b] + w0 + (i - ncmp)) * (int64_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += (double)qh[c] * (double)kk[c];
        s[i] = scale * dot;
      }
      double m = -INFINITY;
      for (int64_t i = 0; i < n; ++i) if (s[i] > m) m = s[i];
      if (sink && (double)sink[h] > m) m = (double)sink[h];
      double Z = 0.0;
      for (int64_t i = 0; i < n; ++i) Z += exp(s[i] - m);
      if (sink) Z += exp((double)sink[h] - m);
      const double lse = m + log(Z);
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int64_t i = 0; i < n; ++i) {
        p[i] = exp(s[i] - lse);
        const float* vv = i < ncmp ? vc + crow[i] * d : vr + (cu[b] + w0 + (i - ncmp)) * (int64_t)d;
        for (int c = 0; c < d; ++c) o[c] += p[i] * (double)vv[c];
      }
      double D = 0.0;
      for (int c = 0; c < d; ++c) D += (double)gh[c] * o[c];
      for (int64_t i = 0; i < n; ++i) {
        const float* vv = i < ncmp ? vc + crow[i] * d : vr + (cu[b] + w0 + (i - ncmp)) * (int64_t)d;
        double dp = 0.0;
        for (int c = 0; c < d; ++c) dp += (double)gh[c] * (double)vv[c];
        ds[i] = p[i] * (dp - D);
      }
      double* dqh = dqq + (int64_t)h * d;
      for (int64_t i = 0; i < n; ++i) {
        const float* kk = i < ncmp ? kc + crow[i] * d : kr + (cu[b] + w0 + (i - ncmp)) * (int64_t)d;
        for (int c = 0; c < d; ++c) {
          dqh[c] += scale * ds[i] * (double)kk[c];
          gk[i * d + c] += scale * ds[i] * (double)qh[c];
          gv[i * d + c] += p[i] * (double)gh[c];
        }
      }
      if (sink) gsink[h] = -exp((double)sink[h] - lse) * D;
    }
#pragma omp critical(oracle_attention_bwd_merge)
    {
      for (int64_t i = 0; i < n; ++i) {
        const int64_t krow = i < ncmp ? crow[i] : cu[b] + w0 + (i - ncmp);
        double* dk = i < ncmp ? dkc : dkr;
        double* dv = i < ncmp ? dvc : dvr;
        for (int c = 0; c < d; ++c) {
          if (dk) dk[krow * d + c] += gk[i * d + c];
          if (dv) dv[krow * d + c] += gv[i * d + c];
        }
      }
      if (dsink && sink)
        for (int h = 0; h < H; ++h) dsink[h] += gsink[h];
    }
    free(gsink); free(gv); free(gk); free(o); free(ds); free(p); free(s); free(crow);
  }
}

/* Indexer KL auxiliary loss for a list of query rows (§3 equation; §2 phase
 * table: dense warm-up teacher over every visible entry, sparse mode over the
 * selected set; §9 FP32 loss math).
 *   C_t     = valid entries of idx row (idx != NULL) or every visible entry
 *   pi_h(j) = softmax over j in C_t of scale * q[t,h,:] . K_j
 *   p(j)    = (1/H) sum_h pi_h(j)            (teacher, a_{t,j} = log p(j))
 *   q(j)    = softmax over j in C_t of i_{t,j} (indexer logits)
 *   KL_t    = sum_j p(j) (log p(j) - log q(j))
 * kl[q] = KL_t (0 when C_t is empty), csize[q] = |C_t|.
 * err[q] = 1 when an idx entry lies outside the visible entries (skipped). */
void oracle_indexer_kl(const float* q, const float* kc, const float* qI,
                       const float* w, const float* kI, const int32_t* idx,
                       int k_pad, const int32_t* cu, const int32_t* cu_cmp,
                       int B, int H, int d, int H_I, int dI, int r,
                       double scale, const int64_t* rows, int nq, double* kl,
                       int32_t* csize, int32_t* err) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int qi = 0; qi < nq; ++qi) {
    const int64_t row = rows[qi];
    kl[qi] = 0.0; csize[qi] = 0; err[qi] = 0;
    const int b = owner_sequence(cu, B, row);
    if (b < 0) continue;
    const int64_t t = row - cu[b];
    const int64_t nvis = visible_count(t, r);
    int64_t cap = idx ? k_pad : nvis;
    int64_t* cj = (int64_t*)malloc(sizeof(int64_t) * (cap > 0 ? cap : 1));
    int64_t n = 0;
    if (idx) {
      for (int i = 0; i < k_pad; ++i) {
        const int64_t g = idx[row * (int64_t)k_pad + i];
        if (g < 0) continue;
        if (g < cu_cmp[b] || g >= cu_cmp[b] + nvis) { err[qi] = 1; continue; }
        cj[n++] = g - cu_cmp[b];
      }
    } else {
      for (int64_t j = 0; j < nvis; ++j) cj[n++] = j;
    }
    csize[qi] = (int32_t)n;
    if (n == 0) { free(cj); continue; }
    /* student: indexer logits over C_t */
    double* all_i = (double*)malloc(sizeof(double) * (nvis > 0 ? nvis : 1));
    indexer_logits_one(qI, w, kI, row, cu_cmp[b], nvis, H_I, dI, all_i);
    double* ilog = (double*)malloc(sizeof(double) * n);
    for (int64_t k = 0; k < n; ++k) ilog[k] = all_i[cj[k]];
    double mi = -INFINITY;
    for (int64_t k = 0; k < n; ++k) if (ilog[k] > mi) mi = ilog[k];
    double Zi = 0.0;
    for (int64_t k = 0; k < n; ++k) Zi += exp(ilog[k] - mi);
    const double lse_i = mi + log(Zi);
    /* teacher: per-head softmax over C_t, then the head average */
    double* p = (double*)calloc((size_t)n, sizeof(double));
    double* s = (double*)malloc(sizeof(double) * n);
    for (int h = 0; h < H; ++h) {
      const float* qh = q + (row * H + h) * (int64_t)d;
      for (int64_t k = 0; k < n; ++k) {
        const float* kk = kc + (cu_cmp[b] + cj[k]) * (int64_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += (double)qh[c] * (double)kk[c];
        s[k] = scale * dot;
      }
      double m = -INFINITY;
      for (int64_t k = 0; k < n; ++k) if (s[k] > m) m = s[k];
      double Z = 0.0;
      for (int64_t k = 0; k < n; ++k) Z += exp(s[k] - m);
      for (int64_t k = 0; k < n; ++k) p[k] += exp(s[k] - m) / Z;
    }
    double acc = 0.0;
    for (int64_t k = 0; k < n; ++k) {
      const double pk = p[k] / H;
      if (pk > 0.0) acc += pk * (log(pk) - (ilog[k] - lse_i));
    }
    kl[qi] = acc;
    free(s); free(p); free(ilog); free(all_i); free(cj);
  }
}

/* Backward of the indexer KL loss for a list of query rows (§8.2 "indexer
 * backward": the discrete top-k has no LM-loss gradient, so the indexer is
 * trained only through this auxiliary loss; "teacher operands are detached").
 * With p(j) the teacher and q(j) = softmax over C_t of i_{t,j} as in
 * oracle_indexer_kl, the gradient of KL(p || q) with respect to the indexer
 * logit is g_j = q(j) - p(j) (p sums to 1); times the upstream loss gradient
 * grad_scale, and through i_{t,j} = sum_h w[t,h] ReLU(qI[t,h,:] . kI[j,:]):
 *   dw[t,h]     = sum_j g_j ReLU(a_{h,j}),            a_{h,j} = qI[t,h,:] . kI[j,:]
 *   dqI[t,h,:]  = w[t,h] sum_j g_j [a_{h,j} > 0] kI[j,:]
 *   dkI[j,:]   += sum_h g_j w[t,h] [a_{h,j} > 0] qI[t,h,:]   (accumulated over rows)
 * dqI is [nq, H_I, dI], dw [nq, H_I], dkI [rows of kI, dI] (the caller zeroes
 * it; may be NULL).  Rows with an empty C_t and capacity rows give zeros.
 * err[q] as in oracle_indexer_kl. */
void oracle_indexer_kl_bwd(const float* q, const float* kc, const float* qI,
                           const float* w, const float* kI, const int32_t* idx,
                           int k_pad, const int32_t* cu, const int32_t* cu_cmp,
                           int B, int H, int d, int H_I, int dI, int r,
                           double scale, double grad_scale, const int64_t* rows, int nq,
                           double* dqI, double* dw, double* dkI, int32_t* err) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int qi = 0; qi < nq; ++qi) {
    const int64_t row = rows[qi];
    double* dqq = dqI + (int64_t)qi * H_I * dI;
    double* dwq = dw + (int64_t)qi * H_I;
    for (int64_t e = 0; e < (int64_t)H_I * dI; ++e) dqq[e] = 0.0;
    for (int h = 0; h < H_I; ++h) dwq[h] = 0.0;
    err[qi] = 0;
    const int b = owner_sequence(cu, B, row);
    if (b < 0) continue;
    const int64_t t = row - cu[b];
    const int64_t nvis = visible_count(t, r);
    int64_t cap = idx ? k_pad : nvis;
    int64_t* cj = (int64_t*)malloc(sizeof(int64_t) * (cap > 0 ? cap : 1));
    int64_t n = 0;
    if (idx) {
      for (int i = 0; i < k_pad; ++i) {
        const int64_t g = idx[row * (int64_t)k_pad + i];
        if (g < 0) continue;
        if (g < cu_cmp[b] || g >= cu_cmp[b] + nvis) { err[qi] = 1; continue; }
        cj[n++] = g - cu_cmp[b];
      }
    } else {
      for (int64_t j = 0; j < nvis; ++j) cj[n++] = j;
    }
    if (n == 0) { free(cj); continue; }
    /* student distribution over C_t */
    double* all_i = (double*)malloc(sizeof(double) * (nvis > 0 ? nvis : 1));
    indexer_logits_one(qI, w, kI, row, cu_cmp[b], nvis, H_I, dI, all_i);
    double mi = -INFINITY;
    for (int64_t k = 0; k < n; ++k) if (all_i[cj[k]] > mi) mi = all_i[cj[k]];
    double Zi = 0.0;
    for (int64_t k = 0; k < n; ++k) Zi += exp(all_i[cj[k]] - mi);
    /* teacher: head average of per-head softmaxes over C_t */
    double* p = (double*)calloc((size_t)n, sizeof(double));
    double* s = (double*)malloc(sizeof(double) * n);
    for (int h = 0; h < H; ++h) {
      const float* qh = q + (row * H + h) * (int64_t)d;
      for (int64_t k = 0; k < n; ++k) {
        const float* kk = kc + (cu_cmp[b] + cj[k]) * (int64_t)d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += (double)qh[c] * (double)kk[c];
        s[k] = scale * dot;
      }
      double m = -INFINITY;
      for (int64_t k = 0; k < n; ++k) if (s[k] > m) m = s[k];
      double Z = 0.0;
      for (int64_t k = 0; k < n; ++k) Z += exp(s[k] - m);
      for (int64_t k = 0; k < n; ++k) p[k] += exp(s[k] - m) / Z;
    }
    /* g_j and the chain rule through the indexer logit */
    double* gk = dkI ? (double*)calloc((size_t)n * dI, sizeof(double)) : NULL;
    for (int64_t k = 0; k < n; ++k) {
      const double g = grad_scale * (exp(all_i[cj[k]] - mi) / Zi - p[k] / H);
      const float* kr = kI + (cu_cmp[b] + cj[k]) * (int64_t)dI;
      for (int h = 0; h < H_I; ++h) {
        const float* qh = qI + (row * H_I + h) * (int64_t)dI;
        double a = 0.0;
        for (int c = 0; c < dI; ++c) a += (double)qh[c] * (double)kr[c];
        if (a <= 0.0) continue;
        const double wh = (double)w[row * H_I + h];
        dwq[h] += g * a;
        for (int c = 0; c < dI; ++c) {
          dqq[(int64_t)h * dI + c] += g * wh * (double)kr[c];
          if (gk) gk[k * dI + c] += g * wh * (double)qh[c];
        }
      }
    }
    if (gk) {
#pragma omp critical(oracle_indexer_kl_bwd_merge)
      for (int64_t k = 0; k < n; ++k)
        for (int c = 0; c < dI; ++c) dkI[(cu_cmp[b] + cj[k]) * (int64_t)dI + c] += gk[k * dI + c];
      free(gk);
    }
    free(s); free(p); free(all_i); free(cj);
  }
}

/* FP8 (E4M3) quantisation of the indexer operands (§1 and §9: the FP8 indexer
 * for the index-search term).  The E4M3 format of the OCP 8-bit floating
 * point specification: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormals below 2^-6 in steps of 2^-9, largest finite value 448.
 * Each row of x gets a power-of-two scale s = 2^e, the smallest with
 * max|x| / s <= 448 (s = 1 for an all-zero row), and the code of x / s
 * rounded to the nearest representable value, ties to even.  The scale
 * decision takes max|x| / 448 in float32.  codes [rows, cols], scales [rows]. */
static uint8_t e4m3_encode(double v) {
  uint8_t sign = 0;
  if (signbit(v)) { sign = 0x80; v = -v; }   /* E4M3 has signed zeros: -0 -> 0x80 */
  if (v == 0.0) return sign;
  if (v < 0.015625) {                       /* below 2^-6: subnormal steps of 2^-9 */
    const double m = nearbyint(v * 512.0);  /* m == 8 is the smallest normal, code 0x08 */
    return (uint8_t)(sign | (uint8_t)m);
  }
  int e;
  const double f = frexp(v, &e);            /* v = f 2^e, f in [0.5, 1) */
  int E = e - 1;                            /* v = (1 + mant) 2^E */
  double m = nearbyint((2.0 * f - 1.0) * 8.0);
  if (m == 8.0) { m = 0.0; E += 1; }
  return (uint8_t)(sign | (uint8_t)((E + 7) << 3) | (uint8_t)m);
}

double oracle_e4m3_value(uint8_t code) {
  const double s = (code & 0x80) ? -1.0 : 1.0;
  const int ef = (code >> 3) & 15, m = code & 7;
  if (ef == 15 && m == 7) return NAN;
  if (ef == 0) return s * m * (1.0 / 512.0);
  return s * ldexp(1.0 + m / 8.0, ef - 7);
}

void oracle_quantize_fp8(const float* x, int64_t rows, int cols, uint8_t* codes, float* scales) {
  for (int64_t i = 0; i < rows; ++i) {
    float amax = 0.f;
    for (int c = 0; c < cols; ++c) {
      const float a = fabsf(x[i * cols + c]);
      if (a > amax) amax = a;
    }
    int e = 0;
    if (amax > 0.f) {
      const float ratio = amax / 448.0f;    /* float32, as the decision is specified */
      int fe;
      const float fm = frexpf(ratio, &fe);  /* ratio = fm 2^fe, fm in [0.5, 1) */
      e = (fm == 0.5f) ? fe - 1 : fe;       /* smallest e with ratio <= 2^e */
    }
    scales[i] = ldexpf(1.0f, e);
    const double inv = ldexp(1.0, -e);
    for (int c = 0; c < cols; ++c) codes[i * cols + c] = e4m3_encode((double)x[i * cols + c] * inv);
  }
}
