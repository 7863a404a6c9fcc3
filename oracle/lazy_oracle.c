/*
 * lazy_oracle.c -- plain, slow, fp64 CPU reference for LazyAttention over a
 * paged, position-agnostic KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path (the CUDA
 * library) shares no code, header, table or helper with it.
 *
 * What it computes, and where the definition comes from:
 *
 *  - Rotary position embedding R_n, rotate-half pairing (i, i+d/2) with
 *    omega_i = theta^(-2i/d) (lo_rope_rotate_ex / lo_attention_ex also take an
 *    explicit frequency vector, e.g. lo_llama3_freqs, and the interleaved pairing
 *    (2i, 2i+1); lo_rope_rotate_partial / lo_attention_partial rotate only the
 *    first r dims, as partial-rotary models do, and lo_attention_partial adds an
 *    optional ALiBi bias):
 *        y_i     = x_i cos(n w_i) - x_{i+h} sin(n w_i)
 *        y_{i+h} = x_{i+h} cos(n w_i) + x_i sin(n w_i)
 *    The LazyAttention technical summary ("Mathematical Equivalence") relies on
 *    RoPE scores depending only on the relative offset; the pages do not print
 *    the pairing or frequencies, so this is the Llama/vLLM "neox" form.
 *
 *  - Stored K: each cached document's key rows are stored rotated at their
 *    document-local positions 0..len-1; V is stored unrotated; a document used
 *    at global offset p contributes keys at absolute positions p+j
 *    (summary, "Methodology: Deferred Positional Encoding").
 *
 *  - Attention (lo_attention): for every sequence the oracle MATERIALISES the
 *    position-adjusted copy K_adj[j] = R_p K_stored[j] -- the eager baseline the
 *    summary's "Problem Statement" describes -- then, for each query row at
 *    absolute position m, rotates q' = R_m q and evaluates the textbook
 *    softmax(q' K_adj^T / sqrt(d)) V over the keys whose absolute position is
 *    <= m (causal attention in absolute positions; "Por qué existe un KV Cache",
 *    "Lo que hace el decoding autorregresivo", step 2). Softmax is one-shot
 *    (max-subtracted) in fp64.
 *
 *  - lo_tiled_softmax_dot: the running (max, sum) softmax over key tiles from
 *    "KV Cache, Flash Attention & Otimização de Inferência", section
 *    "Flash Attention -- tiling" and "Passo 2: tiled softmax", written from its
 *    description; lo_softmax_dot is the one-shot form it must equal.
 *
 *  - lo_kv_cache_bytes: the cache size formula 2*L*H*d_h*S*B*s from
 *    "Por qué existe un KV Cache", section "El precio".
 *
 * Inputs are the stored bits (fp32 or bf16) and are upcast exactly to fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { LO_F32 = 0, LO_BF16 = 1 };

static double lo_load(const void *base, int dtype, int64_t idx) {
  if (dtype == LO_F32) return (double)((const float *)base)[idx];
  uint32_t u = (uint32_t)((const uint16_t *)base)[idx] << 16; /* bf16 -> fp32 is exact */
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

int lo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void lo_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Partial rotary (GPT-NeoX / GPT-J rotary_dim): y = R_n x on the first r dims only,
 * pairs (i, i + r/2) (rotate-half) or (2i, 2i+1) (`interleaved`), i < r/2, with
 * frequencies w[i] (NULL: theta^(-2i/r), the exponent taken over the rotated dims);
 * dims r .. d-1 are copied. r = d is the full rotation. x and y may alias. */
void lo_rope_rotate_partial(int d, int r, double theta, const double *w, int interleaved, double n,
                            const double *x, double *y) {
  int h = r / 2;
  for (int c = r; c < d; c++) y[c] = x[c];
  for (int i = 0; i < h; i++) {
    double wi = w ? w[i] : pow(theta, -2.0 * (double)i / (double)r);
    double c = cos(n * wi), s = sin(n * wi);
    int ia = interleaved ? 2 * i : i, ib = interleaved ? 2 * i + 1 : i + h;
    double a = x[ia], b = x[ib];
    y[ia] = a * c - b * s;
    y[ib] = b * c + a * s;
  }
}

/* y = R_n x with frequencies w[i] (NULL: theta^(-2i/d)) and pairing (i, i+d/2), or
 * (2i, 2i+1) when `interleaved` (GPT-J style). x and y may alias. */
void lo_rope_rotate_ex(int d, double theta, const double *w, int interleaved, double n, const double *x,
                       double *y) {
  lo_rope_rotate_partial(d, d, theta, w, interleaved, n, x, y);
}

/* y = R_n x, rotate-half pairing, omega_i = theta^(-2i/d). x and y may alias. */
void lo_rope_rotate(int d, double theta, double n, const double *x, double *y) {
  lo_rope_rotate_ex(d, theta, NULL, 0, n, x, y);
}

/* Llama-3.1 frequency scaling of omega_i = theta^(-2i/d), i < d/2 (the rule published
 * with Llama 3.1): with wavelength lambda = 2 pi / omega, lambda_hi = L / high_ff and
 * lambda_lo = L / low_ff (L the original context length), a frequency is kept when
 * lambda < lambda_hi, divided by `factor` when lambda > lambda_lo, and otherwise
 * interpolated: s = (L / lambda - low_ff) / (high_ff - low_ff),
 * omega' = (1 - s) omega / factor + s omega. */
void lo_llama3_freqs(int d, double theta, double factor, double low_ff, double high_ff, double orig_max,
                     double *out) {
  const double two_pi = 6.283185307179586476925286766559;
  const double lam_hi = orig_max / high_ff, lam_lo = orig_max / low_ff;
  for (int i = 0; i < d / 2; i++) {
    const double w = pow(theta, -2.0 * (double)i / (double)d);
    const double lam = two_pi / w;
    if (lam < lam_hi) {
      out[i] = w;
    } else if (lam > lam_lo) {
      out[i] = w / factor;
    } else {
      const double s = (orig_max / lam - low_ff) / (high_ff - low_ff);
      out[i] = (1.0 - s) * w / factor + s * w;
    }
  }
}

/* out = softmax(K q) V computed in one shot; K, V are [n][d]. */
void lo_softmax_dot(int n, int d, const double *q, const double *K, const double *V, double *out) {
  double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double mx = -INFINITY, den = 0.0;
  for (int j = 0; j < n; j++) {
    double acc = 0.0;
    for (int c = 0; c < d; c++) acc += q[c] * K[(size_t)j * d + c];
    s[j] = acc;
    if (acc > mx) mx = acc;
  }
  for (int c = 0; c < d; c++) out[c] = 0.0;
  for (int j = 0; j < n; j++) {
    double e = exp(s[j] - mx);
    den += e;
    for (int c = 0; c < d; c++) out[c] += e * V[(size_t)j * d + c];
  }
  if (den > 0.0)
    for (int c = 0; c < d; c++) out[c] /= den;
  free(s);
}

/* Running-softmax form: keys are visited in tiles of `tile`; a running maximum
 * m and running denominator l are kept, and the accumulated numerator is
 * rescaled by exp(m_old - m_new) whenever a tile raises the maximum. */
void lo_tiled_softmax_dot(int n, int d, const double *q, const double *K, const double *V, int tile,
                          double *out) {
  double m = -INFINITY, l = 0.0;
  double *sc = (double *)malloc(sizeof(double) * (size_t)(tile > 0 ? tile : 1));
  for (int c = 0; c < d; c++) out[c] = 0.0;
  for (int t0 = 0; t0 < n; t0 += tile) {
    int t1 = t0 + tile < n ? t0 + tile : n;
    double m_new = m;
    for (int j = t0; j < t1; j++) {
      double acc = 0.0;
      for (int c = 0; c < d; c++) acc += q[c] * K[(size_t)j * d + c];
      sc[j - t0] = acc;
      if (acc > m_new) m_new = acc;
    }
    double scale_old = (m == -INFINITY) ? 0.0 : exp(m - m_new);
    l *= scale_old;
    for (int c = 0; c < d; c++) out[c] *= scale_old;
    for (int j = t0; j < t1; j++) {
      double e = exp(sc[j - t0] - m_new);
      l += e;
      for (int c = 0; c < d; c++) out[c] += e * V[(size_t)j * d + c];
    }
    m = m_new;
  }
  if (l > 0.0)
    for (int c = 0; c < d; c++) out[c] /= l;
  free(sc);
}

double lo_kv_cache_bytes(double layers, double heads, double head_dim, double seq, double batch,
                         double elt_bytes) {
  return 2.0 * layers * heads * head_dim * seq * batch * elt_bytes;
}

/*
 * Attention for `nq` query rows.
 *   q        [nq][hq][d]   stored bits, unrotated
 *   q_seq    [nq]          sequence of each row
 *   q_m      [nq]          absolute position of each row
 *   k_pool, v_pool [num_pool_blocks][hkv][16][d] stored bits
 *   seg_indptr [num_seqs+1], seg_doc, seg_len: the documents of each sequence in
 *            order; a segment uses the first seg_len tokens of its document
 *   seq_pos0 [num_seqs]    absolute position of each sequence's first key
 *   doc_block_indptr, doc_blocks: physical block ids of each document, in order
 *   out      [nq][hq][d]   fp64
 * Returns 0, or -1 on a malformed layout.
 */
/* ALiBi: with alibi[hq] given, every score of q-head h also gets the linear bias
 * -alibi[h] * (m - n) for a key at absolute position n and a query at m (the bias is
 * added to the scaled score, before the softmax). NULL: no bias. */
int lo_attention_partial(int num_seqs, int hq, int hkv, int d, int rot_dims, double theta, const double *freqs,
                         int interleaved, double sm_scale, int dtype, int nq, const void *q, const int32_t *q_seq,
                         const int32_t *q_m, const void *k_pool, const void *v_pool, int64_t num_pool_blocks,
                         const int32_t *seg_indptr, const int32_t *seg_doc, const int32_t *seg_len,
                         const int32_t *seq_pos0, const int32_t *doc_block_indptr, const int32_t *doc_blocks,
                         const double *alibi, double *out) {
  if (hkv <= 0 || hq % hkv != 0 || d <= 0 || d % 2 != 0) return -1;
  if (rot_dims <= 0) rot_dims = d;
  if (rot_dims > d || rot_dims % 2 != 0) return -1;
  const int g = hq / hkv;
  if (sm_scale <= 0.0) sm_scale = 1.0 / sqrt((double)d);
  int bad = 0;

  /* Validate every segment's blocks before touching the pool. */
  for (int s = 0; s < num_seqs; s++)
    for (int k = seg_indptr[s]; k < seg_indptr[s + 1]; k++) {
      int doc = seg_doc[k], len = seg_len[k];
      int nb = doc_block_indptr[doc + 1] - doc_block_indptr[doc];
      if (len < 0 || len > nb * 16) return -1;
      for (int b = 0; b < (len + 15) / 16; b++) {
        int32_t phys = doc_blocks[doc_block_indptr[doc] + b];
        if (phys < 0 || phys >= num_pool_blocks) return -1;
      }
    }
  for (int r = 0; r < nq; r++)
    if (q_seq[r] < 0 || q_seq[r] >= num_seqs) return -1;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t task = 0; task < (int64_t)num_seqs * hkv; task++) {
    const int s = (int)(task / hkv), kvh = (int)(task % hkv);
    int has_query = 0;
    for (int r = 0; r < nq && !has_query; r++) has_query = (q_seq[r] == s);
    if (!has_query) continue;

    /* 1-2: upcast the stored rows and materialise K_adj = R_p K_stored. */
    int64_t n = 0;
    for (int k = seg_indptr[s]; k < seg_indptr[s + 1]; k++) n += seg_len[k];
    double *Kadj = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * d);
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    double *row = (double *)malloc(sizeof(double) * d);
    double *qr = (double *)malloc(sizeof(double) * d);
    double *sc = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!Kadj || !V || !pos || !row || !qr || !sc) {
#pragma omp atomic write
      bad = 1;
      free(Kadj), free(V), free(pos), free(row), free(qr), free(sc);
      continue;
    }
    int64_t t = 0, p = seq_pos0 ? seq_pos0[s] : 0;
    for (int k = seg_indptr[s]; k < seg_indptr[s + 1]; k++) {
      const int doc = seg_doc[k];
      for (int j = 0; j < seg_len[k]; j++, t++) {
        const int64_t phys = doc_blocks[doc_block_indptr[doc] + j / 16];
        const int64_t base = ((phys * hkv + kvh) * 16 + (j % 16)) * (int64_t)d;
        for (int c = 0; c < d; c++) row[c] = lo_load(k_pool, dtype, base + c);
        lo_rope_rotate_partial(d, rot_dims, theta, freqs, interleaved, (double)p, row, &Kadj[t * d]);
        for (int c = 0; c < d; c++) V[t * d + c] = lo_load(v_pool, dtype, base + c);
        pos[t] = p + j;
      }
      p += seg_len[k];
    }

    /* 3-4: per query row and q-head of this KV head, rotate q and attend. */
    for (int r = 0; r < nq; r++) {
      if (q_seq[r] != s) continue;
      const int64_t m = q_m[r];
      for (int h = kvh * g; h < (kvh + 1) * g; h++) {
        for (int c = 0; c < d; c++) row[c] = lo_load(q, dtype, ((int64_t)r * hq + h) * d + c);
        lo_rope_rotate_partial(d, rot_dims, theta, freqs, interleaved, (double)m, row, qr);
        double mx = -INFINITY;
        for (int64_t j = 0; j < n; j++) {
          if (pos[j] > m) { sc[j] = -INFINITY; continue; }
          double acc = 0.0;
          for (int c = 0; c < d; c++) acc += qr[c] * Kadj[j * d + c];
          sc[j] = acc * sm_scale;
          if (alibi) sc[j] -= alibi[h] * (double)(m - pos[j]);
          if (sc[j] > mx) mx = sc[j];
        }
        double *o = &out[((int64_t)r * hq + h) * d];
        for (int c = 0; c < d; c++) o[c] = 0.0;
        if (mx == -INFINITY) continue; /* no visible key: output 0 */
        double den = 0.0;
        for (int64_t j = 0; j < n; j++) {
          if (sc[j] == -INFINITY) continue;
          double e = exp(sc[j] - mx);
          den += e;
          for (int c = 0; c < d; c++) o[c] += e * V[j * d + c];
        }
        for (int c = 0; c < d; c++) o[c] /= den;
      }
    }
    free(Kadj), free(V), free(pos), free(row), free(qr), free(sc);
  }
  return bad ? -1 : 0;
}

/* lo_attention_ex with theta^(-2i/d) frequencies and rotate-half pairing. */
int lo_attention_ex(int num_seqs, int hq, int hkv, int d, double theta, const double *freqs, int interleaved,
                    double sm_scale, int dtype, int nq, const void *q, const int32_t *q_seq, const int32_t *q_m,
                    const void *k_pool, const void *v_pool, int64_t num_pool_blocks, const int32_t *seg_indptr,
                    const int32_t *seg_doc, const int32_t *seg_len, const int32_t *seq_pos0,
                    const int32_t *doc_block_indptr, const int32_t *doc_blocks, double *out) {
  return lo_attention_partial(num_seqs, hq, hkv, d, d, theta, freqs, interleaved, sm_scale, dtype, nq, q, q_seq, q_m,
                              k_pool, v_pool, num_pool_blocks, seg_indptr, seg_doc, seg_len, seq_pos0,
                              doc_block_indptr, doc_blocks, NULL, out);
}

int lo_attention(int num_seqs, int hq, int hkv, int d, double theta, double sm_scale, int dtype, int nq,
                 const void *q, const int32_t *q_seq, const int32_t *q_m, const void *k_pool,
                 const void *v_pool, int64_t num_pool_blocks, const int32_t *seg_indptr,
                 const int32_t *seg_doc, const int32_t *seg_len, const int32_t *seq_pos0,
                 const int32_t *doc_block_indptr, const int32_t *doc_blocks, double *out) {
  return lo_attention_ex(num_seqs, hq, hkv, d, theta, NULL, 0, sm_scale, dtype, nq, q, q_seq, q_m, k_pool, v_pool,
                         num_pool_blocks, seg_indptr, seg_doc, seg_len, seq_pos0, doc_block_indptr, doc_blocks,
                         out);
}
