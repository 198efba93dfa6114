/*
 * Oracle for the FLUX.2 joint RoPE attention: plain, slow, fp64, CPU only.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the timed
 * CPU baseline of the bench load this file's library. The product path (the
 * CUDA library under diffusion_transformer_joint_gb300/csrc) shares no code,
 * header, table or constant with it.
 *
 * What it computes, written out from the definitions on the pages:
 *
 *   1. Position ids. Every token carries one id per RoPE axis; FLUX.2 uses
 *      four axes (T, H, W, L), and the id tensor's last dimension must equal
 *      the number of axes. Text ids come first, then image (and reference)
 *      ids: the joint sequence is [txt ; img].
 *      ("Diffusers 中 Flux2Transformer2DModel 全面解析", section
 *      "前向传播输入输出约定": 4-d (T,H,W,L) ids, last dim = len(axes_dims_rope).)
 *
 *   2. N-D RoPE (EmbedND / Flux2PosEmbed): a 1-D RoPE is built per axis and
 *      the axes are concatenated; axes_dims = (32,32,32,32), theta = 2000.
 *      (Same page, sections "前向传播输入输出约定" and "模型配置参数全解";
 *      "FLUX.2 [klein]" survey page, section "模型架构".)
 *      Per axis a with width d_a and pair j < d_a/2 the frequency is
 *      omega_j = theta^(-2j/d_a) and the angle is id[a] * omega_j; pair j of
 *      axis a is the channel pair (2p, 2p+1) with p = (sum_{a'<a} d_a'/2) + j.
 *      The pair (x_2p, x_2p+1) is multiplied, as a complex number
 *      x_2p + i x_2p+1, by exp(i * angle).
 *
 *   3. Attention ("Transformer架构解析FLUX.2-klein-base-9b-nvfp4", section 2
 *      "核心引擎自注意力机制如何工作": scaled dot-product attention):
 *      out_i = sum_j softmax_j(q^_i . k^_j / sqrt(d)) v_j over all S tokens,
 *      non-causal, per batch element and head, d = head_dim = 128, with q^ and
 *      k^ the RoPE-rotated queries and keys; V is not rotated.
 *
 *   4. Optional QK RMS normalisation before the rotation ("Diffusers 中
 *      Flux2Transformer2DModel 全面解析", section "内部架构双流块与单流块": in
 *      the joint attention Q and K are RMS-normalised right after their
 *      projections, with separate norms for the text and the image stream;
 *      section "并行化支持": the norm acts on the whole head_dim of a head;
 *      section "模型配置参数全解": eps = 1e-6). For one head vector x[D] with
 *      a learned per-channel weight w[D]:
 *        y_c = x_c / sqrt(mean over c' of x_c'^2 + eps) * w_c,
 *      text tokens (the first S_txt) with the text weights, the others with
 *      the image weights; V is not normalised.
 *
 *   5. Reference-image KV modes ("Diffusers 中 Flux2Transformer2DModel 全面解析",
 *      section "参考图 KV 缓存机制": the cache holds the reference tokens' K
 *      after RoPE and their V, [B, n_ref, H, D]; in "extract" mode the
 *      sequence is [txt, ref, img], reference queries attend to reference
 *      keys only while text and image queries attend to every token, and the
 *      reference K / V are stored to the cache; in "cached" mode the sequence
 *      is [txt, img] and the cached reference K / V are inserted between the
 *      text and the image keys and values). With the QK normalisation of
 *      step 4 the modes see q and k normalised first (reference tokens take
 *      the image stream's weights), so the cache holds normalised, rotated K.
 *
 *   6. The single-stream block's fused input projection ("Diffusers 中
 *      Flux2Transformer2DModel 全面解析", section "内部架构双流块与单流块": one
 *      linear layer, to_qkv_mlp_proj, produces 3 * inner_dim + mlp_hidden_dim *
 *      mlp_mult_factor features: the Q, K and V projections and the MLP's input
 *      projection in one; section "激活函数与 FFN": the SwiGLU gate projection
 *      is fused into the preceding linear layer and the activation halves the
 *      width; section "并行化支持": that packed projection splits into two equal
 *      halves, gate and linear). For a token row x[dim] and the weight
 *      W[n_out, dim] (rows are output features):
 *        y_n = sum_c W[n, c] x[c],  n < n_out = 3 * inner + 2 * mlp,
 *        q = y[0, inner), k = y[inner, 2 inner), v = y[2 inner, 3 inner), each
 *        read as [H, D] (inner = H * D, channel h * D + d is head h, dim d),
 *        a_j = silu(y[3 inner + j]) * y[3 inner + mlp + j],  j < mlp,
 *        silu(g) = g / (1 + exp(-g)).
 *      No bias (the pages name none).
 *
 * Layout: q, k, v, out are [B, S, H, D] row-major (D fastest), in double.
 * ids are [S, n_axes] int32 and are shared by every batch element.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Frequencies and per-token angles, step 2 above. cos_out/sin_out are
 * [S, P] with P = sum(axes_dims)/2. Returns 0, or -1 on a bad axis width. */
int oracle_rope_tables(const int32_t *ids, int64_t S, const int32_t *axes_dims,
                       int n_axes, double theta, double *cos_out,
                       double *sin_out) {
  int P = 0;
  for (int a = 0; a < n_axes; ++a) {
    if (axes_dims[a] <= 0 || axes_dims[a] % 2 != 0) return -1;
    P += axes_dims[a] / 2;
  }
  for (int64_t s = 0; s < S; ++s) {
    int p = 0;
    for (int a = 0; a < n_axes; ++a) {
      int d_a = axes_dims[a];
      for (int j = 0; j < d_a / 2; ++j, ++p) {
        double omega = pow(theta, -2.0 * (double)j / (double)d_a);
        double angle = (double)ids[s * n_axes + a] * omega;
        cos_out[s * P + p] = cos(angle);
        sin_out[s * P + p] = sin(angle);
      }
    }
  }
  return 0;
}

/* Rotation of one head vector x[D] by the token's table row, step 2 above:
 * (x_2p + i x_2p+1) * (c_p + i s_p). */
void oracle_rope_apply_vec(const double *x, const double *c, const double *sn,
                           int D, double *y) {
  for (int p = 0; p < D / 2; ++p) {
    double re = x[2 * p], im = x[2 * p + 1];
    y[2 * p] = re * c[p] - im * sn[p];
    y[2 * p + 1] = re * sn[p] + im * c[p];
  }
}

/* RMS normalisation of one head vector, step 4 above. */
void oracle_rms_norm_vec(const double *x, const double *w, int D, double eps,
                         double *y) {
  double ss = 0.0;
  for (int c = 0; c < D; ++c) ss += x[c] * x[c];
  const double r = 1.0 / sqrt(ss / (double)D + eps);
  for (int c = 0; c < D; ++c) y[c] = x[c] * r * w[c];
}

/* RMS normalisation of every head vector of a [B, S, H, D] tensor with one
 * weight vector w[D]. */
void oracle_rms_norm(const double *x, int B, int64_t S, int H, int D,
                     const double *w, double eps, double *y) {
  for (int64_t n = 0; n < (int64_t)B * S * H; ++n)
    oracle_rms_norm_vec(x + n * D, w, D, eps, y + n * D);
}

/* Rotation of a whole [B, S, H, D] tensor with tables [S, D/2]. */
void oracle_rope_apply(const double *x, int B, int64_t S, int H, int D,
                       const double *cos_t, const double *sin_t, double *y) {
  for (int b = 0; b < B; ++b)
    for (int64_t s = 0; s < S; ++s)
      for (int h = 0; h < H; ++h) {
        int64_t off = (((int64_t)b * S + s) * H + h) * D;
        oracle_rope_apply_vec(x + off, cos_t + s * (D / 2), sin_t + s * (D / 2),
                              D, y + off);
      }
}

/* ---- attention, step 3 ------------------------------------------------- */

typedef struct {
  const double *q, *k, *v, *cos_t, *sin_t;
  /* optional RMS-norm weights [D] (all NULL: no normalisation) */
  const double *qw_txt, *kw_txt, *qw_img, *kw_img;
  int64_t S_txt;
  double eps;
  int B, H, D;
  int64_t S;
  const int64_t *rows; /* query token indices to evaluate */
  int64_t n_rows;
  double *out; /* [B, n_rows, H, D] */
  int64_t next_unit; /* shared work counter over (b, h) */
  pthread_mutex_t lock;
} attn_job;

/* One (batch, head) pair: rotate every key of that head, then evaluate each
 * requested query row straight from the definition. */
static void attn_unit(attn_job *J, int b, int h) {
  const int D = J->D, H = J->H;
  const int64_t S = J->S;
  const double scale = 1.0 / sqrt((double)D);
  double *khat = (double *)malloc(sizeof(double) * (size_t)S * D);
  double *z = (double *)malloc(sizeof(double) * (size_t)S);
  double *qhat = (double *)malloc(sizeof(double) * (size_t)D);
  double *xn = (double *)malloc(sizeof(double) * (size_t)D);
  const int norm = J->qw_txt != NULL;
  for (int64_t j = 0; j < S; ++j) {
    int64_t off = (((int64_t)b * S + j) * H + h) * D;
    const double *kj = J->k + off;
    if (norm) {
      oracle_rms_norm_vec(kj, j < J->S_txt ? J->kw_txt : J->kw_img, D, J->eps, xn);
      kj = xn;
    }
    oracle_rope_apply_vec(kj, J->cos_t + j * (D / 2),
                          J->sin_t + j * (D / 2), D, khat + j * D);
  }
  for (int64_t r = 0; r < J->n_rows; ++r) {
    int64_t i = J->rows[r];
    int64_t qoff = (((int64_t)b * S + i) * H + h) * D;
    const double *qi = J->q + qoff;
    if (norm) {
      oracle_rms_norm_vec(qi, i < J->S_txt ? J->qw_txt : J->qw_img, D, J->eps, xn);
      qi = xn;
    }
    oracle_rope_apply_vec(qi, J->cos_t + i * (D / 2),
                          J->sin_t + i * (D / 2), D, qhat);
    /* logits z_j = q^_i . k^_j / sqrt(D) */
    double zmax = -INFINITY;
    for (int64_t j = 0; j < S; ++j) {
      double acc = 0.0;
      for (int c = 0; c < D; ++c) acc += qhat[c] * khat[j * D + c];
      z[j] = acc * scale;
      if (z[j] > zmax) zmax = z[j];
    }
    /* softmax over all keys (the max is subtracted only to keep exp finite;
     * it cancels in the ratio), then the weighted sum of V */
    double denom = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      z[j] = exp(z[j] - zmax);
      denom += z[j];
    }
    double *o = J->out + (((int64_t)b * J->n_rows + r) * H + h) * D;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < S; ++j) {
      const double *vj = J->v + (((int64_t)b * S + j) * H + h) * D;
      double w = z[j] / denom;
      for (int c = 0; c < D; ++c) o[c] += w * vj[c];
    }
  }
  free(khat);
  free(z);
  free(qhat);
  free(xn);
}

static void *attn_worker(void *arg) {
  attn_job *J = (attn_job *)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int64_t u = J->next_unit++;
    pthread_mutex_unlock(&J->lock);
    if (u >= (int64_t)J->B * J->H) break;
    attn_unit(J, (int)(u / J->H), (int)(u % J->H));
  }
  return NULL;
}

/* Joint RoPE attention for the query tokens listed in rows[0..n_rows) (every
 * token when rows is NULL), all batch elements and heads. ids = [txt ; img]
 * already concatenated, [S, n_axes]. out is [B, n_rows, H, D]. Work over
 * (b, h) is spread on n_threads POSIX threads; the arithmetic of each output
 * does not depend on the thread count. Returns 0, or -1 on bad arguments. */
static int joint_attention(const double *q, const double *k, const double *v,
                           int B, int64_t S, int H, int D, const int32_t *ids,
                           const int32_t *axes_dims, int n_axes, double theta,
                           const double *qw_txt, const double *kw_txt,
                           const double *qw_img, const double *kw_img,
                           int64_t S_txt, double eps, const int64_t *rows,
                           int64_t n_rows, int n_threads, double *out) {
  int sum = 0;
  for (int a = 0; a < n_axes; ++a) sum += axes_dims[a];
  if (sum != D || D % 2 != 0 || S <= 0 || B <= 0 || H <= 0) return -1;
  double *cos_t = (double *)malloc(sizeof(double) * (size_t)S * (D / 2));
  double *sin_t = (double *)malloc(sizeof(double) * (size_t)S * (D / 2));
  int64_t *all_rows = NULL;
  if (oracle_rope_tables(ids, S, axes_dims, n_axes, theta, cos_t, sin_t) != 0) {
    free(cos_t);
    free(sin_t);
    return -1;
  }
  if (rows == NULL) {
    all_rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)S);
    for (int64_t i = 0; i < S; ++i) all_rows[i] = i;
    rows = all_rows;
    n_rows = S;
  }
  attn_job J;
  J.q = q; J.k = k; J.v = v; J.cos_t = cos_t; J.sin_t = sin_t;
  J.qw_txt = qw_txt; J.kw_txt = kw_txt; J.qw_img = qw_img; J.kw_img = kw_img;
  J.S_txt = S_txt; J.eps = eps;
  J.B = B; J.H = H; J.D = D; J.S = S;
  J.rows = rows; J.n_rows = n_rows; J.out = out; J.next_unit = 0;
  pthread_mutex_init(&J.lock, NULL);
  if (n_threads < 1) n_threads = 1;
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, attn_worker, &J);
  for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.lock);
  free(th);
  free(all_rows);
  free(cos_t);
  free(sin_t);
  return 0;
}

int oracle_joint_rope_attention(const double *q, const double *k,
                                const double *v, int B, int64_t S, int H, int D,
                                const int32_t *ids, const int32_t *axes_dims,
                                int n_axes, double theta, const int64_t *rows,
                                int64_t n_rows, int n_threads, double *out) {
  return joint_attention(q, k, v, B, S, H, D, ids, axes_dims, n_axes, theta, NULL,
                         NULL, NULL, NULL, 0, 0.0, rows, n_rows, n_threads, out);
}

/* The same with the QK RMS normalisation of step 4 before the rotation:
 * weights [D] for the text tokens (the first S_txt) and for the others. */
int oracle_joint_qknorm_rope_attention(
    const double *q, const double *k, const double *v, int B, int64_t S, int H,
    int D, const int32_t *ids, const int32_t *axes_dims, int n_axes, double theta,
    const double *qw_txt, const double *kw_txt, const double *qw_img,
    const double *kw_img, int64_t S_txt, double eps, const int64_t *rows,
    int64_t n_rows, int n_threads, double *out) {
  if (qw_txt == NULL || kw_txt == NULL || qw_img == NULL || kw_img == NULL ||
      S_txt < 0 || S_txt > S || !(eps >= 0.0))
    return -1;
  return joint_attention(q, k, v, B, S, H, D, ids, axes_dims, n_axes, theta, qw_txt,
                         kw_txt, qw_img, kw_img, S_txt, eps, rows, n_rows, n_threads,
                         out);
}

/* ---- reference KV modes, step 5 --------------------------------------- */

/* Softmax-weighted sum over keys [k_lo, k_hi) of rotated keys khat (rows of
 * D) and values vrow(j) for one rotated query qhat. */
static void attend_range(const double *qhat, const double *khat, const double *const *vrows,
                         int64_t k_lo, int64_t k_hi, int D, double *z, double *o) {
  const double scale = 1.0 / sqrt((double)D);
  double zmax = -INFINITY;
  for (int64_t j = k_lo; j < k_hi; ++j) {
    double acc = 0.0;
    for (int c = 0; c < D; ++c) acc += qhat[c] * khat[j * D + c];
    z[j] = scale * acc;
    if (z[j] > zmax) zmax = z[j];
  }
  double denom = 0.0;
  for (int64_t j = k_lo; j < k_hi; ++j) {
    z[j] = exp(z[j] - zmax);
    denom += z[j];
  }
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  for (int64_t j = k_lo; j < k_hi; ++j) {
    const double wj = z[j] / denom;
    for (int c = 0; c < D; ++c) o[c] += wj * vrows[j][c];
  }
}

/* Extract mode. Tokens [txt ; ref ; img] (S_txt, S_ref, then the rest), ids
 * [S, n_axes] in the same order. Reference queries attend to the reference
 * keys, every other query to all S keys; out [B, n_rows, H, D] for the query
 * tokens rows[0 .. n_rows) (every token when rows is NULL). cache_k /
 * cache_v [B, S_ref, H, D]: the reference tokens' rotated K and their V.
 * Single threaded. Returns 0, or -1 on bad arguments. */
int oracle_attention_extract(const double *q, const double *k, const double *v, int B,
                             int64_t S, int H, int D, const int32_t *ids,
                             const int32_t *axes_dims, int n_axes, double theta,
                             int64_t S_txt, int64_t S_ref, const int64_t *rows, int64_t n_rows,
                             double *out, double *cache_k, double *cache_v) {
  int sum = 0;
  for (int a = 0; a < n_axes; ++a) sum += axes_dims[a];
  if (sum != D || D % 2 != 0 || S <= 0 || B <= 0 || H <= 0 || S_txt < 0 || S_ref < 0 ||
      S_txt + S_ref > S)
    return -1;
  double *cos_t = (double *)malloc(sizeof(double) * (size_t)S * (D / 2));
  double *sin_t = (double *)malloc(sizeof(double) * (size_t)S * (D / 2));
  if (oracle_rope_tables(ids, S, axes_dims, n_axes, theta, cos_t, sin_t) != 0) {
    free(cos_t);
    free(sin_t);
    return -1;
  }
  double *khat = (double *)malloc(sizeof(double) * (size_t)S * D);
  double *qhat = (double *)malloc(sizeof(double) * (size_t)D);
  double *z = (double *)malloc(sizeof(double) * (size_t)S);
  const double **vrows = (const double **)malloc(sizeof(double *) * (size_t)S);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      for (int64_t j = 0; j < S; ++j) {
        const int64_t off = (((int64_t)b * S + j) * H + h) * D;
        oracle_rope_apply_vec(k + off, cos_t + j * (D / 2), sin_t + j * (D / 2), D,
                              khat + j * D);
        vrows[j] = v + off;
      }
      for (int64_t r = 0; r < (rows ? n_rows : S); ++r) {
        const int64_t i = rows ? rows[r] : r;
        const int64_t off = (((int64_t)b * S + i) * H + h) * D;
        const int64_t ooff = (((int64_t)b * (rows ? n_rows : S) + r) * H + h) * D;
        oracle_rope_apply_vec(q + off, cos_t + i * (D / 2), sin_t + i * (D / 2), D, qhat);
        const int is_ref = i >= S_txt && i < S_txt + S_ref;
        attend_range(qhat, khat, vrows, is_ref ? S_txt : 0, is_ref ? S_txt + S_ref : S, D, z,
                     out + ooff);
      }
      for (int64_t r = 0; r < S_ref; ++r) {
        const int64_t coff = (((int64_t)b * S_ref + r) * H + h) * D;
        for (int c = 0; c < D; ++c) {
          cache_k[coff + c] = khat[(S_txt + r) * D + c];
          cache_v[coff + c] = vrows[S_txt + r][c];
        }
      }
    }
  free(khat);
  free(qhat);
  free(z);
  free(vrows);
  free(cos_t);
  free(sin_t);
  return 0;
}

/* Cached mode. Queries, keys and values of the tokens [txt ; img] (S_txt,
 * then the rest; ids [S, n_axes] in that order) and a cache [B, S_ref, H, D]
 * of reference keys (already rotated) and values. Every query attends to the
 * keys [txt ; cached ref ; img]. out [B, n_rows, H, D] for the query tokens
 * rows[0 .. n_rows) (every token when rows is NULL). Single threaded.
 * Returns 0, or -1 on bad arguments. */
int oracle_attention_cached(const double *q, const double *k, const double *v, int B,
                            int64_t S, int H, int D, const int32_t *ids,
                            const int32_t *axes_dims, int n_axes, double theta, int64_t S_txt,
                            const double *cache_k, const double *cache_v, int64_t S_ref,
                            const int64_t *rows, int64_t n_rows, double *out) {
  int sum = 0;
  for (int a = 0; a < n_axes; ++a) sum += axes_dims[a];
  if (sum != D || D % 2 != 0 || S <= 0 || B <= 0 || H <= 0 || S_txt < 0 || S_txt > S ||
      S_ref < 0)
    return -1;
  const int64_t Sk = S + S_ref;
  double *cos_t = (double *)malloc(sizeof(double) * (size_t)S * (D / 2));
  double *sin_t = (double *)malloc(sizeof(double) * (size_t)S * (D / 2));
  if (oracle_rope_tables(ids, S, axes_dims, n_axes, theta, cos_t, sin_t) != 0) {
    free(cos_t);
    free(sin_t);
    return -1;
  }
  double *khat = (double *)malloc(sizeof(double) * (size_t)Sk * D);
  double *qhat = (double *)malloc(sizeof(double) * (size_t)D);
  double *z = (double *)malloc(sizeof(double) * (size_t)Sk);
  const double **vrows = (const double **)malloc(sizeof(double *) * (size_t)Sk);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < H; ++h) {
      /* keys in the order [txt ; cached ref ; img] */
      for (int64_t j = 0; j < Sk; ++j) {
        if (j >= S_txt && j < S_txt + S_ref) {
          const int64_t coff = (((int64_t)b * S_ref + (j - S_txt)) * H + h) * D;
          for (int c = 0; c < D; ++c) khat[j * D + c] = cache_k[coff + c];
          vrows[j] = cache_v + coff;
        } else {
          const int64_t t = j < S_txt ? j : j - S_ref; /* token of [txt ; img] */
          const int64_t off = (((int64_t)b * S + t) * H + h) * D;
          oracle_rope_apply_vec(k + off, cos_t + t * (D / 2), sin_t + t * (D / 2), D,
                                khat + j * D);
          vrows[j] = v + off;
        }
      }
      for (int64_t r = 0; r < (rows ? n_rows : S); ++r) {
        const int64_t i = rows ? rows[r] : r;
        const int64_t off = (((int64_t)b * S + i) * H + h) * D;
        const int64_t ooff = (((int64_t)b * (rows ? n_rows : S) + r) * H + h) * D;
        oracle_rope_apply_vec(q + off, cos_t + i * (D / 2), sin_t + i * (D / 2), D, qhat);
        attend_range(qhat, khat, vrows, 0, Sk, D, z, out + ooff);
      }
    }
  free(khat);
  free(qhat);
  free(z);
  free(vrows);
  free(cos_t);
  free(sin_t);
  return 0;
}

/* Step 6: the fused Q / K / V / SwiGLU-MLP input projection of the single-stream
 * block for the token rows `rows` (all M rows when rows is NULL). x [M, dim],
 * w [3 * H * D + 2 * mlp, dim]; q, k, v [n, H, D] and act [n, mlp] for the n
 * requested rows. Returns -1 on bad sizes. */
static double proj_dot(const double *x, const double *w, int dim, int64_t n_out, int64_t n) {
  double acc = 0.0;
  const double *wn = w + n * dim; /* row n of W [n_out, dim] */
  (void)n_out;
  for (int c = 0; c < dim; ++c) acc += wn[c] * x[c];
  return acc;
}

int oracle_qkv_mlp_proj(const double *x, const double *w, int64_t M, int dim, int H, int D,
                        int64_t mlp, const int64_t *rows, int64_t n_rows, double *q, double *k,
                        double *v, double *act) {
  if (M < 0 || dim < 1 || H < 1 || D < 1 || mlp < 0) return -1;
  const int64_t inner = (int64_t)H * D;
  const int64_t n_out = 3 * inner + 2 * mlp;
  const int64_t n = rows ? n_rows : M;
  for (int64_t r = 0; r < n; ++r) {
    const int64_t i = rows ? rows[r] : r;
    if (i < 0 || i >= M) return -1;
    const double *xi = x + i * dim;
    for (int64_t c = 0; c < inner; ++c) {
      q[r * inner + c] = proj_dot(xi, w, dim, n_out, c);
      k[r * inner + c] = proj_dot(xi, w, dim, n_out, inner + c);
      v[r * inner + c] = proj_dot(xi, w, dim, n_out, 2 * inner + c);
    }
    for (int64_t j = 0; j < mlp; ++j) {
      const double g = proj_dot(xi, w, dim, n_out, 3 * inner + j);
      const double u = proj_dot(xi, w, dim, n_out, 3 * inner + mlp + j);
      act[r * mlp + j] = g / (1.0 + exp(-g)) * u;
    }
  }
  return 0;
}

/* Steps 4 and 5 together: the KV modes with the QK RMS normalisation before
 * RoPE. q and k are normalised token by token (the first S_txt tokens, text,
 * with the text weights; every other token, reference or image, with the
 * image weights) and then go through the mode unchanged; the cache holds the
 * normalised, rotated K. */
static int qk_normed_copies(const double *q, const double *k, int B, int64_t S, int H, int D,
                            const double *qw_txt, const double *kw_txt, const double *qw_img,
                            const double *kw_img, int64_t S_txt, double eps, double **qn,
                            double **kn) {
  if (qw_txt == NULL || kw_txt == NULL || qw_img == NULL || kw_img == NULL || S_txt < 0 ||
      S_txt > S || !(eps >= 0.0))
    return -1;
  const size_t n = (size_t)B * (size_t)S * (size_t)H * (size_t)D;
  *qn = (double *)malloc(sizeof(double) * (n ? n : 1));
  *kn = (double *)malloc(sizeof(double) * (n ? n : 1));
  for (int b = 0; b < B; ++b)
    for (int64_t t = 0; t < S; ++t)
      for (int h = 0; h < H; ++h) {
        const int64_t off = (((int64_t)b * S + t) * H + h) * D;
        oracle_rms_norm_vec(q + off, t < S_txt ? qw_txt : qw_img, D, eps, *qn + off);
        oracle_rms_norm_vec(k + off, t < S_txt ? kw_txt : kw_img, D, eps, *kn + off);
      }
  return 0;
}

int oracle_qknorm_attention_extract(const double *q, const double *k, const double *v, int B,
                                    int64_t S, int H, int D, const int32_t *ids,
                                    const int32_t *axes_dims, int n_axes, double theta,
                                    int64_t S_txt, int64_t S_ref, const double *qw_txt,
                                    const double *kw_txt, const double *qw_img,
                                    const double *kw_img, double eps, const int64_t *rows,
                                    int64_t n_rows, double *out, double *cache_k,
                                    double *cache_v) {
  double *qn = NULL, *kn = NULL;
  if (qk_normed_copies(q, k, B, S, H, D, qw_txt, kw_txt, qw_img, kw_img, S_txt, eps, &qn, &kn))
    return -1;
  const int rc = oracle_attention_extract(qn, kn, v, B, S, H, D, ids, axes_dims, n_axes, theta,
                                          S_txt, S_ref, rows, n_rows, out, cache_k, cache_v);
  free(qn);
  free(kn);
  return rc;
}

int oracle_qknorm_attention_cached(const double *q, const double *k, const double *v, int B,
                                   int64_t S, int H, int D, const int32_t *ids,
                                   const int32_t *axes_dims, int n_axes, double theta,
                                   int64_t S_txt, const double *cache_k, const double *cache_v,
                                   int64_t S_ref, const double *qw_txt, const double *kw_txt,
                                   const double *qw_img, const double *kw_img, double eps,
                                   const int64_t *rows, int64_t n_rows, double *out) {
  double *qn = NULL, *kn = NULL;
  if (qk_normed_copies(q, k, B, S, H, D, qw_txt, kw_txt, qw_img, kw_img, S_txt, eps, &qn, &kn))
    return -1;
  const int rc = oracle_attention_cached(qn, kn, v, B, S, H, D, ids, axes_dims, n_axes, theta,
                                         S_txt, cache_k, cache_v, S_ref, rows, n_rows, out);
  free(qn);
  free(kn);
  return rc;
}
