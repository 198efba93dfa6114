/*
 * flux_attn.h: C-ABI of the GB300 (sm_103a) joint RoPE attention library.
 *
 * The operation is the attention core of the FLUX.2 MMDiT denoiser: the text
 * and image (plus reference-image) tokens form one joint sequence, queries
 * and keys are rotated by a 4-axis N-D RoPE built from per-token (T, H, W, L)
 * position ids, and every token attends to every token.
 *
 * Sources for the definition:
 *   - "Diffusers 中 Flux2Transformer2DModel 全面解析", sections
 *     "模型配置参数全解" (attention_head_dim 128, axes_dims_rope (32,32,32,32),
 *     rope_theta 2000), "前向传播输入输出约定" (4-d position ids whose last
 *     dimension equals the number of axes; one id set shared by the batch;
 *     each axis gets its own 1-D RoPE and the axes are concatenated) and
 *     "内部架构双流块与单流块" (text and image streams concatenated for one
 *     joint attention).
 *   - "FLUX.2 [klein]" survey page, section "模型架构" (axes_dim always
 *     [32,32,32,32], theta 2000; N-D RoPE (EmbedND); reference-image tokens
 *     concatenated with the noisy tokens).
 *   - "Transformer架构解析FLUX.2-klein-base-9b-nvfp4", section 2
 *     "核心引擎自注意力机制如何工作" (scaled dot-product attention:
 *     softmax(Q K^T / sqrt(d_k)) V with d_k the head size).
 *
 * Entry points: the RoPE tables (fp32 and packed); the joint attention in one
 * call (tables + attention) or with a caller-built table, both also with the
 * QK RMS normalisation fused in front of the rotation; the one-call attention
 * over a range of heads or over a slice of the query rows (for tensor- and
 * sequence-parallel callers); the reference-image KV
 * modes (extract, cached); and the single-stream block's fused input
 * projection (Q, K, V and the SwiGLU-activated MLP input from one GEMM), the
 * producer of the attention's inputs.
 *
 * Conventions shared by every entry point:
 *   - Device pointers refer to memory on the CUDA device that is current on
 *     the calling thread; the caller owns every buffer, and the library
 *     allocates nothing and frees nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Work is enqueued asynchronously; nothing synchronises.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns a negative flux_status and enqueues nothing. A launch
 *     failure returns FLUX_ERR_CUDA.
 *   - Device-side failures (a bounded wait inside a kernel that ran out)
 *     never trap: the kernel records FLUX_ERR_DEVICE_TIMEOUT in a status word
 *     and returns. Entry points with a workspace keep the word at its start
 *     (read it with flux_query_status()); the tabled attention and the
 *     projection take a caller-owned device int32 instead.
 */
#ifndef FLUX_ATTN_H
#define FLUX_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLUX_OK = 0,
  FLUX_ERR_NULL = -1,           /* a required pointer is NULL */
  FLUX_ERR_SHAPE = -2,          /* B, H, S or D out of the supported range */
  FLUX_ERR_AXES = -3,           /* axes_dims not even / not summing to D / n_axes out of range */
  FLUX_ERR_ALIGN = -4,          /* a pointer is not 16-byte aligned */
  FLUX_ERR_WORKSPACE = -5,      /* workspace NULL, misaligned (256 B) or too small */
  FLUX_ERR_CUDA = -6,           /* a CUDA runtime call or launch failed */
  FLUX_ERR_DEVICE_TIMEOUT = -7, /* a kernel's bounded wait ran out (see flux_query_status) */
  FLUX_ERR_UNSUPPORTED = -8,    /* the current device is not sm_103 */
  FLUX_ERR_ALIAS = -9           /* an output or scratch buffer overlaps an input or another output */
} flux_status;

/* Checked builds of the library only (compiled with -DFLUX_DEBUG): when one of
 * the attention kernel's index checks fails, the kernel skips that access and
 * its status word reads FLUX_DEBUG_STATUS_BASE - site, site >= 1 naming the
 * access (see DbgSite in csrc/attention_sm103a.cu). Release builds never
 * produce these codes. */
#define FLUX_DEBUG_STATUS_BASE (-1000)

/* Largest number of RoPE axes accepted (FLUX.2 uses 4). */
#define FLUX_MAX_AXES 8

/*
 * flux_rope_tables: cos/sin tables of the N-D RoPE.
 *
 * For token s and rotation pair p (channels 2p and 2p+1 of a head), with p in
 * axis a's block [o_a, o_a + axes_dims[a]/2), o_a = sum_{a'<a} axes_dims[a']/2,
 * and j = p - o_a:
 *     angle(s, p) = ids[s, a] * theta^(-2 j / axes_dims[a])
 *     cos_out[s, p] = cos(angle),  sin_out[s, p] = sin(angle)
 * The frequency theta^(-2j/d_a) / (2 pi) turns per unit id is formed on the
 * host in extended precision as a 0.64 fixed-point fraction; per entry the
 * angle's fractional turn is the exact 64-bit product id * frequency
 * (mod 2^64), and cosine and sine of it are evaluated in fp32, so outputs are
 * accurate to a few 1e-7 for any int32 id.
 *
 *   ids        device, int32 [S, n_axes] row-major (one row per token).
 *   S          number of tokens, 1 <= S <= 2^31 - 1.
 *   axes_dims  HOST, int32 [n_axes]; each entry positive and even, the sum
 *              P2 = sum(axes_dims) at most 512.
 *   n_axes     1 .. FLUX_MAX_AXES.
 *   theta      frequency base, > 0 (2000 for FLUX.2).
 *   cos_out, sin_out  device, fp32 [S, P2/2] row-major; written, not read.
 *   stream     cudaStream_t as void*.
 * Returns FLUX_OK or a negative flux_status.
 */
int flux_rope_tables(const int32_t *ids, int64_t S, const int32_t *axes_dims, int n_axes,
                     double theta, float *cos_out, float *sin_out, void *stream);

/*
 * flux_rope_tables_packed: the same table, one 32-bit word per (token, pair):
 * fp16 cos in bits 0-15 and fp16 sin in bits 16-31 (round to nearest even,
 * |error| <= 2^-12). This is the format the attention kernel stages next to
 * each key tile; flux_joint_rope_attention_tabled takes it.
 *
 *   ids, S, axes_dims, n_axes, theta, stream  as for flux_rope_tables.
 *   table_out  device, uint32 [S, sum(axes_dims)/2] row-major, 16-byte aligned.
 */
int flux_rope_tables_packed(const int32_t *ids, int64_t S, const int32_t *axes_dims, int n_axes,
                            double theta, uint32_t *table_out, void *stream);

/*
 * flux_joint_rope_attention_workspace: bytes of device workspace that
 * flux_joint_rope_attention needs for a joint sequence of S tokens and head
 * width D: a 256-byte status block plus the packed RoPE table
 * (S * (D/2) * 4 bytes, rounded up to 256). Returns 0 when S < 1 or D is not
 * positive and even.
 */
size_t flux_joint_rope_attention_workspace(int64_t S, int D);

/*
 * flux_joint_rope_attention_krot_bytes: bytes of the optional exchange
 * buffer for [B, S, H, D] inputs (D == 128): one 8-byte flag per (batch,
 * head, 128-key tile, RoPE warp) padded to 256 bytes, then bf16 [B, S, H, D]
 * copies of K and of Q after RoPE. With it the thread blocks that work on one
 * head at the same time rotate different K tiles, publish them there and load
 * the tiles others published instead of rotating every tile themselves, and
 * each block rotates its next work item's Q rows ahead of time; the result is
 * bit-identical either way. Contents need no initialisation and are
 * meaningless after a call. Returns 0 for shapes the attention rejects.
 *
 * flux_joint_rope_attention_workspace_shared: flux_joint_rope_attention_workspace
 * (S, D) + flux_joint_rope_attention_krot_bytes(B, S, H, D); a workspace at
 * least this large makes flux_joint_rope_attention use the exchange buffer.
 */
size_t flux_joint_rope_attention_krot_bytes(int B, int64_t S, int H, int D);
size_t flux_joint_rope_attention_workspace_shared(int B, int64_t S, int H, int D);

/*
 * flux_joint_rope_attention: out = softmax(RoPE(q) RoPE(k)^T / sqrt(D)) v
 * over the joint token sequence [txt ; img], non-causal, per batch element
 * and head.
 *
 *   q, k, v    device, bf16 [B, S, H, D] row-major (D fastest), S = S_txt + S_img,
 *              text tokens first. 16-byte aligned.
 *   txt_ids    device, int32 [S_txt, n_axes]; may be NULL when S_txt == 0.
 *   img_ids    device, int32 [S_img, n_axes]; may be NULL when S_img == 0.
 *              The same ids apply to every batch element.
 *   B, H       batch and heads, >= 1, B * H * ceil(S/128) < 2^31.
 *   D          head width; must be 128.
 *   axes_dims  HOST, int32 [n_axes], even entries summing to D.
 *   theta      RoPE frequency base (2000 for FLUX.2).
 *   out        device, bf16 [B, S, H, D], 16-byte aligned, must not overlap q/k/v.
 *   workspace  device, >= flux_joint_rope_attention_workspace(S, D) bytes,
 *              256-byte aligned, owned by the caller and not shared by calls
 *              in flight at the same time; must not overlap q, k, v or out
 *              (FLUX_ERR_ALIAS). Its status word is cleared by each call
 *              before the attention kernel runs. With at least
 *              flux_joint_rope_attention_workspace_shared(B, S, H, D) bytes
 *              its tail serves as the rotated-K exchange buffer.
 *   stream     cudaStream_t as void*.
 *
 * Numerics: bf16 inputs; the RoPE table is built in fp64/fp32 and stored as
 * fp16 (cos, sin) pairs; the rotation runs in fp32 and is rounded to bf16 for
 * the tensor-core products; fp32 accumulation and softmax; P is rounded to
 * bf16 for the P V product; bf16 output rounded to nearest even.
 *
 * Returns FLUX_OK when both kernels were enqueued, else a negative status.
 * Requires an sm_103 device (GB300).
 */
int flux_joint_rope_attention(const void *q, const void *k, const void *v,
                              const int32_t *txt_ids, int64_t S_txt,
                              const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                              const int32_t *axes_dims, int n_axes, double theta, void *out,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * flux_joint_rope_attention_heads: flux_joint_rope_attention restricted to
 * the heads h0 .. h0 + H_local - 1 of [B, S, H, D] tensors, for
 * tensor-parallel callers ("Diffusers 中 Flux2Transformer2DModel 全面解析",
 * section 并行化支持: Q, K and V are projected column-wise, so each rank owns
 * a contiguous range of heads and attention needs no exchange between ranks).
 *
 *   q, k, v, out   the full [B, S, H, D] tensors (token stride H * D); only the
 *                  rows of heads h0 .. h0 + H_local - 1 are read or written,
 *                  the other heads of out are left untouched.
 *   h0, H_local    0 <= h0, H_local >= 1, h0 + H_local <= H (else FLUX_ERR_SHAPE).
 *   workspace      >= flux_joint_rope_attention_workspace(S, D) bytes; with at
 *                  least flux_joint_rope_attention_workspace_shared(B, S,
 *                  H_local, D) bytes the exchange buffer (sized for the H_local
 *                  heads) is used.
 * Everything else as flux_joint_rope_attention, whose output for these heads
 * it reproduces bit for bit.
 */
int flux_joint_rope_attention_heads(const void *q, const void *k, const void *v,
                                    const int32_t *txt_ids, int64_t S_txt,
                                    const int32_t *img_ids, int64_t S_img, int B, int H, int h0,
                                    int H_local, int D, const int32_t *axes_dims, int n_axes,
                                    double theta, void *out, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * flux_joint_rope_attention_rows: the joint attention of a contiguous slice of
 * the query tokens over every key, for sequence-parallel callers ("Diffusers
 * 中 Flux2Transformer2DModel 全面解析", section 并行化支持: the context-parallel
 * plan splits the sequence dimension; each rank keeps its query rows and needs
 * every key and value, which the caller gathers before this call).
 *
 *   q          device, bf16 [B, S_q, H, D]: the query rows of joint tokens
 *              q0 .. q0 + S_q - 1 of the sequence [txt ; img].
 *   q0, S_q    0 <= q0, S_q >= 1, q0 + S_q <= S = S_txt + S_img.
 *   k, v       device, bf16 [B, S, H, D]: every token's key and value.
 *   txt_ids, img_ids  the ids of the whole sequence, as flux_joint_rope_attention.
 *   out        device, bf16 [B, S_q, H, D]: the output rows of those tokens.
 *   workspace  >= flux_joint_rope_attention_workspace(S, D) bytes (status word
 *              and the table of all S tokens); with at least
 *              flux_joint_rope_attention_rows_workspace(B, S_q, S, H, D) bytes
 *              its tail serves as the exchange buffer.
 * Everything else as flux_joint_rope_attention. The query rows are processed
 * in their own 256-row blocks, so the summation order over keys may differ
 * from a call over the whole sequence (the result agrees to rounding).
 */
int flux_joint_rope_attention_rows(const void *q, int64_t q0, int64_t S_q, const void *k,
                                   const void *v, const int32_t *txt_ids, int64_t S_txt,
                                   const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                   const int32_t *axes_dims, int n_axes, double theta, void *out,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Workspace of flux_joint_rope_attention_rows with the exchange buffer; 0 for
 * unsupported sizes. */
size_t flux_joint_rope_attention_rows_workspace(int B, int64_t S_q, int64_t S, int H, int D);

/*
 * flux_joint_rope_attention_tabled: the same attention, with the RoPE table
 * supplied by the caller (built once by flux_rope_tables_packed for the joint
 * id sequence and reused, e.g. by every attention layer of one denoiser step:
 * the position ids do not change between layers).
 *
 *   q, k, v, out  as for flux_joint_rope_attention, [B, S, H, D], D == 128.
 *   table         device, uint32 [S, D/2] as written by flux_rope_tables_packed;
 *                 16-byte aligned.
 *   status        device int32 word; the kernel writes FLUX_ERR_DEVICE_TIMEOUT
 *                 there if a bounded wait runs out and never writes it
 *                 otherwise (the caller clears it).
 *   krot_scratch  device, NULL or >= flux_joint_rope_attention_krot_bytes(B, S,
 *                 H, D) bytes (krot_bytes), 256-byte aligned, not overlapping
 *                 q, k, v or out, not shared by calls in flight at the same
 *                 time: the rotated-K exchange buffer. NULL: every thread
 *                 block rotates every K tile it loads.
 *   stream        cudaStream_t as void*.
 * Returns FLUX_OK when the kernel was enqueued, else a negative status
 * (FLUX_ERR_WORKSPACE for a misaligned or short krot_scratch).
 */
int flux_joint_rope_attention_tabled(const void *q, const void *k, const void *v,
                                     const uint32_t *table, int B, int64_t S, int H, int D,
                                     void *out, int32_t *status, void *krot_scratch,
                                     size_t krot_bytes, void *stream);

/*
 * flux_joint_qknorm_rope_attention: flux_joint_rope_attention with the QK RMS
 * normalisation that precedes RoPE in FLUX.2's attention ("Diffusers 中
 * Flux2Transformer2DModel 全面解析", sections 内部架构双流块与单流块: Q and K
 * are RMS-normalised right after their projections, text and image streams
 * with their own weights; 并行化支持: over the whole head_dim; 模型配置参数全解:
 * eps 1e-6). Every Q and K head vector x[D] becomes
 *   x / sqrt(mean over the D channels of x^2 + eps) * w
 * before the rotation, with w the text weights for the first S_txt tokens and
 * the image weights for the others; V is not normalised.
 *
 *   q_norm_txt, k_norm_txt, q_norm_img, k_norm_img
 *                device fp32 [D], 16-byte aligned (pass the same vectors for
 *                both streams to use one weight set).
 *   eps          finite, >= 0.
 * Other arguments, layouts and return codes as flux_joint_rope_attention.
 * Numerics: the norm and the rotation run in fp32 and round to bf16 once.
 */
int flux_joint_qknorm_rope_attention(const void *q, const void *k, const void *v,
                                     const int32_t *txt_ids, int64_t S_txt,
                                     const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                     const int32_t *axes_dims, int n_axes, double theta,
                                     const float *q_norm_txt, const float *k_norm_txt,
                                     const float *q_norm_img, const float *k_norm_img, float eps,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * flux_joint_qknorm_rope_attention_tabled: flux_joint_rope_attention_tabled
 * with the QK normalisation above; S_txt (0 .. S) is the number of leading
 * text tokens, which use the text weights.
 */
int flux_joint_qknorm_rope_attention_tabled(const void *q, const void *k, const void *v,
                                            const uint32_t *table, int B, int64_t S, int H, int D,
                                            int64_t S_txt, const float *q_norm_txt,
                                            const float *k_norm_txt, const float *q_norm_img,
                                            const float *k_norm_img, float eps, void *out,
                                            int32_t *status, void *krot_scratch,
                                            size_t krot_bytes, void *stream);

/*
 * Reference-image KV modes ("Diffusers 中 Flux2Transformer2DModel 全面解析",
 * section 参考图 KV 缓存机制). The cache holds the reference tokens' K after
 * RoPE and their V, bf16 [B, S_ref, H, D] each.
 *
 * flux_joint_rope_attention_extract: tokens [txt ; ref ; img] (the order of
 * the extract mode; q, k, v, out are [B, S, H, D] with S = S_txt + S_ref +
 * S_img, ids given per segment, each [S_seg, n_axes], NULL when empty).
 * Reference queries attend to the reference keys only; text and image
 * queries attend to every key. cache_k / cache_v (device, [B, S_ref, H, D],
 * 16-byte aligned, not overlapping anything else; may be NULL when S_ref is
 * 0) receive the reference tokens' rotated K (the bf16 values the kernel
 * used) and their V.
 *   workspace  >= flux_joint_rope_attention_extract_workspace(B, S_txt, S_ref,
 *              S_img, H, D) bytes, 256-byte aligned (status word first, as for
 *              flux_query_status).
 * Other arguments and return codes as flux_joint_rope_attention.
 */
size_t flux_joint_rope_attention_extract_workspace(int B, int64_t S_txt, int64_t S_ref,
                                                   int64_t S_img, int H, int D);
int flux_joint_rope_attention_extract(const void *q, const void *k, const void *v,
                                      const int32_t *txt_ids, int64_t S_txt,
                                      const int32_t *ref_ids, int64_t S_ref,
                                      const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                      const int32_t *axes_dims, int n_axes, double theta,
                                      void *out, void *cache_k, void *cache_v, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * flux_joint_rope_attention_cached: the cached mode. q, k, v, out are
 * [B, S_txt + S_img, H, D] for the tokens [txt ; img]; every query attends to
 * the keys [txt ; cached ref ; img] and the values in the same order. The
 * cached K is used as stored (already rotated, not rotated again); the
 * kernel reads the cache in place, after the keys of k (the order of the
 * keys does not change non-causal attention).
 *   cache_k, cache_v  device [B, S_ref, H, D] bf16, 16-byte aligned, as
 *                     written by flux_joint_rope_attention_extract; NULL when
 *                     S_ref is 0.
 *   workspace  >= flux_joint_rope_attention_cached_workspace(B, S_txt, S_img,
 *              S_ref, H, D) bytes, 256-byte aligned: the status word, the
 *              table of [txt ; img] and the exchange buffer of rotated K / Q.
 * Other arguments and return codes as flux_joint_rope_attention.
 */
size_t flux_joint_rope_attention_cached_workspace(int B, int64_t S_txt, int64_t S_img,
                                                  int64_t S_ref, int H, int D);
int flux_joint_rope_attention_cached(const void *q, const void *k, const void *v,
                                     const int32_t *txt_ids, int64_t S_txt,
                                     const int32_t *img_ids, int64_t S_img, const void *cache_k,
                                     const void *cache_v, int64_t S_ref, int B, int H, int D,
                                     const int32_t *axes_dims, int n_axes, double theta,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * flux_qkv_mlp_proj: the single-stream block's fused input projection
 * ("Diffusers 中 Flux2Transformer2DModel 全面解析", sections 内部架构双流块与单流块:
 * one linear layer, to_qkv_mlp_proj, yields Q, K, V and the MLP input; 激活函数与
 * FFN: the SwiGLU gate is fused into it and the activation halves the width;
 * 并行化支持: the packed MLP features are two equal halves, gate then linear).
 * With y = x W^T (fp32 accumulation, no bias) and inner = H * D:
 *   q = y[:, 0:inner], k = y[:, inner:2 inner], v = y[:, 2 inner:3 inner],
 *   act = silu(y[:, 3 inner:3 inner + mlp]) * y[:, 3 inner + mlp:3 inner + 2 mlp],
 * silu(g) = g / (1 + exp(-g)); every output rounded once to bf16 (nearest even).
 *
 *   x          device, bf16 [M, dim] row-major (M = B * S tokens), 16-byte aligned.
 *   w          device, bf16 [3 * H * D + 2 * mlp_hidden, dim] row-major (a
 *              linear layer's weight: one row per output feature), 16-byte aligned.
 *   M          tokens, >= 1.  dim: a multiple of 64.  D == 128.
 *   mlp_hidden MLP width (mlp_ratio * inner for FLUX.2), a multiple of 128; 0: none.
 *   q, k, v    device, bf16 [M, H, D] each (= [B, S, H, D], the attention's
 *              layout), 16-byte aligned; written, not read.
 *   act        device, bf16 [M, mlp_hidden], 16-byte aligned; NULL when
 *              mlp_hidden is 0.
 *   status     device int32 word; the kernel writes FLUX_ERR_DEVICE_TIMEOUT
 *              there if a bounded wait runs out and never writes it otherwise.
 *   No output may overlap x, w, status or another output (FLUX_ERR_ALIAS).
 * Returns FLUX_OK when the kernel was enqueued, else a negative status.
 */
int flux_qkv_mlp_proj(const void *x, const void *w, int64_t M, int dim, int H, int D,
                      int64_t mlp_hidden, void *q, void *k, void *v, void *act, int32_t *status,
                      void *stream);

/*
 * flux_joint_qknorm_rope_attention_extract / _cached: the two KV modes with
 * the QK RMS normalisation before RoPE (as flux_joint_qknorm_rope_attention:
 * text tokens, the first S_txt, with the text weights; every other token,
 * reference or image, with the image weights). In extract mode the cache
 * receives the normalised, rotated K; in cached mode the cached K is used as
 * stored (normalised and rotated already) while q and the keys of k are
 * normalised. Workspace sizes as for the plain modes; other arguments and
 * return codes as flux_joint_rope_attention_extract / _cached and
 * flux_joint_qknorm_rope_attention.
 */
int flux_joint_qknorm_rope_attention_extract(
    const void *q, const void *k, const void *v, const int32_t *txt_ids, int64_t S_txt,
    const int32_t *ref_ids, int64_t S_ref, const int32_t *img_ids, int64_t S_img, int B, int H,
    int D, const int32_t *axes_dims, int n_axes, double theta, const float *q_norm_txt,
    const float *k_norm_txt, const float *q_norm_img, const float *k_norm_img, float eps,
    void *out, void *cache_k, void *cache_v, void *workspace, size_t workspace_bytes,
    void *stream);
int flux_joint_qknorm_rope_attention_cached(
    const void *q, const void *k, const void *v, const int32_t *txt_ids, int64_t S_txt,
    const int32_t *img_ids, int64_t S_img, const void *cache_k, const void *cache_v,
    int64_t S_ref, int B, int H, int D, const int32_t *axes_dims, int n_axes, double theta,
    const float *q_norm_txt, const float *k_norm_txt, const float *q_norm_img,
    const float *k_norm_img, float eps, void *out, void *workspace, size_t workspace_bytes,
    void *stream);

/* Largest joint sequence (S_txt + S_img) that flux_joint_rope_attention_noalloc
 * accepts. Its scratch array is 256 + 32768 * 64 * 4 bytes (8 MiB + 256 B: the
 * status word and one packed (cos, sin) table) on every device that loads this
 * library, held until the process exits. */
#define FLUX_NOALLOC_MAX_TOKENS 32768

/*
 * flux_joint_rope_attention_noalloc: flux_joint_rope_attention without a
 * caller workspace. The pages have no counterpart; it exists for callers that
 * cannot allocate device memory: a plugin inside a host application whose
 * allocator owns all device memory and gives plugins none, or code that must
 * not call cudaMalloc because it can synchronise the device and stall other
 * streams. The caller still passes inputs and outputs; nothing is allocated
 * or freed (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 * Scratch (the status word and the RoPE table) lives in one fixed file-scope
 * device array of the library, one per device. Consequences:
 *   - S_txt + S_img above FLUX_NOALLOC_MAX_TOKENS returns FLUX_ERR_SHAPE and
 *     launches nothing; D must be 128 as for the regular entry point.
 *   - The array has no room for the rotated-K exchange buffer, so every
 *     thread block rotates every K tile it loads. The output is bit-identical
 *     to flux_joint_rope_attention's on the same inputs.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins on the device.
 *   - Every call shares the one array and it keeps the last call's contents.
 *     Each call clears the status word and rewrites the table before the
 *     attention kernel reads them, so results do not depend on earlier
 *     calls; but calls that overlap on the GPU (different streams, or
 *     different host threads, without ordering between them) race on the
 *     array and give undefined results. Order them on one stream.
 * Arguments, layouts and the other return codes are those of
 * flux_joint_rope_attention, with the device check made first; FLUX_ERR_CUDA
 * also when the address lookup fails.
 */
int flux_joint_rope_attention_noalloc(const void *q, const void *k, const void *v,
                                      const int32_t *txt_ids, int64_t S_txt,
                                      const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                      const int32_t *axes_dims, int n_axes, double theta,
                                      void *out, void *stream);

/*
 * flux_joint_rope_attention_noalloc_status: synchronises `stream` and returns
 * the device status word that the last flux_joint_rope_attention_noalloc call
 * on the current device left in the library's array: FLUX_OK, or
 * FLUX_ERR_DEVICE_TIMEOUT when its kernel gave up a bounded wait (its output
 * is then not valid). Pass the stream that call was made on; a later call
 * clears the word. FLUX_ERR_CUDA when the synchronisation, the copy or the
 * address lookup fails; FLUX_ERR_UNSUPPORTED on a device that is not sm_103.
 * Allocates nothing.
 */
int flux_joint_rope_attention_noalloc_status(void *stream);

/*
 * flux_query_status: synchronises `stream`, reads the device status word of
 * `workspace` and returns it (FLUX_OK, or FLUX_ERR_DEVICE_TIMEOUT when a
 * kernel of the last call gave up a bounded wait). FLUX_ERR_CUDA when the
 * synchronisation or the copy fails.
 */
int flux_query_status(const void *workspace, void *stream);

/* flux_status_string: static description of a status code (never NULL). */
const char *flux_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* FLUX_ATTN_H */
