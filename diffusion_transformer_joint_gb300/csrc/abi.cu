// C-ABI entry points declared in include/flux_attn.h: argument checks, the
// workspace layout, and the two launches (RoPE tables, then attention).
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "flux_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

namespace flux {

// sm_103 check, cached per device ordinal.
int check_device() {
  static std::atomic<int> cached[64];  // 0 unknown, 1 ok, -1 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLUX_ERR_CUDA;
  if (dev < 0 || dev >= 64) return FLUX_ERR_UNSUPPORTED;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FLUX_ERR_CUDA;
    c = (major == 10 && minor == 3) ? 1 : -1;
    cached[dev].store(c, std::memory_order_relaxed);
  }
  return c == 1 ? FLUX_OK : FLUX_ERR_UNSUPPORTED;
}

}  // namespace flux

using flux::check_device;

extern "C" {

const char *flux_status_string(int status) {
  switch (status) {
    case FLUX_OK: return "ok";
    case FLUX_ERR_NULL: return "a required pointer is NULL";
    case FLUX_ERR_SHAPE: return "B, H, S or D out of the supported range";
    case FLUX_ERR_AXES: return "axes_dims must be positive, even, sum to D; 1 <= n_axes <= 8";
    case FLUX_ERR_ALIGN: return "q, k, v and out must be 16-byte aligned";
    case FLUX_ERR_WORKSPACE: return "workspace NULL, not 256-byte aligned, or too small";
    case FLUX_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case FLUX_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait (device timeout)";
    case FLUX_ERR_UNSUPPORTED: return "the current device is not sm_103 (GB300)";
    case FLUX_ERR_ALIAS: return "an output or scratch buffer overlaps an input or another output";
    default:
      if (status < FLUX_DEBUG_STATUS_BASE && status > FLUX_DEBUG_STATUS_BASE - 100)
        return "a checked index was out of range (checked build)";
      return "unknown status";
  }
}

int flux_rope_tables(const int32_t *ids, int64_t S, const int32_t *axes_dims, int n_axes,
                     double theta, float *cos_out, float *sin_out, void *stream) {
  if (ids == nullptr || cos_out == nullptr || sin_out == nullptr || axes_dims == nullptr)
    return FLUX_ERR_NULL;
  if (S < 1 || S > 0x7FFFFFFFLL) return FLUX_ERR_SHAPE;
  flux::RopePairs pp;
  const int rc = flux::make_rope_pairs(axes_dims, n_axes, theta, &pp);
  if (rc != FLUX_OK) return rc;
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;
  const cudaError_t e =
      flux::launch_rope_tables(ids, S, nullptr, 0, pp, flux::TableFormat::kF32Pair, cos_out,
                               sin_out, nullptr, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FLUX_OK : FLUX_ERR_CUDA;
}

int flux_rope_tables_packed(const int32_t *ids, int64_t S, const int32_t *axes_dims, int n_axes,
                            double theta, uint32_t *table_out, void *stream) {
  if (ids == nullptr || table_out == nullptr || axes_dims == nullptr) return FLUX_ERR_NULL;
  if (S < 1 || S > 0x7FFFFFFFLL) return FLUX_ERR_SHAPE;
  flux::RopePairs pp;
  const int rc = flux::make_rope_pairs(axes_dims, n_axes, theta, &pp);
  if (rc != FLUX_OK) return rc;
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;
  const cudaError_t e =
      flux::launch_rope_tables(ids, S, nullptr, 0, pp, flux::TableFormat::kPackedF16, nullptr,
                               nullptr, table_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FLUX_OK : FLUX_ERR_CUDA;
}

size_t flux_joint_rope_attention_workspace(int64_t S, int D) {
  if (S < 1 || S > 0x7FFFFFFFLL || D <= 0 || (D & 1)) return 0;
  return flux::kStatusBytes + flux::packed_table_bytes(S, D);
}
size_t flux_joint_rope_attention_krot_bytes(int B, int64_t S, int H, int D) {
  if (B < 1 || H < 1 || S < 1 || S > 0x7FFFFFFFLL || B > 65535 || H > 65535) return 0;
  return flux::krot_scratch_bytes(B, S, H, D);
}
size_t flux_joint_rope_attention_workspace_shared(int B, int64_t S, int H, int D) {
  const size_t base = flux_joint_rope_attention_workspace(S, D);
  const size_t krot = flux_joint_rope_attention_krot_bytes(B, S, H, D);
  return (base == 0 || krot == 0) ? 0 : base + krot;
}

}  // extern "C"

namespace {

// Checks of the QK-norm arguments: all four weight vectors or none; 16-byte
// aligned fp32 [128]; eps finite and >= 0; S_txt within the sequence.
int check_norm(const float *const w[4], float eps, int64_t S_txt, int64_t S) {
  if (w[0] == nullptr || w[1] == nullptr || w[2] == nullptr || w[3] == nullptr)
    return FLUX_ERR_NULL;
  for (int i = 0; i < 4; ++i)
    if (!aligned16(w[i])) return FLUX_ERR_ALIGN;
  if (!(eps >= 0.f) || !(eps < 3.0e38f) || S_txt < 0 || S_txt > S) return FLUX_ERR_SHAPE;
  return FLUX_OK;
}

// The one-call attention over heads h0 .. h0 + Hl - 1 of [B, S, H, D] tensors.
int one_call(const void *q, const void *k, const void *v, const int32_t *txt_ids, int64_t S_txt,
             const int32_t *img_ids, int64_t S_img, int B, int H, int D,
             const int32_t *axes_dims, int n_axes, double theta, const float *const norm_w[4],
             float eps, void *out, void *workspace, size_t workspace_bytes, void *stream,
             int h0, int Hl) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || axes_dims == nullptr)
    return FLUX_ERR_NULL;
  if ((S_txt > 0 && txt_ids == nullptr) || (S_img > 0 && img_ids == nullptr)) return FLUX_ERR_NULL;
  if (S_txt < 0 || S_img < 0) return FLUX_ERR_SHAPE;
  const int64_t S = S_txt + S_img;
  if (D != 128 || B < 1 || H < 1 || S < 1 || S > 0x7FFFFFFFLL || B > 65535 || H > 65535)
    return FLUX_ERR_SHAPE;
  if (h0 < 0 || Hl < 1 || h0 > H - Hl) return FLUX_ERR_SHAPE;
  if (static_cast<int64_t>(B) * H * ((S + 127) / 128) > 0x7FFFFFFFLL) return FLUX_ERR_SHAPE;
  flux::RopePairs pp;
  const int rc = flux::make_rope_pairs(axes_dims, n_axes, theta, &pp);
  if (rc != FLUX_OK) return rc;
  if (2 * pp.n_pairs != D) return FLUX_ERR_AXES;
  if (norm_w != nullptr) {
    const int nc = check_norm(norm_w, eps, S_txt, S);
    if (nc != FLUX_OK) return nc;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FLUX_ERR_ALIGN;
  const size_t tensor_bytes = static_cast<size_t>(B) * static_cast<size_t>(S) *
                              static_cast<size_t>(H) * static_cast<size_t>(D) * 2;
  if (overlaps(out, tensor_bytes, q, tensor_bytes) || overlaps(out, tensor_bytes, k, tensor_bytes) ||
      overlaps(out, tensor_bytes, v, tensor_bytes))
    return FLUX_ERR_ALIAS;
  const size_t need = flux_joint_rope_attention_workspace(S, D);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < need)
    return FLUX_ERR_WORKSPACE;
  // a workspace large enough for the exchange buffer (of the Hl heads) enables it
  const size_t need_shared = flux_joint_rope_attention_workspace_shared(B, S, Hl, D);
  const size_t used = (need_shared != 0 && workspace_bytes >= need_shared) ? need_shared : need;
  if (overlaps(workspace, used, q, tensor_bytes) || overlaps(workspace, used, k, tensor_bytes) ||
      overlaps(workspace, used, v, tensor_bytes) || overlaps(workspace, used, out, tensor_bytes))
    return FLUX_ERR_ALIAS;
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  uint32_t *table = reinterpret_cast<uint32_t *>(ws + flux::kStatusBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the table kernel clears the status word; the attention kernel overlaps
  // its start with it (programmatic dependent launch)
  if (flux::launch_rope_tables(txt_ids, S_txt, img_ids, S_img, pp, flux::TableFormat::kPackedF16,
                               nullptr, nullptr, table, st, status) != cudaSuccess)
    return FLUX_ERR_CUDA;
  void *krot = used == need ? nullptr : static_cast<void *>(ws + need);
  flux::QkNormArgs nargs{};
  if (norm_w != nullptr) nargs = {norm_w[0], norm_w[1], norm_w[2], norm_w[3], S_txt, eps};
  if (flux::launch_joint_attention(q, k, v, out, table, status, B, S, H, krot,
                                   norm_w != nullptr ? &nargs : nullptr, st, true, h0,
                                   Hl) != cudaSuccess)
    return FLUX_ERR_CUDA;
  return FLUX_OK;
}

int tabled(const void *q, const void *k, const void *v, const uint32_t *table, int B, int64_t S,
           int H, int D, int64_t S_txt, const float *const norm_w[4], float eps, void *out,
           int32_t *status, void *krot_scratch, size_t krot_bytes, void *stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || table == nullptr ||
      status == nullptr)
    return FLUX_ERR_NULL;
  if (D != 128 || B < 1 || H < 1 || S < 1 || S > 0x7FFFFFFFLL || B > 65535 || H > 65535)
    return FLUX_ERR_SHAPE;
  if (static_cast<int64_t>(B) * H * ((S + 127) / 128) > 0x7FFFFFFFLL) return FLUX_ERR_SHAPE;
  if (norm_w != nullptr) {
    const int nc = check_norm(norm_w, eps, S_txt, S);
    if (nc != FLUX_OK) return nc;
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(table))
    return FLUX_ERR_ALIGN;
  const size_t tensor_bytes = static_cast<size_t>(B) * static_cast<size_t>(S) *
                              static_cast<size_t>(H) * static_cast<size_t>(D) * 2;
  if (overlaps(out, tensor_bytes, q, tensor_bytes) || overlaps(out, tensor_bytes, k, tensor_bytes) ||
      overlaps(out, tensor_bytes, v, tensor_bytes))
    return FLUX_ERR_ALIAS;
  if (krot_scratch != nullptr) {
    if ((reinterpret_cast<uintptr_t>(krot_scratch) & 255u) != 0 ||
        krot_bytes < flux_joint_rope_attention_krot_bytes(B, S, H, D))
      return FLUX_ERR_WORKSPACE;
    const size_t kb = flux_joint_rope_attention_krot_bytes(B, S, H, D);
    if (overlaps(krot_scratch, kb, q, tensor_bytes) || overlaps(krot_scratch, kb, k, tensor_bytes) ||
        overlaps(krot_scratch, kb, v, tensor_bytes) ||
        overlaps(krot_scratch, kb, out, tensor_bytes))
      return FLUX_ERR_ALIAS;
  }
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;
  flux::QkNormArgs nargs{};
  if (norm_w != nullptr) nargs = {norm_w[0], norm_w[1], norm_w[2], norm_w[3], S_txt, eps};
  if (flux::launch_joint_attention(q, k, v, out, table, status, B, S, H, krot_scratch,
                                   norm_w != nullptr ? &nargs : nullptr,
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FLUX_ERR_CUDA;
  return FLUX_OK;
}

}  // namespace

extern "C" {

int flux_joint_rope_attention(const void *q, const void *k, const void *v,
                              const int32_t *txt_ids, int64_t S_txt, const int32_t *img_ids,
                              int64_t S_img, int B, int H, int D, const int32_t *axes_dims,
                              int n_axes, double theta, void *out, void *workspace,
                              size_t workspace_bytes, void *stream) {
  return one_call(q, k, v, txt_ids, S_txt, img_ids, S_img, B, H, D, axes_dims, n_axes, theta,
                  nullptr, 0.f, out, workspace, workspace_bytes, stream, 0, H);
}

int flux_joint_rope_attention_heads(const void *q, const void *k, const void *v,
                                    const int32_t *txt_ids, int64_t S_txt,
                                    const int32_t *img_ids, int64_t S_img, int B, int H, int h0,
                                    int H_local, int D, const int32_t *axes_dims, int n_axes,
                                    double theta, void *out, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  return one_call(q, k, v, txt_ids, S_txt, img_ids, S_img, B, H, D, axes_dims, n_axes, theta,
                  nullptr, 0.f, out, workspace, workspace_bytes, stream, h0, H_local);
}

int flux_joint_qknorm_rope_attention(const void *q, const void *k, const void *v,
                                     const int32_t *txt_ids, int64_t S_txt,
                                     const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                     const int32_t *axes_dims, int n_axes, double theta,
                                     const float *q_norm_txt, const float *k_norm_txt,
                                     const float *q_norm_img, const float *k_norm_img, float eps,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     void *stream) {
  const float *const w[4] = {q_norm_txt, k_norm_txt, q_norm_img, k_norm_img};
  return one_call(q, k, v, txt_ids, S_txt, img_ids, S_img, B, H, D, axes_dims, n_axes, theta, w,
                  eps, out, workspace, workspace_bytes, stream, 0, H);
}

int flux_joint_rope_attention_tabled(const void *q, const void *k, const void *v,
                                     const uint32_t *table, int B, int64_t S, int H, int D,
                                     void *out, int32_t *status, void *krot_scratch,
                                     size_t krot_bytes, void *stream) {
  return tabled(q, k, v, table, B, S, H, D, 0, nullptr, 0.f, out, status, krot_scratch,
                krot_bytes, stream);
}

int flux_joint_qknorm_rope_attention_tabled(const void *q, const void *k, const void *v,
                                            const uint32_t *table, int B, int64_t S, int H, int D,
                                            int64_t S_txt, const float *q_norm_txt,
                                            const float *k_norm_txt, const float *q_norm_img,
                                            const float *k_norm_img, float eps, void *out,
                                            int32_t *status, void *krot_scratch,
                                            size_t krot_bytes, void *stream) {
  const float *const w[4] = {q_norm_txt, k_norm_txt, q_norm_img, k_norm_img};
  return tabled(q, k, v, table, B, S, H, D, S_txt, w, eps, out, status, krot_scratch, krot_bytes,
                stream);
}

// ---------------------------------------------- a slice of the query rows

size_t flux_joint_rope_attention_rows_workspace(int B, int64_t S_q, int64_t S, int H, int D) {
  if (D != 128 || B < 1 || H < 1 || S_q < 1 || S < S_q || S > 0x7FFFFFFFLL || B > 65535 ||
      H > 65535 || static_cast<int64_t>(B) * H * ((S + 127) / 128) > 0x7FFFFFFFLL)
    return 0;
  const flux::AttnSegment seg{0, S_q, 0, S, 0, 0};
  return flux::kStatusBytes + flux::packed_table_bytes(S, D) +
         flux::exchange_bytes(B, S_q, S, H, &seg, 1);
}

int flux_joint_rope_attention_rows(const void *q, int64_t q0, int64_t S_q, const void *k,
                                   const void *v, const int32_t *txt_ids, int64_t S_txt,
                                   const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                   const int32_t *axes_dims, int n_axes, double theta, void *out,
                                   void *workspace, size_t workspace_bytes, void *stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || axes_dims == nullptr)
    return FLUX_ERR_NULL;
  if ((S_txt > 0 && txt_ids == nullptr) || (S_img > 0 && img_ids == nullptr)) return FLUX_ERR_NULL;
  if (S_txt < 0 || S_img < 0 || S_txt > 0x7FFFFFFFLL || S_img > 0x7FFFFFFFLL)
    return FLUX_ERR_SHAPE;
  const int64_t S = S_txt + S_img;
  if (D != 128 || B < 1 || H < 1 || S < 1 || S > 0x7FFFFFFFLL || B > 65535 || H > 65535)
    return FLUX_ERR_SHAPE;
  if (q0 < 0 || S_q < 1 || q0 > S - S_q) return FLUX_ERR_SHAPE;
  if (static_cast<int64_t>(B) * H * ((S + 127) / 128) > 0x7FFFFFFFLL) return FLUX_ERR_SHAPE;
  flux::RopePairs pp;
  const int rc = flux::make_rope_pairs(axes_dims, n_axes, theta, &pp);
  if (rc != FLUX_OK) return rc;
  if (2 * pp.n_pairs != D) return FLUX_ERR_AXES;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FLUX_ERR_ALIGN;
  const size_t row = static_cast<size_t>(H) * D * 2;
  const size_t qb = static_cast<size_t>(B) * static_cast<size_t>(S_q) * row;
  const size_t kb = static_cast<size_t>(B) * static_cast<size_t>(S) * row;
  if (overlaps(out, qb, q, qb) || overlaps(out, qb, k, kb) || overlaps(out, qb, v, kb))
    return FLUX_ERR_ALIAS;
  const size_t need = flux_joint_rope_attention_workspace(S, D);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < need)
    return FLUX_ERR_WORKSPACE;
  const size_t need_shared = flux_joint_rope_attention_rows_workspace(B, S_q, S, H, D);
  const size_t used = (need_shared != 0 && workspace_bytes >= need_shared) ? need_shared : need;
  if (overlaps(workspace, used, q, qb) || overlaps(workspace, used, k, kb) ||
      overlaps(workspace, used, v, kb) || overlaps(workspace, used, out, qb))
    return FLUX_ERR_ALIAS;
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  uint32_t *table = reinterpret_cast<uint32_t *>(ws + flux::kStatusBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (flux::launch_rope_tables(txt_ids, S_txt, img_ids, S_img, pp, flux::TableFormat::kPackedF16,
                               nullptr, nullptr, table, st, status) != cudaSuccess)
    return FLUX_ERR_CUDA;
  // queries: rows q0 .. q0 + S_q - 1 of the joint sequence, whose table rows
  // start q0 rows into the table; keys: every token
  const flux::AttnSegment seg{0, S_q, 0, S, 0, 0};
  void *xbuf = used == need ? nullptr : static_cast<void *>(ws + need);
  if (flux::launch_attention_segments(q, k, v, out, table + q0 * (D / 2), table, status, B, S_q,
                                      S, H, &seg, 1, nullptr, xbuf, nullptr, st,
                                      true) != cudaSuccess)
    return FLUX_ERR_CUDA;
  return FLUX_OK;
}

// ---------------------------------------------- reference-image KV modes

namespace {

size_t pad256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Segments of extract mode over tokens [txt ; ref ; img]: text and image
// queries over every key (key range 0), reference queries over the
// reference keys (key range 1). Returns the number of segments.
int extract_segments(int64_t S_txt, int64_t S_ref, int64_t S_img, flux::AttnSegment *sg) {
  const int64_t S = S_txt + S_ref + S_img;
  int n = 0;
  if (S_txt > 0) sg[n++] = {0, S_txt, 0, S, 0, 0};
  if (S_img > 0) sg[n++] = {S_txt + S_ref, S, 0, S, 0, 0};
  if (S_ref > 0) sg[n++] = {S_txt, S_txt + S_ref, S_txt, S_txt + S_ref, 1, 0};
  return n;
}

bool kv_shape_ok(int B, int H, int D, int64_t S) {
  return D == 128 && B >= 1 && H >= 1 && S >= 1 && S <= 0x7FFFFFFFLL && B <= 65535 &&
         H <= 65535 && static_cast<int64_t>(B) * H * ((S + 127) / 128) <= 0x3FFFFFFFLL;
}

}  // namespace

size_t flux_joint_rope_attention_extract_workspace(int B, int64_t S_txt, int64_t S_ref,
                                                   int64_t S_img, int H, int D) {
  if (S_txt < 0 || S_ref < 0 || S_img < 0 || !kv_shape_ok(B, H, D, S_txt + S_ref + S_img))
    return 0;
  const int64_t S = S_txt + S_ref + S_img;
  flux::AttnSegment sg[flux::kMaxSegments];
  const int n = extract_segments(S_txt, S_ref, S_img, sg);
  return flux::kStatusBytes + flux::packed_table_bytes(S, D) +
         flux::exchange_bytes(B, S, S, H, sg, n);
}

static int extract_call(const void *q, const void *k, const void *v, const int32_t *txt_ids,
                        int64_t S_txt, const int32_t *ref_ids, int64_t S_ref,
                        const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                        const int32_t *axes_dims, int n_axes, double theta,
                        const float *const norm_w[4], float eps, void *out, void *cache_k,
                        void *cache_v, void *workspace, size_t workspace_bytes, void *stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || axes_dims == nullptr)
    return FLUX_ERR_NULL;
  if ((S_txt > 0 && txt_ids == nullptr) || (S_ref > 0 && ref_ids == nullptr) ||
      (S_img > 0 && img_ids == nullptr) || (S_ref > 0 && (cache_k == nullptr || cache_v == nullptr)))
    return FLUX_ERR_NULL;
  if (S_txt < 0 || S_ref < 0 || S_img < 0) return FLUX_ERR_SHAPE;
  const int64_t S = S_txt + S_ref + S_img;
  if (!kv_shape_ok(B, H, D, S)) return FLUX_ERR_SHAPE;
  if (norm_w != nullptr) {
    const int nc = check_norm(norm_w, eps, S_txt, S);
    if (nc != FLUX_OK) return nc;
  }
  flux::RopePairs pp;
  const int rc = flux::make_rope_pairs(axes_dims, n_axes, theta, &pp);
  if (rc != FLUX_OK) return rc;
  if (2 * pp.n_pairs != D) return FLUX_ERR_AXES;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (S_ref > 0 && (!aligned16(cache_k) || !aligned16(cache_v))))
    return FLUX_ERR_ALIGN;
  const size_t row = static_cast<size_t>(H) * D * 2;  // bytes of one token of all heads
  const size_t tb = static_cast<size_t>(B) * S * row;
  const size_t cb = static_cast<size_t>(B) * S_ref * row;
  const size_t need = flux_joint_rope_attention_extract_workspace(B, S_txt, S_ref, S_img, H, D);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < need)
    return FLUX_ERR_WORKSPACE;
  const void *ins[3] = {q, k, v};
  for (const void *x : ins)
    if (overlaps(out, tb, x, tb) || overlaps(workspace, need, x, tb) ||
        (cb > 0 && (overlaps(cache_k, cb, x, tb) || overlaps(cache_v, cb, x, tb))))
      return FLUX_ERR_ALIAS;
  if (overlaps(workspace, need, out, tb) ||
      (cb > 0 && (overlaps(cache_k, cb, out, tb) || overlaps(cache_v, cb, out, tb) ||
                  overlaps(cache_k, cb, cache_v, cb) || overlaps(workspace, need, cache_k, cb) ||
                  overlaps(workspace, need, cache_v, cb))))
    return FLUX_ERR_ALIAS;
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  uint32_t *table = reinterpret_cast<uint32_t *>(ws + flux::kStatusBytes);
  void *xbuf = ws + flux::kStatusBytes + flux::packed_table_bytes(S, D);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the table of [txt ; ref ; img]: two launches of the two-segment table
  // kernel, the first of which clears the status word
  if (flux::launch_rope_tables(txt_ids, S_txt, ref_ids, S_ref, pp, flux::TableFormat::kPackedF16,
                               nullptr, nullptr, table, st, status) != cudaSuccess ||
      (S_img > 0 &&
       flux::launch_rope_tables(img_ids, S_img, nullptr, 0, pp, flux::TableFormat::kPackedF16,
                                nullptr, nullptr, table + (S_txt + S_ref) * (D / 2), st) !=
           cudaSuccess))
    return FLUX_ERR_CUDA;
  flux::AttnSegment sg[flux::kMaxSegments];
  const int n = extract_segments(S_txt, S_ref, S_img, sg);
  // with the norm, reference tokens (after the text) take the image weights
  flux::QkNormArgs nargs{};
  if (norm_w != nullptr) nargs = {norm_w[0], norm_w[1], norm_w[2], norm_w[3], S_txt, eps};
  if (flux::launch_attention_segments(q, k, v, out, table, table, status, B, S, S, H, sg, n,
                                      nullptr, xbuf, norm_w != nullptr ? &nargs : nullptr, st,
                                      true) != cudaSuccess)
    return FLUX_ERR_CUDA;
  if (S_ref > 0) {
    // the cache: every key tile was rotated once into the exchange buffer's
    // K copy (each is loaded by some item of a key range covering it)
    size_t flags = 0;
    {
      flux::AttnSegment one[flux::kMaxSegments];
      const int m = extract_segments(S_txt, S_ref, S_img, one);
      flags = flux::exchange_bytes(B, S, S, H, one, m) - 2 * tb;
    }
    const uint8_t *krot = static_cast<const uint8_t *>(xbuf) + flags;
    const size_t width = static_cast<size_t>(S_ref) * row, pitch = static_cast<size_t>(S) * row;
    if (cudaMemcpy2DAsync(cache_k, width, krot + S_txt * row, pitch, width, B,
                          cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
        cudaMemcpy2DAsync(cache_v, width, static_cast<const uint8_t *>(v) + S_txt * row, pitch,
                          width, B, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return FLUX_ERR_CUDA;
  }
  return FLUX_OK;
}

size_t flux_joint_rope_attention_cached_workspace(int B, int64_t S_txt, int64_t S_img,
                                                  int64_t S_ref, int H, int D) {
  if (S_txt < 0 || S_img < 0 || S_ref < 0 || S_txt + S_img < 1 ||
      !kv_shape_ok(B, H, D, S_txt + S_img + S_ref))
    return 0;
  const int64_t S_q = S_txt + S_img;
  const flux::AttnSegment all{0, S_q, 0, S_q, 0, S_ref};
  return flux::kStatusBytes + flux::packed_table_bytes(S_q, D) +
         flux::exchange_bytes(B, S_q, S_q, H, &all, 1);
}

static int cached_call(const void *q, const void *k, const void *v, const int32_t *txt_ids,
                       int64_t S_txt, const int32_t *img_ids, int64_t S_img,
                       const void *cache_k, const void *cache_v, int64_t S_ref, int B, int H,
                       int D, const int32_t *axes_dims, int n_axes, double theta,
                       const float *const norm_w[4], float eps, void *out, void *workspace,
                       size_t workspace_bytes, void *stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr || axes_dims == nullptr)
    return FLUX_ERR_NULL;
  if ((S_txt > 0 && txt_ids == nullptr) || (S_img > 0 && img_ids == nullptr) ||
      (S_ref > 0 && (cache_k == nullptr || cache_v == nullptr)))
    return FLUX_ERR_NULL;
  if (S_txt < 0 || S_img < 0 || S_ref < 0 || S_txt + S_img < 1) return FLUX_ERR_SHAPE;
  const int64_t S_q = S_txt + S_img, S_k = S_q + S_ref;
  if (!kv_shape_ok(B, H, D, S_k)) return FLUX_ERR_SHAPE;
  if (norm_w != nullptr) {
    const int nc = check_norm(norm_w, eps, S_txt, S_q);
    if (nc != FLUX_OK) return nc;
  }
  flux::RopePairs pp;
  const int rc = flux::make_rope_pairs(axes_dims, n_axes, theta, &pp);
  if (rc != FLUX_OK) return rc;
  if (2 * pp.n_pairs != D) return FLUX_ERR_AXES;
  if (n_axes > 8) return FLUX_ERR_AXES;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (S_ref > 0 && (!aligned16(cache_k) || !aligned16(cache_v))))
    return FLUX_ERR_ALIGN;
  const size_t row = static_cast<size_t>(H) * D * 2;
  const size_t tb = static_cast<size_t>(B) * S_q * row;
  const size_t cb = static_cast<size_t>(B) * S_ref * row;
  const size_t need = flux_joint_rope_attention_cached_workspace(B, S_txt, S_img, S_ref, H, D);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < need)
    return FLUX_ERR_WORKSPACE;
  const void *ins[5] = {q, k, v, cache_k, cache_v};
  const size_t sz[5] = {tb, tb, tb, cb, cb};
  for (int i = 0; i < 5; ++i)
    if (sz[i] > 0 && (overlaps(out, tb, ins[i], sz[i]) || overlaps(workspace, need, ins[i], sz[i])))
      return FLUX_ERR_ALIAS;
  if (overlaps(workspace, need, out, tb)) return FLUX_ERR_ALIAS;
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;

  // workspace: status | table of [txt ; img] | exchange buffer. The keys are
  // [txt ; img] from k, rotated here, then the cache's rows, rotated already
  // (key order does not change non-causal attention).
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  uint32_t *table = reinterpret_cast<uint32_t *>(ws + flux::kStatusBytes);
  void *xbuf = ws + flux::kStatusBytes + flux::packed_table_bytes(S_q, D);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (flux::launch_rope_tables(txt_ids, S_txt, img_ids, S_img, pp, flux::TableFormat::kPackedF16,
                               nullptr, nullptr, table, st, status) != cudaSuccess)
    return FLUX_ERR_CUDA;
  const flux::AttnSegment all{0, S_q, 0, S_q, 0, S_ref};
  const flux::PreRotatedKV cache{cache_k, cache_v, S_ref};
  // the norm acts on q and the keys of k; the cached keys arrive normalised
  flux::QkNormArgs nargs{};
  if (norm_w != nullptr) nargs = {norm_w[0], norm_w[1], norm_w[2], norm_w[3], S_txt, eps};
  if (flux::launch_attention_segments(q, k, v, out, table, table, status, B, S_q, S_q, H, &all, 1,
                                      &cache, xbuf, norm_w != nullptr ? &nargs : nullptr, st,
                                      true) != cudaSuccess)
    return FLUX_ERR_CUDA;
  return FLUX_OK;
}

int flux_joint_rope_attention_extract(const void *q, const void *k, const void *v,
                                      const int32_t *txt_ids, int64_t S_txt,
                                      const int32_t *ref_ids, int64_t S_ref,
                                      const int32_t *img_ids, int64_t S_img, int B, int H, int D,
                                      const int32_t *axes_dims, int n_axes, double theta,
                                      void *out, void *cache_k, void *cache_v, void *workspace,
                                      size_t workspace_bytes, void *stream) {
  return extract_call(q, k, v, txt_ids, S_txt, ref_ids, S_ref, img_ids, S_img, B, H, D,
                      axes_dims, n_axes, theta, nullptr, 0.f, out, cache_k, cache_v, workspace,
                      workspace_bytes, stream);
}

int flux_joint_qknorm_rope_attention_extract(
    const void *q, const void *k, const void *v, const int32_t *txt_ids, int64_t S_txt,
    const int32_t *ref_ids, int64_t S_ref, const int32_t *img_ids, int64_t S_img, int B, int H,
    int D, const int32_t *axes_dims, int n_axes, double theta, const float *q_norm_txt,
    const float *k_norm_txt, const float *q_norm_img, const float *k_norm_img, float eps,
    void *out, void *cache_k, void *cache_v, void *workspace, size_t workspace_bytes,
    void *stream) {
  const float *const w[4] = {q_norm_txt, k_norm_txt, q_norm_img, k_norm_img};
  return extract_call(q, k, v, txt_ids, S_txt, ref_ids, S_ref, img_ids, S_img, B, H, D,
                      axes_dims, n_axes, theta, w, eps, out, cache_k, cache_v, workspace,
                      workspace_bytes, stream);
}

int flux_joint_rope_attention_cached(const void *q, const void *k, const void *v,
                                     const int32_t *txt_ids, int64_t S_txt,
                                     const int32_t *img_ids, int64_t S_img, const void *cache_k,
                                     const void *cache_v, int64_t S_ref, int B, int H, int D,
                                     const int32_t *axes_dims, int n_axes, double theta,
                                     void *out, void *workspace, size_t workspace_bytes,
                                     void *stream) {
  return cached_call(q, k, v, txt_ids, S_txt, img_ids, S_img, cache_k, cache_v, S_ref, B, H, D,
                     axes_dims, n_axes, theta, nullptr, 0.f, out, workspace, workspace_bytes,
                     stream);
}

int flux_joint_qknorm_rope_attention_cached(
    const void *q, const void *k, const void *v, const int32_t *txt_ids, int64_t S_txt,
    const int32_t *img_ids, int64_t S_img, const void *cache_k, const void *cache_v,
    int64_t S_ref, int B, int H, int D, const int32_t *axes_dims, int n_axes, double theta,
    const float *q_norm_txt, const float *k_norm_txt, const float *q_norm_img,
    const float *k_norm_img, float eps, void *out, void *workspace, size_t workspace_bytes,
    void *stream) {
  const float *const w[4] = {q_norm_txt, k_norm_txt, q_norm_img, k_norm_img};
  return cached_call(q, k, v, txt_ids, S_txt, img_ids, S_img, cache_k, cache_v, S_ref, B, H, D,
                     axes_dims, n_axes, theta, w, eps, out, workspace, workspace_bytes, stream);
}

int flux_query_status(const void *workspace, void *stream) {
  if (workspace == nullptr) return FLUX_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return FLUX_ERR_CUDA;
  int status = 0;
  if (cudaMemcpy(&status, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FLUX_ERR_CUDA;
  return status;
}

int flux_qkv_mlp_proj(const void *x, const void *w, int64_t M, int dim, int H, int D,
                      int64_t mlp_hidden, void *q, void *k, void *v, void *act, int32_t *status,
                      void *stream) {
  if (x == nullptr || w == nullptr || q == nullptr || k == nullptr || v == nullptr ||
      status == nullptr || (mlp_hidden > 0 && act == nullptr))
    return FLUX_ERR_NULL;
  if (D != 128 || M < 1 || M > 0x7FFFFFFFLL || dim < 64 || dim % 64 != 0 || H < 1 ||
      H > 65535 || mlp_hidden < 0 || mlp_hidden % 128 != 0 || mlp_hidden > 0x3FFFFFFFLL)
    return FLUX_ERR_SHAPE;
  const int64_t inner = static_cast<int64_t>(H) * D;
  if (3 * inner + 2 * mlp_hidden > 0x7FFFFFFFLL) return FLUX_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      (mlp_hidden > 0 && !aligned16(act)))
    return FLUX_ERR_ALIGN;
  const size_t xb = static_cast<size_t>(M) * dim * 2;
  const size_t wb = static_cast<size_t>(3 * inner + 2 * mlp_hidden) * dim * 2;
  const size_t tb = static_cast<size_t>(M) * inner * 2;
  const size_t ab = static_cast<size_t>(M) * mlp_hidden * 2;
  const void *outs[4] = {q, k, v, act};
  const size_t osz[4] = {tb, tb, tb, ab};
  for (int i = 0; i < 4; ++i) {
    if (osz[i] == 0) continue;
    if (overlaps(outs[i], osz[i], x, xb) || overlaps(outs[i], osz[i], w, wb) ||
        overlaps(outs[i], osz[i], status, sizeof(int32_t)))
      return FLUX_ERR_ALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (osz[j] > 0 && overlaps(outs[i], osz[i], outs[j], osz[j])) return FLUX_ERR_ALIAS;
  }
  const int dc = check_device();
  if (dc != FLUX_OK) return dc;
  if (flux::launch_qkv_mlp_proj(x, w, M, dim, H, mlp_hidden, q, k, v, act, status,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FLUX_ERR_CUDA;
  return FLUX_OK;
}

}  // extern "C"
