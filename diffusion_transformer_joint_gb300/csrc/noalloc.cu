// flux_joint_rope_attention_noalloc: the joint RoPE attention for callers
// that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a plugin inside a host
// application whose allocator owns every byte of device memory and hands out
// none, or code on a latency-critical path where cudaMalloc's implicit
// device synchronisation would stall other streams. The regular entry point
// needs a caller-provided workspace (status word + RoPE table); this one
// keeps exactly that workspace in a file-scope device array instead, so the
// caller passes only inputs and outputs. The array holds no room for the
// optional rotated-K exchange buffer, so every thread block rotates every K
// tile it loads; the output is bit-identical to the regular entry point's.
#include <cuda_runtime.h>

#include <mutex>

#include "flux_internal.h"

namespace {

constexpr int64_t kMaxTokens = FLUX_NOALLOC_MAX_TOKENS;
// status block + the packed (cos, sin) table of kMaxTokens tokens
constexpr size_t kScratchBytes = flux::kStatusBytes + static_cast<size_t>(kMaxTokens) * 64 * 4;
static_assert(kScratchBytes == 256 + 8u * 1024 * 1024, "the size the header states");

// One copy per device that loads the library, held until the process exits.
// In host code this name is a host-side stand-in, never a device address:
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];  // device address of g_scratch, per device

// Looks up (once per device, with that device current) the device address
// of g_scratch. Returns nullptr if the runtime call fails, after clearing
// the error it left pending so that it cannot surface in a later call.
void *scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int flux_joint_rope_attention_noalloc(const void *q, const void *k, const void *v,
                                                 const int32_t *txt_ids, int64_t S_txt,
                                                 const int32_t *img_ids, int64_t S_img, int B,
                                                 int H, int D, const int32_t *axes_dims,
                                                 int n_axes, double theta, void *out,
                                                 void *stream) {
  if (S_txt < 0 || S_img < 0 || S_txt > kMaxTokens || S_img > kMaxTokens - S_txt)
    return FLUX_ERR_SHAPE;
  if (D != 128) return FLUX_ERR_SHAPE;
  const int dc = flux::check_device();
  if (dc != FLUX_OK) return dc;
  void *ws = scratch_for_current_device();
  if (ws == nullptr) return FLUX_ERR_CUDA;
  // exactly the regular workspace of S tokens: the exchange buffer stays off
  const size_t bytes = flux_joint_rope_attention_workspace(S_txt + S_img, D);
  return flux_joint_rope_attention(q, k, v, txt_ids, S_txt, img_ids, S_img, B, H, D, axes_dims,
                                   n_axes, theta, out, ws, bytes, stream);
}

extern "C" int flux_joint_rope_attention_noalloc_status(void *stream) {
  const int dc = flux::check_device();
  if (dc != FLUX_OK) return dc;
  void *ws = scratch_for_current_device();
  if (ws == nullptr) return FLUX_ERR_CUDA;
  return flux_query_status(ws, stream);
}
