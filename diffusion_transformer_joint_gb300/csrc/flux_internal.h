// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "flux_attn.h"

namespace flux {

// FLUX_OK if the current device is an sm_103 part (cached per device),
// FLUX_ERR_UNSUPPORTED if not, FLUX_ERR_CUDA if the runtime cannot tell.
int check_device();

// Number of SMs of the current device (cached per device ordinal, atomically);
// 0 if the runtime cannot tell.
int sm_count_current_device();

// Largest rotation-pair count of one head (head width 512).
constexpr int kMaxPairs = 256;

// Per-pair RoPE parameters handed to the table kernel by value: the axis a
// pair belongs to, and its frequency in turns per unit of position id,
// theta^(-2j/d_a) / (2 pi) (j the pair's index inside its axis of width
// d_a), as an unsigned 0.64 fixed-point fraction of a turn (it is < 1).
struct RopePairs {
  int n_pairs;
  int n_axes;
  uint8_t axis[kMaxPairs];
  uint64_t turns_q64[kMaxPairs];
};

// Fills `pp` from host axes_dims; returns FLUX_OK or FLUX_ERR_AXES.
int make_rope_pairs(const int32_t *axes_dims, int n_axes, double theta, RopePairs *pp);

// Output formats of the table kernel.
enum class TableFormat {
  kF32Pair,    // cos [S, P] and sin [S, P] fp32 (flux_rope_tables)
  kPackedF16,  // one uint32 per (token, pair): fp16 cos in bits 0-15, fp16 sin in 16-31
};

// Enqueues the table kernel over the joint id sequence [seg0 ; seg1]. For
// kPackedF16 the table goes to `packed` ([S, P] uint32) and cos/sin are unused.
// `clear` (nullable): a device int the kernel sets to 0 (a call's status
// word). The kernel lets a programmatically dependent launch (an attention
// kernel launched with pdl) begin as soon as it starts.
cudaError_t launch_rope_tables(const int32_t *ids0, int64_t S0, const int32_t *ids1, int64_t S1,
                               const RopePairs &pp, TableFormat fmt, float *cos_out,
                               float *sin_out, uint32_t *packed, cudaStream_t stream,
                               int *clear = nullptr);

// Workspace layout of flux_joint_rope_attention: a 256-byte status block,
// then the packed table [S, D/2] uint32, padded to 256 bytes.
constexpr size_t kStatusBytes = 256;
inline size_t packed_table_bytes(int64_t S, int D) {
  size_t b = static_cast<size_t>(S) * static_cast<size_t>(D / 2) * sizeof(uint32_t);
  return (b + 255) & ~static_cast<size_t>(255);
}

// Exchange buffer of the attention kernel for [B, S, H, D] inputs: one 8-byte
// flag per (batch, head, key tile, RoPE warp), padded to 256 bytes, then a
// [B, S, H, D] bf16 copy of K after RoPE, then one of Q after RoPE. 0 if D is
// not 128 or the shape is empty.
inline size_t krot_flag_bytes(int B, int64_t S, int H) {
  const size_t tiles = static_cast<size_t>((S + 127) / 128);
  size_t b = static_cast<size_t>(B) * static_cast<size_t>(H) * tiles * 4 * sizeof(uint64_t);
  return (b + 255) & ~static_cast<size_t>(255);
}
inline size_t krot_scratch_bytes(int B, int64_t S, int H, int D) {
  if (D != 128 || B < 1 || H < 1 || S < 1) return 0;
  return krot_flag_bytes(B, S, H) +
         2 * static_cast<size_t>(B) * static_cast<size_t>(S) * static_cast<size_t>(H) * 128 * 2;
}

// Optional QK RMS normalisation for launch_joint_attention: fp32 [128] device
// weight vectors for the queries and keys of text tokens (the first s_txt
// tokens) and of the other tokens, and eps.
struct QkNormArgs {
  const float *q_txt, *k_txt, *q_img, *k_img;
  int64_t s_txt;
  float eps;
};

// One segment of a launch: queries [q_lo, q_hi) (rows of Q / out) attend to
// keys [k_lo, k_hi) (rows of K / V). Segments with the same key_range
// (0 .. kMaxSegments-1) must have the same key range and share its
// exchange-buffer flags.
constexpr int kMaxSegments = 3;
struct AttnSegment {
  int64_t q_lo, q_hi, k_lo, k_hi;
  int key_range;
  int64_t n_pre;  // rows [0, n_pre) of the pre-rotated K / V join the key range
};

// Keys that arrive rotated already (a reference-image cache) and their
// values: bf16 [B, S, H, 128]; they skip RoPE.
struct PreRotatedKV {
  const void *k, *v;
  int64_t S;
};

// Bytes of the exchange buffer of launch_attention_segments: the flags of
// each key range, padded to 256 bytes, then bf16 [B, S_k, H, D] rotated K
// and [B, S_q, H, D] rotated Q.
size_t exchange_bytes(int B, int64_t S_q, int64_t S_k, int H, const AttnSegment *segs,
                      int n_segs);

// Enqueues the attention kernel over segments: Q / out [B, S_q, H, 128] and
// K / V [B, S_k, H, 128] bf16; table_q [S_q, 64] and table_k [S_k, 64]
// packed tables for the rows of Q and of K; xbuf (nullable) the exchange
// buffer of exchange_bytes(...) bytes, 256-byte aligned.
// pdl: launch with programmatic stream serialization, so that the kernel's
// prologue and first Q / K / V copies overlap the table kernel enqueued just
// before it on `stream` (which must be the previous kernel in the stream);
// everything that reads the table or the status word waits for it first.
// h0, Hl: attend only heads h0 .. h0 + Hl - 1 of the H heads of Q / K / V /
// out (Hl 0: all H heads); the exchange buffer is laid out for the Hl heads
// (exchange_bytes with H = Hl).
cudaError_t launch_attention_segments(const void *q, const void *k, const void *v, void *out,
                                      const uint32_t *table_q, const uint32_t *table_k,
                                      int *status, int B, int64_t S_q, int64_t S_k, int H,
                                      const AttnSegment *segs, int n_segs,
                                      const PreRotatedKV *pre, void *xbuf,
                                      const QkNormArgs *norm, cudaStream_t stream,
                                      bool pdl = false, int h0 = 0, int Hl = 0);

// The driver's cuTensorMapEncodeTiled for the projection's tensor maps,
// fetched once through the runtime (no -lcuda); NULL when unavailable.
void *tensor_map_encode_entry();

// Enqueues the fused single-stream input projection: x [M, dim] and W
// [3 * H * 128 + 2 * mlp, dim] bf16 row-major; q, k, v [M, H, 128] and act
// [M, mlp] bf16 written. dim a multiple of 64, mlp a multiple of 128.
cudaError_t launch_qkv_mlp_proj(const void *x, const void *w, int64_t M, int dim, int H,
                                int64_t mlp, void *q, void *k, void *v, void *act, int *status,
                                cudaStream_t stream);

// Enqueues the attention kernel. q/k/v/out are [B, S, H, 128] bf16; `table`
// is the packed table of the joint sequence; status is the device status word.
// `krot_scratch` (256-byte aligned, krot_scratch_bytes long) lets the CTAs
// that work on one head share rotated K tiles; NULL makes every CTA rotate
// every K tile it loads. `norm` (nullable) normalises Q and K before RoPE.
cudaError_t launch_joint_attention(const void *q, const void *k, const void *v, void *out,
                                   const uint32_t *table, int *status, int B, int64_t S, int H,
                                   void *krot_scratch, const QkNormArgs *norm,
                                   cudaStream_t stream, bool pdl = false, int h0 = 0,
                                   int Hl = 0);

}  // namespace flux
