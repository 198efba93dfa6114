// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "flux_attn.h"

namespace flux {

// Largest rotation-pair count of one head (head width 512).
constexpr int kMaxPairs = 256;

// Per-pair RoPE parameters handed to the table kernel by value: the axis a
// pair belongs to, its index j inside the axis and the axis width d_a.
struct RopePairs {
  int n_pairs;
  int n_axes;
  double theta;
  uint8_t axis[kMaxPairs];
  uint8_t j[kMaxPairs];
  uint16_t d_axis[kMaxPairs];
};

// Fills `pp` from host axes_dims; returns FLUX_OK or FLUX_ERR_AXES.
int make_rope_pairs(const int32_t *axes_dims, int n_axes, double theta, RopePairs *pp);

// Enqueues the table kernel over the joint id sequence [seg0 ; seg1].
cudaError_t launch_rope_tables(const int32_t *ids0, int64_t S0, const int32_t *ids1, int64_t S1,
                               const RopePairs &pp, float *cos_out, float *sin_out,
                               cudaStream_t stream);

// Workspace layout of flux_joint_rope_attention: a 256-byte status block,
// then cos [S, D/2] and sin [S, D/2] fp32, each padded to 256 bytes.
constexpr size_t kStatusBytes = 256;
inline size_t table_bytes(int64_t S, int D) {
  size_t b = static_cast<size_t>(S) * static_cast<size_t>(D / 2) * sizeof(float);
  return (b + 255) & ~static_cast<size_t>(255);
}

// Enqueues the attention kernel. q/k/v/out are [B, S, H, 128] bf16; cos/sin
// are the tables of the joint sequence; status is the device status word.
cudaError_t launch_joint_attention(const void *q, const void *k, const void *v, void *out,
                                   const float *cos_t, const float *sin_t, int *status, int B,
                                   int64_t S, int H, cudaStream_t stream);

}  // namespace flux
