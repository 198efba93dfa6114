// N-D RoPE cos/sin tables (EmbedND / Flux2PosEmbed).
//
// Each axis gets its own 1-D rotary embedding over its share of the head
// width and the axes are concatenated ("Diffusers 中 Flux2Transformer2DModel
// 全面解析", section 前向传播输入输出约定; "FLUX.2 [klein]" survey page,
// section 模型架构: axes (32, 32, 32, 32), theta 2000). Pair j of an axis of
// width d_a turns by id * theta^(-2j/d_a).
//
// The frequencies are formed once per block in double precision. Per table
// entry the angle id * omega is a double product, reduced by a two-constant
// Cody-Waite step (Cody & Waite, "Software Manual for the Elementary
// Functions", 1980) to r in [-pi, pi]; cosine and sine are then taken in
// fp32 on r. This keeps the kernel off the slow fp64 transcendental path.
//
// Two output formats: separate fp32 cos and sin arrays (the public table
// call), or one 32-bit word per (token, pair) holding fp16 cos and sin, the
// format the attention kernel stages by TMA next to each K tile (half the
// bytes; fp16 keeps |error| <= 2^-12, below the bf16 rounding of the rotated
// channels it multiplies).
#include <cuda_fp16.h>

#include <cmath>

#include "flux_internal.h"

namespace flux {
namespace {

// 2*pi split as hi + lo, hi the double nearest 2*pi, lo the remainder.
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

template <TableFormat kFmt>
__global__ void __launch_bounds__(256) rope_tables_kernel(const int32_t *__restrict__ ids0,
                                                          int64_t S0,
                                                          const int32_t *__restrict__ ids1,
                                                          int64_t S, const RopePairs pp,
                                                          float *__restrict__ cos_out,
                                                          float *__restrict__ sin_out,
                                                          uint32_t *__restrict__ packed) {
  __shared__ double omega[kMaxPairs];
  const int P = pp.n_pairs;
  for (int p = threadIdx.x; p < P; p += blockDim.x)
    omega[p] = pow(pp.theta, -2.0 * static_cast<double>(pp.j[p]) / static_cast<double>(pp.d_axis[p]));
  __syncthreads();
  const int64_t total = S * P;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t s = e / P;
    const int p = static_cast<int>(e - s * P);
    const int a = pp.axis[p];
    const int32_t id = (s < S0) ? ids0[s * pp.n_axes + a] : ids1[(s - S0) * pp.n_axes + a];
    const double ang = static_cast<double>(id) * omega[p];
    const double kq = rint(ang * kInvTwoPi);
    double r = fma(-kq, kTwoPiHi, ang);
    r = fma(-kq, kTwoPiLo, r);
    float sn, cs;
    sincosf(static_cast<float>(r), &sn, &cs);
    if constexpr (kFmt == TableFormat::kF32Pair) {
      cos_out[e] = cs;
      sin_out[e] = sn;
    } else {
      packed[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(cs))) |
                  (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(sn))) << 16);
    }
  }
}

}  // namespace

int make_rope_pairs(const int32_t *axes_dims, int n_axes, double theta, RopePairs *pp) {
  if (axes_dims == nullptr) return FLUX_ERR_NULL;
  if (n_axes < 1 || n_axes > FLUX_MAX_AXES || !(theta > 0.0) || !std::isfinite(theta))
    return FLUX_ERR_AXES;
  int p = 0;
  for (int a = 0; a < n_axes; ++a) {
    const int d = axes_dims[a];
    if (d <= 0 || (d & 1) || p + d / 2 > kMaxPairs) return FLUX_ERR_AXES;
    for (int j = 0; j < d / 2; ++j, ++p) {
      pp->axis[p] = static_cast<uint8_t>(a);
      pp->j[p] = static_cast<uint8_t>(j);
      pp->d_axis[p] = static_cast<uint16_t>(d);
    }
  }
  pp->n_pairs = p;
  pp->n_axes = n_axes;
  pp->theta = theta;
  return FLUX_OK;
}

cudaError_t launch_rope_tables(const int32_t *ids0, int64_t S0, const int32_t *ids1, int64_t S1,
                               const RopePairs &pp, TableFormat fmt, float *cos_out,
                               float *sin_out, uint32_t *packed, cudaStream_t stream) {
  const int64_t S = S0 + S1;
  const int64_t total = S * pp.n_pairs;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4 * 152) blocks = 4 * 152;
  if (blocks < 1) blocks = 1;
  if (fmt == TableFormat::kF32Pair)
    rope_tables_kernel<TableFormat::kF32Pair><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        ids0, S0, ids1, S, pp, cos_out, sin_out, packed);
  else
    rope_tables_kernel<TableFormat::kPackedF16><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        ids0, S0, ids1, S, pp, cos_out, sin_out, packed);
  return cudaGetLastError();
}

}  // namespace flux
