// N-D RoPE cos/sin tables (EmbedND / Flux2PosEmbed).
//
// Each axis gets its own 1-D rotary embedding over its share of the head
// width and the axes are concatenated ("Diffusers 中 Flux2Transformer2DModel
// 全面解析", section 前向传播输入输出约定; "FLUX.2 [klein]" survey page,
// section 模型架构: axes (32, 32, 32, 32), theta 2000). Pair j of an axis of
// width d_a turns by id * theta^(-2j/d_a).
//
// The per-pair frequency is formed on the host in extended precision as a
// 0.64 fixed-point fraction of a turn, F = round(2^64 theta^(-2j/d_a) / (2 pi)).
// Per table entry the kernel multiplies it by the position id in 64-bit
// integer arithmetic: id * F mod 2^64 is the angle's fractional turn, exact
// up to the rounding of F (|id| * 2^-64 turns), for any int32 id; its top 32
// bits, read as a signed number, are the angle in [-1/2, 1/2) turns. Sine and
// cosine of that angle are evaluated in fp32 with sincospif. No fp64 work is
// left in the kernel (fp64 is slow on this part).
//
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>

#include "flux_internal.h"
#include "ptx_sm103a.cuh"

namespace flux {
namespace {

// One block row of threads per token: threadIdx.x walks the pairs,
// threadIdx.y the tokens of the block; the grid strides over tokens. The
// per-pair parameters are staged in shared memory once per block: read from
// the parameter space with a different pair per lane, every access would be
// serialised across the warp.
template <TableFormat kFmt>
__global__ void __launch_bounds__(256) rope_tables_kernel(const int32_t *__restrict__ ids0,
                                                          int64_t S0,
                                                          const int32_t *__restrict__ ids1,
                                                          int64_t S, const RopePairs pp,
                                                          float *__restrict__ cos_out,
                                                          float *__restrict__ sin_out,
                                                          uint32_t *__restrict__ packed,
                                                          int *__restrict__ clear) {
  // the attention kernel after this one may begin launching (it waits for
  // this grid before it reads the table or the cleared word)
  grid_dep_launch_dependents();
  if (clear != nullptr && blockIdx.x == 0 && threadIdx.x == 0 && threadIdx.y == 0) *clear = 0;
  __shared__ uint64_t turns_q64[kMaxPairs];
  __shared__ uint8_t axis[kMaxPairs];
  const int P = pp.n_pairs;
  for (int p = threadIdx.y * blockDim.x + threadIdx.x; p < P; p += blockDim.x * blockDim.y) {
    turns_q64[p] = pp.turns_q64[p];
    axis[p] = pp.axis[p];
  }
  __syncthreads();
  for (int64_t s = static_cast<int64_t>(blockIdx.x) * blockDim.y + threadIdx.y; s < S;
       s += static_cast<int64_t>(gridDim.x) * blockDim.y) {
    const int32_t *row = (s < S0) ? ids0 + s * pp.n_axes : ids1 + (s - S0) * pp.n_axes;
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
      const uint64_t prod =
          static_cast<uint64_t>(static_cast<int64_t>(row[axis[p]])) * turns_q64[p];
      const int32_t turn_q32 = static_cast<int32_t>(prod >> 32);  // [-1/2, 1/2) turns, Q0.32
      const float two_f = static_cast<float>(turn_q32) * 4.656612873077393e-10f;  // 2^-31
      float sn, cs;
      sincospif(two_f, &sn, &cs);
      const int64_t e = s * P + p;
      if constexpr (kFmt == TableFormat::kF32Pair) {
        cos_out[e] = cs;
        sin_out[e] = sn;
      } else {
        packed[e] = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(cs))) |
                    (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(sn))) << 16);
      }
    }
  }
}

}  // namespace

int sm_count_current_device() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int make_rope_pairs(const int32_t *axes_dims, int n_axes, double theta, RopePairs *pp) {
  if (axes_dims == nullptr) return FLUX_ERR_NULL;
  if (n_axes < 1 || n_axes > FLUX_MAX_AXES || !(theta > 0.0) || !std::isfinite(theta))
    return FLUX_ERR_AXES;
  int p = 0;
  const long double two_pi = 6.283185307179586476925286766559L;
  const long double two_64 = 18446744073709551616.0L;
  for (int a = 0; a < n_axes; ++a) {
    const int d = axes_dims[a];
    if (d <= 0 || (d & 1) || p + d / 2 > kMaxPairs) return FLUX_ERR_AXES;
    for (int j = 0; j < d / 2; ++j, ++p) {
      pp->axis[p] = static_cast<uint8_t>(a);
      const long double turns =
          std::pow(static_cast<long double>(theta),
                   -2.0L * static_cast<long double>(j) / static_cast<long double>(d)) /
          two_pi;
      // turns <= 1 / (2 pi) < 1, so the scaled value fits in 64 bits
      pp->turns_q64[p] = static_cast<uint64_t>(turns * two_64 + 0.5L);
    }
  }
  pp->n_pairs = p;
  pp->n_axes = n_axes;
  return FLUX_OK;
}

cudaError_t launch_rope_tables(const int32_t *ids0, int64_t S0, const int32_t *ids1, int64_t S1,
                               const RopePairs &pp, TableFormat fmt, float *cos_out,
                               float *sin_out, uint32_t *packed, cudaStream_t stream,
                               int *clear) {
  const int64_t S = S0 + S1;
  const dim3 block(64, 4);
  int64_t blocks = (S + block.y - 1) / block.y;
  const int sms = sm_count_current_device();
  if (sms == 0) return cudaErrorUnknown;
  if (blocks > 8 * sms) blocks = 8 * sms;
  if (blocks < 1) blocks = 1;
  if (fmt == TableFormat::kF32Pair)
    rope_tables_kernel<TableFormat::kF32Pair><<<static_cast<unsigned>(blocks), block, 0, stream>>>(
        ids0, S0, ids1, S, pp, cos_out, sin_out, packed, clear);
  else
    rope_tables_kernel<TableFormat::kPackedF16><<<static_cast<unsigned>(blocks), block, 0, stream>>>(
        ids0, S0, ids1, S, pp, cos_out, sin_out, packed, clear);
  return cudaGetLastError();
}

}  // namespace flux
