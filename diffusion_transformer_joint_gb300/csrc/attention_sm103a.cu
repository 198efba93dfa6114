// Joint RoPE attention forward for sm_103a (GB300): tcgen05 MMAs with TMEM
// accumulators, RoPE applied to Q and K while their tiles are staged into
// shared memory.
//
// Definition ("Transformer架构解析FLUX.2-klein-base-9b-nvfp4", section 2:
// scaled dot-product attention; "Diffusers 中 Flux2Transformer2DModel 全面解析",
// section 内部架构双流块与单流块: text and image tokens form one sequence):
//   out[b, i, h, :] = sum_j softmax_j(q^_i . k^_j / sqrt(128)) v[b, j, h, :]
// with q^, k^ the RoPE-rotated rows; non-causal over all S tokens.
//
// One CTA owns 128 query rows of one (batch, head). Per 128-key tile:
//   1. all threads load K (rotating each adjacent channel pair with the
//      token's cos/sin) and V into 128-byte-swizzled shared memory;
//   2. one thread issues S = Q^ K^T as eight 128x128x16 tcgen05 MMAs into TMEM;
//   3. each thread owns one query row (TMEM lane): it reads its 128 scores,
//      runs the online softmax in the log2 domain, writes P as packed bf16
//      and rescales its row of the running output O in TMEM;
//   4. one thread issues O += P V (eight MMAs, V as an MN-major operand).
// The epilogue divides O by the softmax denominator and stores bf16.
#include <cuda_bf16.h>

#include <cmath>

#include "flux_internal.h"
#include "ptx_sm103a.cuh"

namespace flux {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 128;
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // 128 rows x 128 bf16
constexpr uint32_t kBlockBytes = 16384;         // one 64-column swizzle block

#ifdef FLUX_P_VIA_SMEM
constexpr bool kPInTmem = false;
#else
constexpr bool kPInTmem = true;
#endif

constexpr uint32_t kNumTiles = kPInTmem ? 3 : 4;  // Q, K, V (+ P)
constexpr uint32_t kCtrlOffset = kNumTiles * kTileBytes;
constexpr uint32_t kSmemBytes = kCtrlOffset + 64 + 1024;  // + control block + alignment slack
constexpr uint32_t kTmemCols = 256;                        // S: 0..127, O: 128..255

// Byte offset of 16-byte chunk c16 (0..15) of row r in a [128 x 128] bf16
// tile stored as two 64-column blocks, each rows of 128 bytes with the
// 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c16) {
  return static_cast<uint32_t>((c16 >> 3) * kBlockBytes + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}

// K-major operand (rows = M or N, 128 channels = K): slice kk covers
// channels [16 kk, 16 kk + 16).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  return sdesc_sw128(tile + (kk >> 2) * kBlockBytes + (kk & 3) * 32, 16, 1024);
}

// V as the MN-major B operand of P V: rows = keys (K), columns = channels
// (N). Slice kk covers keys [16 kk, 16 kk + 16); the two 64-channel blocks
// are kBlockBytes apart.
__device__ __forceinline__ uint64_t desc_v(uint32_t tile, int kk) {
  return sdesc_sw128(tile + kk * 2048, kBlockBytes, 1024);
}

// Rotate the two bf16 channels packed in `w` by (c, s) and round back.
__device__ __forceinline__ uint32_t rope_pair(uint32_t w, float c, float s) {
  const float x0 = bf16lo_to_f32(w), x1 = bf16hi_to_f32(w);
  return pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
}

// Stage a [128 tokens x 128 channels] tile of one head into swizzled smem,
// rotating it with the tokens' table rows when kRotate. Rows at or past
// `rows_valid` are written as zeros.
template <bool kRotate>
__device__ __forceinline__ void stage_tile(uint32_t sdst, const uint16_t *g, int64_t row_stride,
                                           int rows_valid, const float *cos_t,
                                           const float *sin_t) {
#pragma unroll 4
  for (int i = 0; i < (kBM * 16) / kThreads; ++i) {
    const int x = i * kThreads + static_cast<int>(threadIdx.x);
    const int r = x >> 4, c16 = x & 15;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows_valid) {
      w = ld_global_nc_v4(g + r * row_stride + c16 * 8);
      if (kRotate) {
        const float4 c = ld_global_nc_f4(cos_t + r * (kD / 2) + c16 * 4);
        const float4 s = ld_global_nc_f4(sin_t + r * (kD / 2) + c16 * 4);
        w.x = rope_pair(w.x, c.x, s.x);
        w.y = rope_pair(w.y, c.y, s.y);
        w.z = rope_pair(w.z, c.z, s.z);
        w.w = rope_pair(w.w, c.w, s.w);
      }
    }
    st_shared_v4(sdst + sw128_offset(r, c16), w);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    joint_rope_attention_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                                const uint16_t *__restrict__ v, uint16_t *__restrict__ out,
                                const float *__restrict__ cos_t, const float *__restrict__ sin_t,
                                int *__restrict__ status, int64_t S, int H) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_addr(base);
  const uint32_t sK = sQ + kTileBytes;
  const uint32_t sV = sK + kTileBytes;
  const uint32_t sP = sV + kTileBytes;  // used only when P goes through smem
  uint64_t *bar_mma = reinterpret_cast<uint64_t *>(base + kCtrlOffset);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kCtrlOffset + 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kCtrlOffset + 12);

  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5;
  const int m0 = static_cast<int>(blockIdx.x) * kBM;
  const int h = static_cast<int>(blockIdx.y);
  const int b = static_cast<int>(blockIdx.z);
  const int64_t row_stride = static_cast<int64_t>(H) * kD;
  const int64_t head0 = (static_cast<int64_t>(b) * S * H + h) * kD;  // token 0 of (b, h)
  const uint16_t *qh = q + head0;
  const uint16_t *kh = k + head0;
  const uint16_t *vh = v + head0;

  if (tid == 0) {
    mbar_init(smem_addr(bar_mma), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }

  const int q_valid = static_cast<int>(S - m0 < kBM ? S - m0 : kBM);
  stage_tile<true>(sQ, qh + m0 * row_stride, row_stride, q_valid, cos_t + m0 * (kD / 2),
                   sin_t + m0 * (kD / 2));
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;        // scores, later P (packed bf16 in columns 0..63)
  const uint32_t tO = tmem + 128;  // running output
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
  const uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);
  const uint32_t bar = smem_addr(bar_mma);
  // softmax in the log2 domain: x = s * log2(e) / sqrt(128)
  const float scale_log2 = 1.4426950408889634f * 0.08838834764831845f;

  float m_run = -INFINITY, l_run = 0.f;
  uint32_t phase = 0;
  const int n_tiles = static_cast<int>((S + kBN - 1) / kBN);

  for (int jt = 0; jt < n_tiles; ++jt) {
    const int n0 = jt * kBN;
    const int kv_valid = static_cast<int>(S - n0 < kBN ? S - n0 : kBN);
    // The previous P V has completed (waited below), so K/V/P are free.
    stage_tile<true>(sK, kh + n0 * row_stride, row_stride, kv_valid, cos_t + n0 * (kD / 2),
                     sin_t + n0 * (kD / 2));
    stage_tile<false>(sV, vh + n0 * row_stride, row_stride, kv_valid, nullptr, nullptr);
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk)
        mma_ss(tS, desc_kmajor(sQ, kk), desc_kmajor(sK, kk), idesc_qk, kk > 0 ? 1u : 0u);
      mma_commit(bar);
    }
    mbar_wait(bar, phase, abort_flag);
    phase ^= 1u;
    __syncthreads();
    if (*abort_flag) break;
    tc_fence_after_sync();

    // ---- online softmax on this thread's row
    uint32_t sr[kBN];
#pragma unroll
    for (int c = 0; c < kBN / 32; ++c)
      tmem_ld32(tS + lane_off + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
    tmem_ld_wait();
    float mx = m_run;
#pragma unroll
    for (int j = 0; j < kBN; ++j) {
      const float x = (j < kv_valid) ? __uint_as_float(sr[j]) * scale_log2 : -INFINITY;
      sr[j] = __float_as_uint(x);
      mx = fmaxf(mx, x);
    }
    const float alpha = ex2_approx(m_run - mx);  // 0 on the first tile
    float sum = 0.f;
    uint32_t pk[kBN / 2];
#pragma unroll
    for (int j = 0; j < kBN; j += 2) {
      const float p0 = ex2_approx(__uint_as_float(sr[j]) - mx);
      const float p1 = ex2_approx(__uint_as_float(sr[j + 1]) - mx);
      sum += p0 + p1;
      pk[j / 2] = pack_bf16x2(p0, p1);
    }
    l_run = l_run * alpha + sum;
    m_run = mx;

    if (kPInTmem) {
      tmem_st32(tS + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
    } else {
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16)
        st_shared_v4(sP + sw128_offset(tid, c16),
                     make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]));
    }
    if (jt > 0) {
#pragma unroll
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
        tmem_st32(tO + lane_off + c * 32, o);
      }
    }
    tmem_st_wait();
    if (!kPInTmem) fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint32_t acc = (jt > 0 || kk > 0) ? 1u : 0u;
        if (kPInTmem)
          mma_ts(tO, tS + kk * 8, desc_v(sV, kk), idesc_pv, acc);
        else
          mma_ss(tO, desc_kmajor(sP, kk), desc_v(sV, kk), idesc_pv, acc);
      }
      mma_commit(bar);
    }
    mbar_wait(bar, phase, abort_flag);
    phase ^= 1u;
    __syncthreads();
    if (*abort_flag) break;
    tc_fence_after_sync();
  }

  if (!*abort_flag) {
    const float inv_l = 1.f / l_run;
    const int r = tid;
    uint16_t *orow = out + head0 + static_cast<int64_t>(m0 + r) * row_stride;
#pragma unroll
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + lane_off + c * 32, o);
      tmem_ld_wait();
      if (r < q_valid) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[j]) * inv_l, __uint_as_float(o[j + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o[j + 2]) * inv_l, __uint_as_float(o[j + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o[j + 4]) * inv_l, __uint_as_float(o[j + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o[j + 6]) * inv_l, __uint_as_float(o[j + 7]) * inv_l);
          *reinterpret_cast<uint4 *>(orow + c * 32 + j) = w;
        }
      }
    }
  } else if (tid == 0) {
    atomicExch(status, FLUX_ERR_DEVICE_TIMEOUT);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_joint_attention(const void *q, const void *k, const void *v, void *out,
                                   const float *cos_t, const float *sin_t, int *status, int B,
                                   int64_t S, int H, cudaStream_t stream) {
  static bool attr_done = false;  // per process; the attribute is per function
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(joint_rope_attention_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const dim3 grid(static_cast<unsigned>((S + kBM - 1) / kBM), static_cast<unsigned>(H),
                  static_cast<unsigned>(B));
  joint_rope_attention_kernel<<<grid, kThreads, kSmemBytes, stream>>>(
      static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
      static_cast<const uint16_t *>(v), static_cast<uint16_t *>(out), cos_t, sin_t, status, S, H);
  return cudaGetLastError();
}

}  // namespace flux
