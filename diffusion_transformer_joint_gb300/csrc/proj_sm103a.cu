// Fused input projection of the FLUX.2 single-stream block for sm_103a
// (GB300): one bf16 GEMM on tcgen05 whose epilogue writes Q, K and V in the
// attention's [B, S, H, 128] layout and the SwiGLU activation of the MLP half.
//
// Definition ("Diffusers 中 Flux2Transformer2DModel 全面解析", section
// 内部架构双流块与单流块: the single-stream block fuses the Q, K, V projections
// and the MLP input projection into one linear layer, to_qkv_mlp_proj, of
// 3 * inner + 2 * mlp output features; section 激活函数与 FFN: the SwiGLU gate
// projection is fused into that layer and the activation halves the width;
// section 并行化支持: the packed MLP features are two equal halves, gate then
// linear):
//   y = x W^T, x [M, dim] (M = B * S tokens), W [3 * inner + 2 * mlp, dim]
//   q = y[:, 0:inner], k = y[:, inner:2 inner], v = y[:, 2 inner:3 inner]
//   act = silu(y[:, 3 inner:3 inner + mlp]) * y[:, 3 inner + mlp:]
// with inner = H * 128; q, k, v are stored as [M, H, 128] (= [B, S, H, 128]).
//
// Tiles: 128 token rows x two 128-feature units, 64 channels per pipeline
// stage (one 128-byte swizzle row of bf16). A Q/K/V tile takes two
// consecutive units of the first 3 * inner features (a unit is one head of
// Q, K or V); an MLP tile takes gate unit j and linear unit j, so that the
// epilogue holds both factors of every activation it writes. The B operand
// of a tile is the two units' W rows, copied by TMA as two 128-row boxes into
// one 256-row K-major operand. Every tile is one M128 N256 accumulation over
// all of dim.
//
// Persistent: one CTA per SM walks the tiles round robin, the 128-row blocks
// of one feature tile consecutively, so the CTAs running at the same time
// share a few W slabs and all of x in L2. 8 warps:
//   warp 0: TMA producer (4-stage ring of 48 KB stages);
//   warp 1: MMA issuer (whole warp, elect.sync issues), M128 N256 K16 steps;
//   warp 2: TMEM allocation (two 256-column accumulators);
//   warps 4-7: epilogue, one TMEM lane (token row) per thread: fp32 -> bf16
//   (round to nearest even), SiLU * linear for MLP tiles, 16-byte stores.
// The two accumulators let the epilogue of one tile overlap the next tile's
// MMAs. Every wait is bounded; a wait that runs out aborts the CTA and sets
// the status word to FLUX_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "flux_attn.h"
#include "flux_internal.h"
#include "ptx_sm103a.cuh"

namespace flux {
namespace {

constexpr int kPM = 128;          // token rows per tile
constexpr int kUnit = 128;        // output features per half tile
constexpr int kPN = 2 * kUnit;    // accumulator columns per tile
constexpr int kPK = 64;           // channels per stage
constexpr int kPStages = 4;
constexpr uint32_t kPABytes = kPM * kPK * 2;  // 16 KB
constexpr uint32_t kPBBytes = kPN * kPK * 2;  // 32 KB
constexpr uint32_t kPStageBytes = kPABytes + kPBBytes;
constexpr int kPThreads = 256;
constexpr uint32_t kPTmemCols = 2 * kPN;
constexpr int kBarFull = 0;
constexpr int kBarEmpty = kPStages;
constexpr int kBarAccFull = 2 * kPStages;
constexpr int kBarAccEmpty = 2 * kPStages + 2;
constexpr int kBarDrainP = 2 * kPStages + 4;
constexpr int kPNumBars = 2 * kPStages + 5;
constexpr uint32_t kPOffBar = kPStages * kPStageBytes;
constexpr uint32_t kPOffTmemSlot = kPOffBar + 8 * kPNumBars;
constexpr uint32_t kPOffAbort = kPOffTmemSlot + 8;
constexpr uint32_t kPSmemBytes = kPOffAbort + 8 + 1024;  // + slack for 1024-byte alignment
static_assert(kPSmemBytes <= 232448, "shared memory per CTA");

// The problem: x [M, dim], W [3 * inner + 2 * mlp, dim]; tiles are numbered
// feature tile major, 128-row block minor.
struct ProjShape {
  int64_t M, mlp;
  int dim, H, n_mb, n_qkv_tiles, n_tiles;
};

struct ProjMaps {
  CUtensorMap x, w;
};

__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitBudgetCycles) {
  }
}

// silu(g) * u in fp32: g / (1 + e^-g) * u.
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.f + __expf(-g)) * u; }

__global__ void __launch_bounds__(kPThreads, 1)
    qkv_mlp_proj_kernel(const __grid_constant__ ProjMaps maps, const ProjShape p,
                        uint16_t *__restrict__ qo, uint16_t *__restrict__ ko,
                        uint16_t *__restrict__ vo, uint16_t *__restrict__ act,
                        int *__restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(base);
  auto bar = [&](int i) { return sbase + kPOffBar + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kPOffTmemSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kPOffAbort);
  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t inner = static_cast<int64_t>(p.H) * kUnit;
  const int nk = p.dim / kPK;
  const int n_units = 3 * p.H;

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarAccFull + b), 1);
      mbar_init(bar(kBarAccEmpty + b), 4);
    }
    mbar_init(bar(kBarDrainP), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.w);
    int it = 0;  // stages filled so far
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.n_tiles; t += gridDim.x) {
      const int mb = t % p.n_mb, nt = t / p.n_mb;
      const int m0 = mb * kPM;
      int r0, r1;  // first W rows of the two units
      if (nt < p.n_qkv_tiles) {
        r0 = 2 * nt * kUnit;
        r1 = 2 * nt + 1 < n_units ? r0 + kUnit : r0;  // a missing second unit is not stored
      } else {
        const int64_t j = nt - p.n_qkv_tiles;
        r0 = static_cast<int>(3 * inner + j * kUnit);
        r1 = static_cast<int>(3 * inner + p.mlp + j * kUnit);
      }
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % kPStages;
        const uint32_t use = static_cast<uint32_t>(it / kPStages);
        if (!(ok = mbar_wait(bar(kBarEmpty + s), (use & 1u) ^ 1u, abort_flag))) break;
        const uint32_t dst = sbase + s * kPStageBytes;
        mbar_arrive_expect_tx(bar(kBarFull + s), kPStageBytes);
        tma_load_2d(dst, &maps.x, bar(kBarFull + s), ks * kPK, m0);
        tma_load_2d(dst + kPABytes, &maps.w, bar(kBarFull + s), ks * kPK, r0);
        tma_load_2d(dst + kPABytes + kPBBytes / 2, &maps.w, bar(kBarFull + s), ks * kPK, r1);
      }
    }
    // every copy issued above has landed before the CTA exits
    for (int j = (it > kPStages ? it - kPStages : 0); j < it; ++j)
      drain(bar(kBarFull + j % kPStages), static_cast<uint32_t>(j / kPStages) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kPM, kPN, 0, 0);
    int it = 0;
    int lt = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.n_tiles; t += gridDim.x, ++lt) {
      const int buf = lt & 1;
      if (!(ok = wait_warp(bar(kBarAccEmpty + buf), ((static_cast<uint32_t>(lt) >> 1) & 1u) ^ 1u,
                           abort_flag)))
        break;
      tc_fence_after_sync();
      const uint32_t d = tmem + static_cast<uint32_t>(buf * kPN);
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % kPStages;
        if (!(ok = wait_warp(bar(kBarFull + s), static_cast<uint32_t>(it / kPStages) & 1u,
                             abort_flag)))
          break;
        tc_fence_after_sync();
        const uint64_t da = sdesc_sw128(sbase + s * kPStageBytes, 16, 1024);
        const uint64_t db = sdesc_sw128(sbase + s * kPStageBytes + kPABytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kPK / 16; ++kk)
          mma_ss_elect(d, desc_advance(da, kk * 32), desc_advance(db, kk * 32), idesc,
                       (ks | kk) != 0 ? 1u : 0u);
        mma_commit_elect(bar(kBarEmpty + s));  // the stage may be refilled
      }
      if (!ok) break;
      mma_commit_elect(bar(kBarAccFull + buf));  // the accumulator is complete
    }
    // every MMA issued above has finished before TMEM is released
    mma_commit_elect(bar(kBarDrainP));
    const long long t0 = clock64();
    while (!mbar_try_wait(bar(kBarDrainP), 0) && clock64() - t0 < kWaitBudgetCycles) {
    }
    __syncwarp();
  } else if (warp >= 4) {
    // -------------------------------------------------------------- epilogue
    const int wq = warp & 3;  // TMEM lane quadrant
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    int lt = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.n_tiles; t += gridDim.x, ++lt) {
      const int mb = t % p.n_mb, nt = t / p.n_mb;
      const int buf = lt & 1;
      if (!(ok = wait_warp(bar(kBarAccFull + buf), (static_cast<uint32_t>(lt) >> 1) & 1u,
                           abort_flag)))
        break;
      tc_fence_after_sync();
      const uint32_t tacc = tmem + static_cast<uint32_t>(buf * kPN) + lane_off;
      const int64_t row = static_cast<int64_t>(mb) * kPM + wq * 32 + lane;
      const bool live = row < p.M;
      if (nt < p.n_qkv_tiles) {
        for (int h = 0; h < 2; ++h) {
          const int u = 2 * nt + h;
          if (u >= n_units) break;
          uint16_t *dst = (u < p.H ? qo : u < 2 * p.H ? ko : vo) + row * inner +
                          static_cast<int64_t>(u % p.H) * kUnit;
#pragma unroll 1
          for (int c = 0; c < kUnit / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tacc + h * kUnit + c * 32, r);
            tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint4 w4;
                w4.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1]));
                w4.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3]));
                w4.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5]));
                w4.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7]));
                st_global_v4(dst + c * 32 + 8 * i, w4);
              }
            }
          }
        }
      } else {
        const int64_t j = nt - p.n_qkv_tiles;
        uint16_t *dst = act + row * p.mlp + j * kUnit;
#pragma unroll 1
        for (int c = 0; c < kUnit / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tacc + c * 32, g);
          tmem_ld32(tacc + kUnit + c * 32, u);
          tmem_ld_wait();
          if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float a[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                a[e] = swiglu(__uint_as_float(g[8 * i + e]), __uint_as_float(u[8 * i + e]));
              uint4 w4;
              w4.x = pack_bf16x2(a[0], a[1]);
              w4.y = pack_bf16x2(a[2], a[3]);
              w4.z = pack_bf16x2(a[4], a[5]);
              w4.w = pack_bf16x2(a[6], a[7]);
              st_global_v4(dst + c * 32 + 8 * i, w4);
            }
          }
        }
      }
      // this warp's TMEM reads are complete: the accumulator may be reused
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarAccEmpty + buf));
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kPTmemCols);
  }
  if (tid == 0 && *abort_flag) atomicExch(status, FLUX_ERR_DEVICE_TIMEOUT);
}

// A row-major bf16 matrix [rows, cols] as a 2-D tensor map; one box = 64
// columns (128 bytes, 128-byte swizzle) x 128 rows; rows past the end read
// as zeros.
bool make_rows_map(CUtensorMap *map, const void *x, int64_t rows, int64_t cols) {
  auto fn = reinterpret_cast<CUresult (*)(
      CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill)>(
      tensor_map_encode_entry());
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kPK), static_cast<cuuint32_t>(kPM)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
void *tensor_map_encode_entry() {
  static void *fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
  });
  return fn;
}

cudaError_t launch_qkv_mlp_proj(const void *x, const void *w, int64_t M, int dim, int H,
                                int64_t mlp, void *q, void *k, void *v, void *act, int *status,
                                cudaStream_t stream) {
  if (M < 1 || dim < kPK || dim % kPK != 0 || H < 1 || mlp < 0 || mlp % kUnit != 0)
    return cudaErrorInvalidValue;
  const int64_t inner = static_cast<int64_t>(H) * kUnit;
  const int64_t n_out = 3 * inner + 2 * mlp;
  const int64_t n_mb = (M + kPM - 1) / kPM;
  const int64_t n_qkv = (3 * static_cast<int64_t>(H) + 1) / 2;
  const int64_t n_tiles = n_mb * (n_qkv + mlp / kUnit);
  if (n_out > 0x7FFFFFFFLL || n_tiles > 0x7FFFFFFFLL || M > 0x7FFFFFFFLL)
    return cudaErrorInvalidValue;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev], [&] {
    attr_err = cudaFuncSetAttribute(qkv_mlp_proj_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kPSmemBytes));
  });
  if (attr_err != cudaSuccess) return attr_err;
  ProjMaps maps;
  if (!make_rows_map(&maps.x, x, M, dim) || !make_rows_map(&maps.w, w, n_out, dim))
    return cudaErrorInvalidValue;
  static int sm_count[64];
  if (sm_count[dev] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sm_count[dev] = n;
  }
  ProjShape p;
  p.M = M;
  p.mlp = mlp;
  p.dim = dim;
  p.H = H;
  p.n_mb = static_cast<int>(n_mb);
  p.n_qkv_tiles = static_cast<int>(n_qkv);
  p.n_tiles = static_cast<int>(n_tiles);
  const unsigned grid =
      static_cast<unsigned>(n_tiles < sm_count[dev] ? n_tiles : sm_count[dev]);
  qkv_mlp_proj_kernel<<<grid, kPThreads, kPSmemBytes, stream>>>(
      maps, p, static_cast<uint16_t *>(q), static_cast<uint16_t *>(k),
      static_cast<uint16_t *>(v), static_cast<uint16_t *>(act), status);
  return cudaGetLastError();
}

}  // namespace flux
