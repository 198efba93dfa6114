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
// Tiles: 256 token rows x two 128-feature units, 64 channels per pipeline
// stage (one 128-byte swizzle row of bf16). A Q/K/V tile takes two
// consecutive units of the first 3 * inner features (a unit is one head of
// Q, K or V); an MLP tile takes gate unit j and linear unit j, so that the
// epilogue holds both factors of every activation it writes.
//
// CTA pairs (clusters of two, one CTA per SM): the pair computes a tile with
// one M256 N256 K16 MMA per 16 channels, issued by the even CTA and reading
// both CTAs' shared memory. Each CTA copies its own 128 x rows and one W
// unit (the even CTA the first, the odd CTA the second) into its own stages,
// so per SM a stage is 32 KB and the B operand each SM stores and reads is
// half of the tile's. Each CTA's TMEM receives its 128 rows of the tile.
// Both CTAs' copies of a stage complete on the even CTA's stage barrier.
// The MMA commits arrive on both CTAs' barriers (stage free, accumulator
// full), and the odd CTA's epilogue warps release an accumulator on the
// even CTA's barrier.
//
// Persistent: a pair walks tiles round robin, the 256-row blocks of one
// feature tile consecutively, so the pairs running at the same time share a
// few W slabs and all of x in L2. 8 warps per CTA:
//   warp 0: TMA producer (6-stage ring);
//   warp 1: MMA issuer in the even CTA (whole warp, elect.sync issues);
//   warp 2: TMEM allocation (two 256-column accumulators, pair-wide);
//   warps 4-7: epilogue, one TMEM lane (token row) per thread: fp32 -> bf16
//   (round to nearest even), SiLU * linear for MLP tiles; each warp stages
//   its 32 rows 64 features at a time in a 128-byte-swizzled 4 KB box (two
//   per warp, alternating) and lane 0 stores the box with one TMA copy
//   (rows past M are not written).
// The two accumulators let the epilogue of one tile overlap the next tile's
// MMAs. Every wait is bounded; a wait that runs out aborts the CTA and sets
// the status word to FLUX_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "flux_attn.h"
#include "flux_internal.h"
#include "ptx_sm103a.cuh"

namespace flux {
namespace {

constexpr int kPM = 128;          // token rows per CTA (256 per pair)
constexpr int kUnit = 128;        // output features per half tile
constexpr int kPN = 2 * kUnit;    // accumulator columns per tile
constexpr int kPK = 64;           // channels per stage
constexpr int kPStages = 6;
constexpr uint32_t kPABytes = kPM * kPK * 2;    // 16 KB: this CTA's x rows
constexpr uint32_t kPBBytes = kUnit * kPK * 2;  // 16 KB: this CTA's W unit
constexpr uint32_t kPStageBytes = kPABytes + kPBBytes;
constexpr int kPThreads = 256;
constexpr uint32_t kPTmemCols = 2 * kPN;
constexpr int kBarFull = 0;                   // (even CTA) both CTAs' copies landed
constexpr int kBarEmpty = kPStages;           // the pair's MMAs read the stage
constexpr int kBarAccFull = 2 * kPStages;
constexpr int kBarAccEmpty = 2 * kPStages + 2;  // (even CTA) both epilogues read it
constexpr int kBarDrainP = 2 * kPStages + 4;
constexpr int kPNumBars = 2 * kPStages + 5;
constexpr uint32_t kPBoxBytes = 32 * 128;  // output box: 32 rows x 64 bf16 (128-byte swizzle)
constexpr uint32_t kPOffStage = kPStages * kPStageBytes;  // 2 output boxes per epilogue warp
constexpr uint32_t kPOffBar = kPOffStage + 4 * 2 * kPBoxBytes;
constexpr uint32_t kPOffTmemSlot = kPOffBar + 8 * kPNumBars;
constexpr uint32_t kPOffAbort = kPOffTmemSlot + 8;
constexpr uint32_t kPSmemBytes = kPOffAbort + 8 + 1024;  // + slack for 1024-byte alignment
static_assert(kPSmemBytes <= 232448, "shared memory per CTA");
constexpr uint16_t kPairMask = 0x3;

// The problem: x [M, dim], W [3 * inner + 2 * mlp, dim]; tiles are numbered
// feature tile major, 256-row block minor.
struct ProjShape {
  int64_t M, mlp;
  int dim, H, n_pb, n_qkv_tiles, n_tiles;
};

// x and W as copied in (64-channel x 128-row boxes); q, k, v and act as
// stored (64-feature x 32-row boxes).
struct ProjMaps {
  CUtensorMap x, w, q, k, v, act;
};

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
  const uint32_t crank = cluster_ctarank();  // 0: issues the MMAs
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarAccFull + b), 1);
      mbar_init(bar(kBarAccEmpty + b), 8);  // four epilogue warps of each CTA
    }
    mbar_init(bar(kBarDrainP), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_addr(tmem_slot), kPTmemCols);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- TMA producer
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.w);
    int it = 0;  // stages filled so far
    bool ok = true;
    for (int t = cid; ok && t < p.n_tiles; t += ncl) {
      const int nt = t / p.n_pb;
      const int m0 = (t % p.n_pb) * (2 * kPM) + static_cast<int>(crank) * kPM;
      int r0, r1;  // first W rows of the two units
      if (nt < p.n_qkv_tiles) {
        r0 = 2 * nt * kUnit;
        r1 = 2 * nt + 1 < n_units ? r0 + kUnit : r0;  // a missing second unit is not stored
      } else {
        const int64_t j = nt - p.n_qkv_tiles;
        r0 = static_cast<int>(3 * inner + j * kUnit);
        r1 = static_cast<int>(3 * inner + p.mlp + j * kUnit);
      }
      const int rw = crank == 0 ? r0 : r1;
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % kPStages;
        const uint32_t use = static_cast<uint32_t>(it / kPStages);
        if (!(ok = mbar_wait_cluster(bar(kBarEmpty + s), (use & 1u) ^ 1u, abort_flag))) break;
        const uint32_t dst = sbase + s * kPStageBytes;
        // both CTAs' copies complete on the even CTA's stage barrier
        if (crank == 0) mbar_arrive_expect_tx(bar(kBarFull + s), 2 * kPStageBytes);
        const uint32_t full0 = mapa_shared(bar(kBarFull + s), 0);
        tma_load_2d_pair(dst, &maps.x, full0, ks * kPK, m0);
        tma_load_2d_pair(dst + kPABytes, &maps.w, full0, ks * kPK, rw);
      }
    }
    // every copy of the pair has landed before the CTAs exit (the even CTA's
    // stage barriers count both CTAs' copies; the final cluster barrier
    // keeps the odd CTA until then)
    if (crank == 0)
      for (int j = (it > kPStages ? it - kPStages : 0); j < it; ++j)
        drain(bar(kBarFull + j % kPStages), static_cast<uint32_t>(j / kPStages) & 1u);
  } else if (warp == 1 && crank == 0) {
    // ------------------------------------------------ MMA issuer (even CTA)
    const uint32_t idesc = idesc_bf16_f32(2 * kPM, kPN, 0, 0);
    int it = 0;
    int lt = 0;
    bool ok = true;
    for (int t = cid; ok && t < p.n_tiles; t += ncl, ++lt) {
      const int buf = lt & 1;
      const uint32_t acc_par = ((static_cast<uint32_t>(lt) >> 1) & 1u) ^ 1u;
      if (!(ok = mbar_wait_cluster(bar(kBarAccEmpty + buf), acc_par, abort_flag))) break;
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after_sync();
      const uint32_t d = tmem + static_cast<uint32_t>(buf * kPN);
      for (int ks = 0; ks < nk; ++ks, ++it) {
        const int s = it % kPStages;
        const uint32_t par = static_cast<uint32_t>(it / kPStages) & 1u;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(kBarFull + s), par,
                                                               abort_flag))))
          break;
        tc_fence_after_sync();
        const uint64_t da = sdesc_sw128(sbase + s * kPStageBytes, 16, 1024);
        const uint64_t db = sdesc_sw128(sbase + s * kPStageBytes + kPABytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kPK / 16; ++kk)
          mma_ss_pair_elect(d, desc_advance(da, kk * 32), desc_advance(db, kk * 32), idesc,
                            (ks | kk) != 0 ? 1u : 0u);
        mma_commit_pair_elect(bar(kBarEmpty + s), kPairMask);  // both CTAs may refill
      }
      if (!ok) break;
      mma_commit_pair_elect(bar(kBarAccFull + buf), kPairMask);  // both accumulators complete
    }
    // every MMA issued above has finished before TMEM is released
    mma_commit_pair_elect(bar(kBarDrainP), 0x1);
    const long long t0 = clock64();
    while (!mbar_try_wait(bar(kBarDrainP), 0) && clock64() - t0 < kWaitBudgetCycles) {
    }
    __syncwarp();
  } else if (warp >= 4) {
    // -------------------------------------------------------------- epilogue
    const int wq = warp & 3;  // TMEM lane quadrant
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t acc_empty0 = mapa_shared(bar(kBarAccEmpty), 0);
    const uint32_t stage = sbase + kPOffStage + static_cast<uint32_t>(wq) * 2 * kPBoxBytes;
    int nbox = 0;  // boxes this warp has staged
    int lt = 0;
    bool ok = true;
    for (int t = cid; ok && t < p.n_tiles; t += ncl, ++lt) {
      const int nt = t / p.n_pb;
      const int64_t row0 = static_cast<int64_t>(t % p.n_pb) * (2 * kPM) + crank * kPM;
      const int buf = lt & 1;
      if (!(ok = __all_sync(0xffffffffu,
                            mbar_wait_cluster(bar(kBarAccFull + buf),
                                              (static_cast<uint32_t>(lt) >> 1) & 1u, abort_flag))))
        break;
      tc_fence_after_sync();
      const uint32_t tacc = tmem + static_cast<uint32_t>(buf * kPN) + lane_off;
      // One output box: features [f0, f0 + 64) of tensor `map`, staged from
      // 32-feature pieces; pv(c, w16) yields the 16 packed words of piece c.
      auto store_box = [&](const CUtensorMap *map, int f0, auto &&pv) {
        const uint32_t buf_addr = stage + static_cast<uint32_t>(nbox & 1) * kPBoxBytes;
        if (lane == 0) bulk_wait_read_1();  // the copy that last used this buffer has read it
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t w16[16];
          pv(c, w16);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            st_shared_v4(buf_addr + lane * 128 + (((c * 4 + i) ^ (lane & 7)) << 4),
                         make_uint4(w16[4 * i], w16[4 * i + 1], w16[4 * i + 2], w16[4 * i + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(map, buf_addr, f0, static_cast<int>(row0 + wq * 32));
          bulk_commit();
        }
        ++nbox;
      };
      if (nt < p.n_qkv_tiles) {
        for (int h = 0; h < 2; ++h) {
          const int u = 2 * nt + h;
          if (u >= n_units) break;
          const CUtensorMap *map = u < p.H ? &maps.q : u < 2 * p.H ? &maps.k : &maps.v;
          for (int half = 0; half < 2; ++half)
            store_box(map, (u % p.H) * kUnit + half * 64, [&](int c, uint32_t(&w16)[16]) {
              uint32_t r[32];
              tmem_ld32(tacc + h * kUnit + half * 64 + c * 32, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                w16[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            });
        }
      } else {
        const int j = nt - p.n_qkv_tiles;
        for (int half = 0; half < 2; ++half)
          store_box(&maps.act, j * kUnit + half * 64, [&](int c, uint32_t(&w16)[16]) {
            uint32_t g[32], uu[32];
            tmem_ld32(tacc + half * 64 + c * 32, g);
            tmem_ld32(tacc + kUnit + half * 64 + c * 32, uu);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w16[i] = pack_bf16x2(swiglu(__uint_as_float(g[2 * i]), __uint_as_float(uu[2 * i])),
                                   swiglu(__uint_as_float(g[2 * i + 1]),
                                          __uint_as_float(uu[2 * i + 1])));
          });
      }
      // this warp's TMEM reads are complete: the accumulator may be reused
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * static_cast<uint32_t>(buf));
    }
    if (lane == 0) bulk_wait_all();  // every output store is complete
  }

  // neither CTA leaves while the other may still signal its barriers or
  // read its shared memory
  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kPTmemCols);
  }
  if (tid == 0 && *abort_flag) atomicExch(status, FLUX_ERR_DEVICE_TIMEOUT);
}

// A row-major bf16 matrix [rows, cols] as a 2-D tensor map; one box = 64
// columns (128 bytes, 128-byte swizzle) x box_rows rows; rows past the end
// read as zeros and are not written.
bool make_rows_map(CUtensorMap *map, const void *x, int64_t rows, int64_t cols,
                   uint32_t box_rows = kPM) {
  auto fn = reinterpret_cast<CUresult (*)(
      CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill)>(
      tensor_map_encode_entry());
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kPK), box_rows};
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
  const int64_t n_pb = (M + 2 * kPM - 1) / (2 * kPM);  // 256-row blocks
  const int64_t n_qkv = (3 * static_cast<int64_t>(H) + 1) / 2;
  const int64_t n_tiles = n_pb * (n_qkv + mlp / kUnit);
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
  if (!make_rows_map(&maps.x, x, M, dim) || !make_rows_map(&maps.w, w, n_out, dim) ||
      !make_rows_map(&maps.q, q, M, inner, 32) || !make_rows_map(&maps.k, k, M, inner, 32) ||
      !make_rows_map(&maps.v, v, M, inner, 32) ||
      !make_rows_map(&maps.act, mlp > 0 ? act : q, M, mlp > 0 ? mlp : inner, 32))
    return cudaErrorInvalidValue;
  ProjShape p;
  p.M = M;
  p.mlp = mlp;
  p.dim = dim;
  p.H = H;
  p.n_pb = static_cast<int>(n_pb);
  p.n_qkv_tiles = static_cast<int>(n_qkv);
  p.n_tiles = static_cast<int>(n_tiles);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = kPSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: as many pairs as can be resident at once, no more than tiles
  static std::atomic<int> max_pairs[64];
  int np = max_pairs[dev].load(std::memory_order_relaxed);
  if (np == 0) {
    cfg.gridDim = dim3(2, 1, 1);
    e = cudaOccupancyMaxActiveClusters(&np, qkv_mlp_proj_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (np < 1) return cudaErrorInvalidConfiguration;
    max_pairs[dev].store(np, std::memory_order_relaxed);
  }
  const int64_t pairs = n_tiles < np ? n_tiles : np;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  return cudaLaunchKernelEx(&cfg, qkv_mlp_proj_kernel, maps, p, static_cast<uint16_t *>(q),
                            static_cast<uint16_t *>(k), static_cast<uint16_t *>(v),
                            static_cast<uint16_t *>(act), status);
}

}  // namespace flux
