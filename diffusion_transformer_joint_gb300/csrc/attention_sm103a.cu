// Joint RoPE attention forward for sm_103a (GB300): warp-specialised, with
// tcgen05 MMAs accumulating in tensor memory (TMEM), RoPE applied to Q and K
// while their tiles are staged into shared memory, V staged by TMA.
//
// Definition ("Transformer架构解析FLUX.2-klein-base-9b-nvfp4", section 2:
// scaled dot-product attention; "Diffusers 中 Flux2Transformer2DModel 全面解析",
// section 内部架构双流块与单流块: text and image tokens form one sequence):
//   out[b, i, h, :] = sum_j softmax_j(q^_i . k^_j / sqrt(128)) v[b, j, h, :]
// with q^, k^ the RoPE-rotated rows; non-causal over all S tokens.
//
// Persistent: one CTA per SM walks work items (batch, head, 256-row block)
// round robin; for each it owns 256 query rows (two 128-row tiles Q0, Q1)
// and walks every 128-key tile, starting at a tile that depends on its row
// block (spread evenly over the head). The K/V rings and every barrier phase
// run on across items, so the next item's Q is loaded while the current
// item's last tiles and epilogue finish.
// 16 warps in four warpgroups:
//   WG0  warp 0: TMA producer of Q and of K tiles (2-stage ring);
//        warp 1: MMA issuer (the whole warp walks the schedule, elect.sync
//        picks the issuing lane); warp 2: TMEM allocation;
//        warp 3: TMA producer of V tiles (2-stage ring).
//   WG1  softmax of Q0: thread = TMEM lane = query row.
//   WG2  softmax of Q1.
//   WG3  RoPE, from a work queue the producer fills: prepares the CTA's next
//        item (its Q rows and first two K tiles rotated global to global
//        into the exchange buffer) while the current one runs, and rotates
//        in shared memory any K tile that no CTA has published yet (one
//        adjacent channel pair per 32-bit word, table rows staged by TMA).
// The first item is prepared the same way by all 512 threads before the
// roles start.
// Rotated K is shared between the CTAs that work on one head: a CTA that
// rotates a K tile also stores it to an exchange buffer (a bf16 copy of K's
// layout) and sets one flag per RoPE warp; a CTA whose producer finds all
// four flags set for this launch loads the rotated tile from there straight
// into the K stage (no table, no RoPE warps). Staggered start tiles make
// the CTAs of a head rotate different tiles first. Without the buffer every
// CTA rotates every Q and K tile it loads in shared memory; the results are
// bit-identical.
// Every copy into shared memory is a TMA tile copy (128-byte swizzle for Q,
// K, V; out-of-range tokens read as zeros); only the preparation, off the
// MMA's path, uses plain global loads.
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512); the
// softmax writes P_t as packed bf16 over the first 64 columns of S_t and the
// MMA reads it from there (A operand in TMEM).
//
// Issue order of the MMA warp per key tile j:
//   S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...
// tcgen05 MMAs of one thread execute in order, so S_t(j+1) overwrites P_t(j)
// only after PV_t(j) has read it, and the commit that signals S_t(j+1) also
// covers PV_t(j): a softmax thread that sees S_t(j+1) may rescale O_t.
//
// Softmax runs in the log2 domain with a lazily updated running max: O and l
// are rescaled only when a row's max grows by more than 8 (a factor 256),
// which keeps exp2 arguments <= 8 and is exact after the final 1/l. The row
// max of a full key tile comes from the TMEM loads' own max reduction.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <mutex>
#include <random>

#include "flux_internal.h"
#include "ptx_sm103a.cuh"

namespace flux {
namespace {

constexpr int kD = 128;
constexpr int kBM = 128;  // rows per Q tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kQTiles = 2;
constexpr int kRowsPerCta = kBM * kQTiles;
constexpr int kThreads = 512;
constexpr int kStages = 2;  // K and V ring depth
constexpr int kPairs = kD / 2;
constexpr uint32_t kTileBytes = 128 * 128 * 2;
constexpr uint32_t kBlockBytes = 16384;          // one 64-channel swizzle block
constexpr uint32_t kStageWarpBytes = 32 * 64;  // epilogue staging: 32 rows x 32 channels bf16
constexpr uint32_t kTableRows = 64;              // table rows per shared-memory table load
constexpr uint32_t kTableBytes = kTableRows * kPairs * 4;  // 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kVPrefetch = 2;       // V tiles ahead of the copy that are prefetched into L2
constexpr int kQPrefetchTiles = 6;  // key tiles before an item's end its successor's Q is prefetched
constexpr int kPrepAtTile = 2;      // key tile of an item from which the next one is prepared
constexpr int kPrepMaxGap = 4;      // key tiles between two preparation pieces, at most
constexpr int kPrepChunks = 8;      // 64-row pieces: 4 of Q, 2 per K tile for the first two K tiles
// RoPE work queue entry: x = kind | stage << 4 | phase parity << 8 | tile << 9, y = item
constexpr uint32_t kRqQ = 1;     // rotate the item's two Q tiles in place (Q-raw -> Q-full)
constexpr uint32_t kRqK = 2;     // rotate a raw K tile in place (K-raw -> K-full), publish it
constexpr uint32_t kRqPrep = 3;  // prepare piece (x >> 4) of item y (rotated Q / first K tiles)
constexpr uint32_t kRqEnd = 4;   // no more work

// Shared-memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffQ = 0;                                   // Q0, Q1
constexpr uint32_t kOffK = kOffQ + kQTiles * kTileBytes;         // K ring
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;         // V ring
constexpr uint32_t kOffStage = kOffV + kStages * kTileBytes;     // one buffer per softmax warp
constexpr uint32_t kOffT = kOffStage + 8 * kStageWarpBytes;       // table rows for in-place RoPE
constexpr uint32_t kOffBar = kOffT + kTableBytes;                 // mbarriers
// barrier indices
constexpr int kBarQRaw = 0;
constexpr int kBarQFull = 1;
constexpr int kBarKRaw = 2;                  // + stage
constexpr int kBarKFull = kBarKRaw + kStages;
constexpr int kBarKEmpty = kBarKFull + kStages;
constexpr int kBarVFull = kBarKEmpty + kStages;
constexpr int kBarVEmpty = kBarVFull + kStages;
constexpr int kBarTFull = kBarVEmpty + kStages;  // table buffer loaded
constexpr int kBarTEmpty = kBarTFull + 1;         // every RoPE warp done with it
constexpr int kBarSFull = kBarTEmpty + 1;         // + q tile
constexpr int kBarPFull = kBarSFull + kQTiles;
constexpr int kBarODone = kBarPFull + kQTiles;
constexpr int kBarOFree = kBarODone + kQTiles;  // epilogue done reading O_t
constexpr int kBarQFree = kBarOFree + kQTiles;  // every S MMA of an item done
constexpr int kBarQPrep = kBarQFree + 1;  // next item's rotated Q is in the exchange buffer
constexpr int kRopeQ = 8;                  // RoPE work queue entries
constexpr int kBarRQFull = kBarQPrep + 1;  // + entry
constexpr int kBarRQEmpty = kBarRQFull + kRopeQ;
constexpr int kBarDrain = kBarRQEmpty + kRopeQ;
constexpr int kNumBars = kBarDrain + 1;
constexpr uint32_t kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kOffRQ = (kOffAbort + 4 + 7) & ~7u;  // RoPE work queue: uint2 per entry
constexpr uint32_t kSmemUsed = kOffRQ + 8 * kRopeQ;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");

// Register split (setmaxnreg): 512 threads x 128 registers at launch.
constexpr uint32_t kRegsSoftmax = 168;
constexpr uint32_t kRegsCopyMma = 72;  // WG0: producers, MMA issuer
constexpr uint32_t kRegsRope = 104;
static_assert(128 * (2 * kRegsSoftmax + kRegsCopyMma + kRegsRope) == 512 * 128,
              "warpgroup register shares must add up to the launch allocation");

__device__ __forceinline__ uint32_t sw128_offset(int r, int c16) {
  return static_cast<uint32_t>((c16 >> 3) * kBlockBytes + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  return sdesc_sw128(tile + (kk >> 2) * kBlockBytes + (kk & 3) * 32, 16, 1024);
}

__device__ __forceinline__ uint64_t desc_v(uint32_t tile, int kk) {
  return sdesc_sw128(tile + kk * 2048, kBlockBytes, 1024);
}

// Rotate the two bf16 channels packed in `w` by the fp16 (cos, sin) in `cs`.
__device__ __forceinline__ uint32_t rope_pair(uint32_t w, uint32_t cs) {
  const float x0 = bf16lo_to_f32(w), x1 = bf16hi_to_f32(w);
  const float c = f16lo_to_f32(cs), s = f16hi_to_f32(cs);
  return pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
}

// The same after scaling the two channels by s0 and s1 (the QK norm).
__device__ __forceinline__ uint32_t rope_pair_scaled(uint32_t w, uint32_t cs, float s0, float s1) {
  const float x0 = bf16lo_to_f32(w) * s0, x1 = bf16hi_to_f32(w) * s1;
  const float c = f16lo_to_f32(cs), s = f16hi_to_f32(cs);
  return pack_bf16x2(x0 * c - x1 * s, x0 * s + x1 * c);
}

// QK RMS normalisation applied before the rotation ("Diffusers 中
// Flux2Transformer2DModel 全面解析", sections 内部架构双流块与单流块 and
// 并行化支持: Q and K of each head are RMS-normalised over the head's 128
// channels after their projections, text and image tokens with their own
// learned weights; eps from 模型配置参数全解). For the tensor being rotated:
// the weights of text tokens (token < s_txt) and of the others.
struct QkNorm {
  const float *w_txt, *w_img;
  int64_t s_txt;
  float eps;
};

// This thread's 8 norm weights of each stream (16-byte chunk c16), loaded once
// per rotation call rather than once per row: a thread keeps the same chunk of
// every row it rotates. Only the kNorm paths call this (both pointers set).
struct NormW {
  float4 t0, t1, i0, i1;
};
__device__ __forceinline__ NormW load_norm_w(const QkNorm &nm, int c16) {
  const float4 *t = reinterpret_cast<const float4 *>(nm.w_txt + c16 * 8);
  const float4 *i = reinterpret_cast<const float4 *>(nm.w_img + c16 * 8);
  return NormW{__ldg(t), __ldg(t + 1), __ldg(i), __ldg(i + 1)};
}

// Per-channel scale of this thread's 8 channels (weights `nw`) of a row whose
// 8 bf16 values are `x`: the 16 lanes holding one row sum their squares across
// shuffles, so all 32 lanes of the warp must call this together.
__device__ __forceinline__ void qk_norm_scales(const uint4 &x, const QkNorm &nm, int64_t token,
                                               const NormW &nw, float (&sc)[8]) {
  const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = bf16lo_to_f32(wv[i]), b = bf16hi_to_f32(wv[i]);
    ss = fmaf(a, a, ss);
    ss = fmaf(b, b, ss);
  }
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss * (1.0f / kD) + nm.eps);
  const bool txt = token < nm.s_txt;
  const float4 w0 = txt ? nw.t0 : nw.i0, w1 = txt ? nw.t1 : nw.i1;
  sc[0] = r * w0.x; sc[1] = r * w0.y; sc[2] = r * w0.z; sc[3] = r * w0.w;
  sc[4] = r * w1.x; sc[5] = r * w1.y; sc[6] = r * w1.z; sc[7] = r * w1.w;
}

// Rotates the 8 channels of `x` with the (cos, sin) words `cs`, normalising
// them first when kNorm.
template <bool kNorm>
__device__ __forceinline__ uint4 rope_chunk(const uint4 &x, const uint4 &cs, const QkNorm &nm,
                                            int64_t token, const NormW &nw) {
  uint4 o;
  if (kNorm) {
    float sc[8];
    qk_norm_scales(x, nm, token, nw, sc);
    o.x = rope_pair_scaled(x.x, cs.x, sc[0], sc[1]);
    o.y = rope_pair_scaled(x.y, cs.y, sc[2], sc[3]);
    o.z = rope_pair_scaled(x.z, cs.z, sc[4], sc[5]);
    o.w = rope_pair_scaled(x.w, cs.w, sc[6], sc[7]);
  } else {
    o.x = rope_pair(x.x, cs.x);
    o.y = rope_pair(x.y, cs.y);
    o.z = rope_pair(x.z, cs.z);
    o.w = rope_pair(x.w, cs.w);
  }
  return o;
}

// Hides a value's origin from the optimiser (no code is emitted).
__device__ __forceinline__ void opaque(uint32_t &x) { asm volatile("" : "+r"(x)); }

template <uint32_t kRegs>
__device__ __forceinline__ void reg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void reg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// 128 RoPE threads rotate rows [64 half, 64 half + 64) of a swizzled tile in
// place with the (cos, sin) words of those rows at `tbl` in shared memory
// ([64 rows][64 pairs] uint32; rows past the sequence end hold zeros, as do
// the tile's). Thread u owns 16-byte column chunk u & 15 (channel pairs
// 4(u&15) .. +3) of every 8th row. With kPublish the rotated rows below
// rows_valid also go to global memory at grow + r * row_stride. With kNorm
// the rows (token tok0 + r) are RMS-normalised first.
template <bool kNorm, bool kPublish>
__device__ __forceinline__ void rotate_half(uint32_t tile, uint32_t tbl, int half, int u,
                                            const QkNorm &nm, int64_t tok0, int rows_valid,
                                            uint16_t *grow, int64_t row_stride) {
  const int c16 = u & 15;
  const int rsub = u >> 4;
  const NormW nw = kNorm ? load_norm_w(nm, c16) : NormW{};
  // batches of rows (four, or two with the norm's extra registers): all
  // loads of a batch in flight together
  constexpr int kBatch = kNorm ? 2 : 4;
#pragma unroll
  for (int i0 = 0; i0 < 8; i0 += kBatch) {
    uint4 w[kBatch], cs[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int rh = (i0 + i) * 8 + rsub;
      w[i] = ld_shared_v4(tile + sw128_offset(half * 64 + rh, c16));
      cs[i] = ld_shared_v4(tbl + rh * (kPairs * 4) + c16 * 16);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int r = half * 64 + (i0 + i) * 8 + rsub;
      const uint4 o = rope_chunk<kNorm>(w[i], cs[i], nm, tok0 + r, nw);
      st_shared_v4(tile + sw128_offset(r, c16), o);
      if (kPublish && r < rows_valid) st_global_v4(grow + r * row_stride + c16 * 8, o);
    }
  }
}

// 128 RoPE threads rotate `nrows` rows of one head from global memory to
// global memory: src / dst point at the first row's channel 0, rows are
// src_stride / dst_stride elements apart, `tab` at the first row's packed
// table row. Thread u owns 16-byte chunk u & 15 of rows (u >> 4) + 8 i, the
// row-to-thread map of rotate_half, so RoPE warp w writes the rows r with
// r mod 8 in {2w, 2w+1}.
// With kNorm the rows (token tok0 + r) are RMS-normalised first; every lane
// of the warp runs every iteration (rows past nrows are zeros, not stored).
template <bool kNorm>
__device__ __forceinline__ void rotate_rows_global(const uint16_t *src, uint16_t *dst,
                                                   const uint32_t *tab, int nrows,
                                                   int64_t src_stride, int64_t dst_stride, int u,
                                                   const QkNorm &nm, int64_t tok0) {
  const int c16 = u & 15;
  const int rsub = u >> 4;
  const NormW nw = kNorm ? load_norm_w(nm, c16) : NormW{};
#pragma unroll 1
  for (int i0 = 0; (kNorm ? 8 * i0 : rsub + 8 * i0) < nrows; i0 += 2) {
    uint4 w[2], cs[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = rsub + 8 * (i0 + i);
      w[i] = make_uint4(0u, 0u, 0u, 0u);
      cs[i] = make_uint4(0u, 0u, 0u, 0u);
      if (r < nrows) {
        w[i] = ld_global_nc_v4(src + r * src_stride + c16 * 8);
        cs[i] = ld_global_nc_v4(tab + static_cast<int64_t>(r) * kPairs + c16 * 4);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = rsub + 8 * (i0 + i);
      const uint4 o = rope_chunk<kNorm>(w[i], cs[i], nm, tok0 + r, nw);
      if (r < nrows) st_global_v4(dst + r * dst_stride + c16 * 8, o);
    }
  }
}

// kpre / vpre: keys and values that arrive rotated already (a reference-image
// cache), appended to a segment's key range.
struct Maps {
  CUtensorMap q, k, v, out, krot, qrot, table_q, table_k, kpre, vpre;
};

// A work item: batch b, head h of Q / K / V / out (hx: its index among the
// launch's heads, which lay out the exchange buffer), the 256 query rows from
// m0 (rows of Q / out at or past q_hi belong to another segment: computed,
// never stored), its key
// range: rows [k_lo, k_hi) of K / V in n_main 128-key tiles, then rows
// [0, n_pre) of the pre-rotated K / V in the remaining tiles of n_tiles, all
// walked from tile j0; and the publication flags of the n_main tiles for
// (b, h) ([n_main][4]; null without the exchange buffer).
struct Item {
  int b, h, hx, n_tiles, n_main, j0;
  int64_t m0, q_hi, k_lo, k_hi, n_pre;
  uint64_t *flags;
};

// The segments of one launch, by value: segment g owns items
// [first_item[g], first_item[g + 1]), queries [q_lo, q_hi) in n_rb 256-row
// blocks, keys [k_lo, k_hi) in n_main tiles and n_pre pre-rotated keys, n_tiles
// tiles in all; flag_off is the word offset of its key range's flags in the
// exchange buffer.
struct Segs {
  int n;
  int first_item[kMaxSegments + 1];
  int n_rb[kMaxSegments], n_tiles[kMaxSegments], n_main[kMaxSegments];
  int64_t q_lo[kMaxSegments], q_hi[kMaxSegments], k_lo[kMaxSegments], k_hi[kMaxSegments];
  int64_t n_pre[kMaxSegments], flag_off[kMaxSegments];
};

// mbar_wait for warp-collective roles (softmax, RoPE): every lane waits and the
// lanes agree on the outcome, so an abort never splits a warp between a
// warp-collective instruction (tcgen05.ld/st, __syncwarp) and the exit path.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int *abort_flag) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// One arrival per warp on a hand-off barrier (initialised with the number of
// arriving warps): every lane has finished its part (its smem writes fenced
// for the async proxy, its TMEM stores waited and fenced) before __syncwarp,
// then lane 0 arrives for the warp. Four arrivals instead of 128 shorten the
// hand-off.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// After an abort: wait (bounded, regardless of the abort flag) until the
// phase of a TMA barrier completes, so that no copy this thread issued is
// still in flight when the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitBudgetCycles) {
  }
}

// Checked build (-DFLUX_DEBUG): before each shared-memory, TMEM, TMA and
// global (exchange buffer, flags, tables, inputs, output) access site listed
// in DbgSite, the kernel checks that the region, stage, lane quadrant, column
// range, coordinates and row range it is about to use lie inside what that
// site may touch. A failed check skips the access and records its site (the
// first one of the launch); at exit the CTA writes FLUX_DEBUG_STATUS_BASE -
// site into the status word. Nothing traps. Release builds compile every
// check to `true`.
enum DbgSite {
  kDbgQLoad = 1,       // producer: Q tile copies (raw or rotated)
  kDbgKLoad = 2,       // producer: K tile copies (raw, rotated or pre-rotated)
  kDbgFlagRead = 3,    // producer: publication flags of a K tile
  kDbgVLoad = 4,       // V producer: V tile copies
  kDbgMmaS = 5,        // MMA: S = Q K^T operands
  kDbgMmaPV = 6,       // MMA: O += P V operands
  kDbgSLoad = 7,       // softmax: S columns read from TMEM
  kDbgORescale = 8,    // softmax: O columns rescaled in TMEM
  kDbgPStore = 9,      // softmax: P columns written to TMEM
  kDbgOLoad = 10,      // epilogue: O columns read from TMEM
  kDbgStage = 11,      // epilogue: per-warp staging buffer
  kDbgOutRow = 12,     // epilogue: row-by-row global stores
  kDbgOutTma = 13,     // epilogue: TMA tile stores
  kDbgTableLoad = 14,  // RoPE: table rows copied to shared memory
  kDbgQRotate = 15,    // RoPE: Q tile rotated in place
  kDbgKRotate = 16,    // RoPE: K tile rotated in place and published
  kDbgPrepare = 17,    // RoPE: next item's rows rotated global to global
  kDbgQueue = 18,      // RoPE: work queue entry decoded
};
#ifdef FLUX_DEBUG
__device__ int g_dbg_site;  // first failed check of the current launch, 0 if none
__device__ __forceinline__ bool dbg_check(bool ok, int site) {
  if (!ok) atomicCAS(&g_dbg_site, 0, site);
  return ok;
}
#define FLUX_DBG(cond, site) dbg_check((cond), (site))
#else
#define FLUX_DBG(cond, site) true
#endif

// kNorm: Q and K are RMS-normalised (qn / kn) before the rotation.
template <bool kNorm>
__global__ void __launch_bounds__(kThreads, 1)
    joint_rope_attention_kernel(const __grid_constant__ Maps maps, uint16_t *__restrict__ outg,
                                int *__restrict__ status,
                                const Segs sg, int B, int64_t S_q, int64_t S_k, int H, int h0,
                                int Hl, int n_items, int64_t n_flag_words,
                                uint64_t *__restrict__ kflags, uint16_t *__restrict__ krot,
                                uint16_t *__restrict__ qrot, const uint16_t *__restrict__ qg,
                                const uint16_t *__restrict__ kg,
                                const uint32_t *__restrict__ tabq,
                                const uint32_t *__restrict__ tabk, uint64_t token,
                                const QkNorm qn, const QkNorm kn) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(base);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + kOffTmemSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(base + kOffAbort);

  const int tid = static_cast<int>(threadIdx.x);
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // [addr, addr + bytes) inside the shared-memory region [off, off + size)
  auto in_smem = [&](uint32_t addr, uint32_t bytes, uint32_t off, uint32_t size) {
    return addr >= sbase + off && addr + bytes <= sbase + off + size;
  };
  (void)in_smem;
  // token strides (elements) of Q / K / V / out (all H heads) and of the
  // exchange buffer (the launch's Hl heads h0 .. h0 + Hl - 1)
  const int64_t row_stride = static_cast<int64_t>(H) * kD;
  const int64_t xrow_stride = static_cast<int64_t>(Hl) * kD;
  const bool share = kflags != nullptr;
  // Work items: segment by segment, (batch, head, 256-row block) with the row
  // block fastest, handed out round robin, so CTAs running at the same time
  // share the K/V of a few heads in L2. Key tiles are walked from a start
  // tile that depends on the row block, spread evenly over the key range:
  // the CTAs working on one head at the same time each rotate different K
  // tiles first and publish them (kflags / krot), and later each mostly
  // loads tiles another CTA rotated.
  auto info = [&](int item) {
    Item it;
    int g = 0;
    while (g + 1 < sg.n && item >= sg.first_item[g + 1]) ++g;
    const int local = item - sg.first_item[g];
    const int nrb = sg.n_rb[g];
    const int rb = local % nrb;
    const int bh = local / nrb;
    it.hx = bh % Hl;
    it.h = h0 + it.hx;
    it.b = bh / Hl;
    it.m0 = sg.q_lo[g] + static_cast<int64_t>(rb) * kRowsPerCta;
    it.q_hi = sg.q_hi[g];
    it.k_lo = sg.k_lo[g];
    it.k_hi = sg.k_hi[g];
    it.n_tiles = sg.n_tiles[g];
    it.n_main = sg.n_main[g];
    it.n_pre = sg.n_pre[g];
    it.j0 = static_cast<int>((static_cast<int64_t>(rb) * it.n_tiles) / nrb);
    it.flags = share ? kflags + sg.flag_off[g] +
                           (static_cast<int64_t>(it.b) * Hl + it.hx) * it.n_main * 4
                     : nullptr;
    return it;
  };
  auto tile_at = [&](const Item &it, int j) {
    return it.j0 + j < it.n_tiles ? it.j0 + j : it.j0 + j - it.n_tiles;
  };
  // first key row of tile tj of the item's key range: a row of K / V for the
  // first n_main tiles, of the pre-rotated K / V after them
  auto tile_row = [&](const Item &it, int tj) {
    return tj < it.n_main ? it.k_lo + static_cast<int64_t>(tj) * kBN
                          : static_cast<int64_t>(tj - it.n_main) * kBN;
  };
  // keys of tile tj that belong to the key range (the rest are masked)
  auto tile_keys = [&](const Item &it, int tj) {
    const int64_t kv = (tj < it.n_main ? it.k_hi : it.n_pre) - tile_row(it, tj);
    return static_cast<int>(kv < kBN ? kv : kBN);
  };

  if (tid == 0) {
    mbar_init(bar(kBarQRaw), 1);
    mbar_init(bar(kBarQFull), 4);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarKRaw + s), 1);
      mbar_init(bar(kBarKFull + s), 4);
      mbar_init(bar(kBarKEmpty + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(bar(kBarSFull + t), 1);
      mbar_init(bar(kBarPFull + t), 4);
      mbar_init(bar(kBarODone + t), 1);
      mbar_init(bar(kBarOFree + t), 4);
    }
    mbar_init(bar(kBarQFree), 1);
    mbar_init(bar(kBarQPrep), 4);
    mbar_init(bar(kBarTFull), 1);
    mbar_init(bar(kBarTEmpty), 4);
    for (int e = 0; e < kRopeQ; ++e) {
      mbar_init(bar(kBarRQFull + e), 1);
      mbar_init(bar(kBarRQEmpty + e), 4);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  // The first item is prepared here by all 512 threads, before any role has
  // work: its Q rows and its first two K tiles (those in the main key range)
  // rotated into the exchange buffer, as the RoPE warps prepare every later
  // item while the one before it runs. Thread t owns 16-byte chunk t & 15 of
  // rows (t >> 4) + 32 i: i < 8 the item's 256 Q rows, i >= 8 rows of K tile
  // (i - 8) >> 2. With the norm every thread runs every row (the row sums are
  // shuffles across 16 lanes); rows past the tensor's end are not stored.
  const bool first_prep = share && static_cast<int>(blockIdx.x) < n_items;
  if (first_prep) {
    grid_dep_wait();  // the rotation reads the tables
    const Item it = info(static_cast<int>(blockIdx.x));
    const bool prep_ok = FLUX_DBG(
        it.b < B && it.h < H && it.hx < Hl && it.m0 >= 0 && it.m0 < S_q &&
            it.flags - kflags + static_cast<int64_t>(it.n_main) * 4 <= n_flag_words,
        kDbgPrepare);
    const int r0 = tid >> 4, c16 = tid & 15;
    constexpr int kB = kNorm ? 4 : 8;  // rows with loads in flight together
#pragma unroll 1
    for (int g = 0; g < 16; g += kB) {
      const bool is_q = g < 8;
      const NormW nw = kNorm ? load_norm_w(is_q ? qn : kn, c16) : NormW{};
      uint4 w[kB], cs[kB];
      int64_t tok[kB];
      uint16_t *dst[kB];
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        bool valid;
        const uint16_t *src;
        const uint32_t *tab;
        if (is_q) {
          tok[i] = it.m0 + r0 + 32 * (g + i);
          valid = tok[i] < S_q;
          src = qg + ((static_cast<int64_t>(it.b) * S_q + tok[i]) * H + it.h) * kD;
          dst[i] = qrot + ((static_cast<int64_t>(it.b) * S_q + tok[i]) * Hl + it.hx) * kD;
          tab = tabq;
        } else {
          const int kt = (g + i - 8) >> 2;
          const bool in_main = kt < it.n_tiles && tile_at(it, kt) < it.n_main;
          tok[i] = (in_main ? tile_row(it, tile_at(it, kt)) : 0) + r0 + 32 * ((g + i - 8) & 3);
          valid = in_main && tok[i] < S_k;
          src = kg + ((static_cast<int64_t>(it.b) * S_k + tok[i]) * H + it.h) * kD;
          dst[i] = krot + ((static_cast<int64_t>(it.b) * S_k + tok[i]) * Hl + it.hx) * kD;
          tab = tabk;
        }
        if (!(valid && prep_ok)) dst[i] = nullptr;
        w[i] = make_uint4(0u, 0u, 0u, 0u);
        cs[i] = make_uint4(0u, 0u, 0u, 0u);
        if (dst[i] != nullptr) {
          w[i] = ld_global_nc_v4(src + c16 * 8);
          cs[i] = ld_global_nc_v4(tab + tok[i] * kPairs + c16 * 4);
        }
      }
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        const uint4 o = rope_chunk<kNorm>(w[i], cs[i], is_q ? qn : kn, tok[i], nw);
        if (dst[i] != nullptr) st_global_v4(dst[i] + c16 * 8, o);
      }
    }
    fence_proxy_async_global();  // read by the producer's TMA copies
    fence_acq_rel_gpu();         // ... and by other CTAs once the flags below are set
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (first_prep && tid < 8) {
    // publish the two K tiles: every thread's rows are written (the barrier
    // above); one thread per flag word
    const Item it = info(static_cast<int>(blockIdx.x));
    const int kt = tid >> 2;
    if (kt < it.n_tiles && tile_at(it, kt) < it.n_main &&
        FLUX_DBG(it.flags - kflags + static_cast<int64_t>(tile_at(it, kt)) * 4 + 4 <= n_flag_words,
                 kDbgPrepare)) {
      fence_acq_rel_gpu();
      st_relaxed_gpu_u64(it.flags + static_cast<int64_t>(tile_at(it, kt)) * 4 + (tid & 3), token);
    }
  }
  const uint32_t tmem = *tmem_slot;
  // TMEM columns [col, col + n) of this warp's lane quadrant, inside [lo, hi)
  // of the allocation
  auto in_tmem = [&](uint32_t taddr, uint32_t n, uint32_t lo, uint32_t hi) {
    const uint32_t col = (taddr & 0xFFFFu) - (tmem & 0xFFFFu);
    return (taddr >> 16) - (tmem >> 16) == static_cast<uint32_t>((warp & 3) * 32) && col >= lo &&
           col + n <= hi && hi <= kTmemCols;
  };
  (void)in_tmem;

  const uint32_t idesc_qk = idesc_bf16_f32(128, 128, 0, 0);
  const uint32_t idesc_pv = idesc_bf16_f32(128, 128, 0, 1);

  if (warp < 4) {
    reg_dec<kRegsCopyMma>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------- producer: Q and K
      // Every copy that needs rotating is announced to the RoPE warps through
      // the work queue; already rotated tiles go straight to the MMA.
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      if (share) {
        tma_prefetch_desc(&maps.krot);
        tma_prefetch_desc(&maps.qrot);
      }
      int jt = 0;  // K tiles issued so far (all items)
      int pq = 0;  // queue entries posted so far
      bool ok = true;
      auto post = [&](uint32_t x, uint32_t y) {
        const int e = pq % kRopeQ;
        const uint32_t use = static_cast<uint32_t>(pq / kRopeQ);
        if (!(ok = mbar_wait(bar(kBarRQEmpty + e), (use & 1u) ^ 1u, abort_flag))) return;
        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(sbase + kOffRQ + 8 * e), "r"(x),
                     "r"(y)
                     : "memory");
        mbar_arrive(bar(kBarRQFull + e));  // release: the entry is visible to the waiters
        ++pq;
      };
      int k = 0;
      int q_local = 0;                 // Q loads rotated in place (Q-raw phases)
      // bit s: parity of the raw K copies into stage s so far (K-raw phases)
      uint32_t raw_par = 0;
      int last_q_bar = -1;  // barrier / parity the last Q copy completes
      uint32_t last_q_parity = 0;
      // per K stage s (bit s): the last copy went straight to K-full, and the
      // parity of the phase it completes
      uint32_t last_k_full = 0, last_k_par = 0;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++k) {
        const Item it = info(item);
        const int b = it.b, h = it.h, hx = it.hx, m0 = static_cast<int>(it.m0);
        const int next = item + static_cast<int>(gridDim.x);
        // the previous item's S MMAs no longer read the Q buffers
        if (k > 0 && !(ok = mbar_wait(bar(kBarQFree), static_cast<uint32_t>(k - 1) & 1u, abort_flag)))
          break;
        if (share) {
          // This item's Q is in the exchange buffer, rotated (the first
          // item's by the whole CTA before the roles started, every later
          // one's by the RoPE warps during the previous item): copy it in,
          // completing Q-full (its other three arrivals made here) without
          // the RoPE warps.
          if (k > 0 &&
              !(ok = mbar_wait(bar(kBarQPrep), static_cast<uint32_t>(k - 1) & 1u, abort_flag)))
            break;
          fence_proxy_async_global();
          last_q_bar = kBarQFull;
          last_q_parity = static_cast<uint32_t>(k) & 1u;
          if (FLUX_DBG(hx < Hl && b < B && m0 >= 0 && m0 < S_q, kDbgQLoad)) {
            mbar_arrive_expect_tx(bar(kBarQFull), kQTiles * kTileBytes);
            for (int t = 0; t < kQTiles; ++t) {
              const uint32_t dst = sbase + kOffQ + t * kTileBytes;
              tma_load_4d(dst, &maps.qrot, bar(kBarQFull), 0, hx, m0 + t * kBM, b);
              tma_load_4d(dst + kBlockBytes, &maps.qrot, bar(kBarQFull), 64, hx, m0 + t * kBM, b);
            }
          } else {
            mbar_arrive(bar(kBarQFull));  // checked build: no copy, the phase still completes
          }
          mbar_arrive_n(bar(kBarQFull), 3);
        } else {
          last_q_bar = kBarQRaw;
          last_q_parity = static_cast<uint32_t>(q_local) & 1u;
          const bool q_ok = FLUX_DBG(h < H && b < B && m0 >= 0 && m0 < S_q, kDbgQLoad);
          if (q_ok) mbar_arrive_expect_tx(bar(kBarQRaw), kQTiles * kTileBytes);
          else mbar_arrive(bar(kBarQRaw));  // checked build: no copy, the phase still completes
          for (int t = 0; q_ok && t < kQTiles; ++t) {
            const uint32_t dst = sbase + kOffQ + t * kTileBytes;
            tma_load_4d(dst, &maps.q, bar(kBarQRaw), 0, h, m0 + t * kBM, b);
            tma_load_4d(dst + kBlockBytes, &maps.q, bar(kBarQRaw), 64, h, m0 + t * kBM, b);
          }
          post(kRqQ | (last_q_parity << 8), static_cast<uint32_t>(item));
          ++q_local;
        }
        const int n_tiles = it.n_tiles;
        const int prep_at = n_tiles > kPrepAtTile ? kPrepAtTile : n_tiles - 1;
        // Preparation pieces for the next item are posted every `gap` key
        // tiles: up to kPrepMaxGap apart, and close enough that the last one
        // is posted at least two tiles before the item's end. Posted one per
        // tile the kernel was 2-4% slower (spread out, fewer pieces wait in
        // the RoPE queue ahead of a raw K tile that the MMA needs rotated).
        int pieces = 0;
        const int span = (n_tiles - prep_at - 2) / kPrepChunks;
        const int gap = span < 1 ? 1 : (span > kPrepMaxGap ? kPrepMaxGap : span);
        for (int j = 0; ok && j < n_tiles; ++j, ++jt) {
          const int s = jt % kStages;
          const int tj = tile_at(it, j);
          const int krow = static_cast<int>(tile_row(it, tj));
          const uint32_t use = static_cast<uint32_t>(jt / kStages);
          // Has every RoPE warp of some CTA published tile tj? Decided (and
          // the acquire fence paid) before the ring wait, which hides both.
          // The first two tiles of an item were rotated by this CTA, ordered
          // before this point by the Q-prep wait (the first item's by the
          // barrier before the roles). Pre-rotated tiles need no rotation.
          const bool pre = tj >= it.n_main;
          bool rotated = pre || (share && j < 2);
          if (share && !rotated &&
              FLUX_DBG(it.flags - kflags + static_cast<int64_t>(tj) * 4 + 4 <= n_flag_words &&
                           tj < it.n_main,
                       kDbgFlagRead)) {
            const uint64_t *fl = it.flags + static_cast<int64_t>(tj) * 4;
            uint64_t f0, f1, f2, f3;
            // acquire loads: a set flag orders the publisher's rows before
            // this thread's later accesses (a full GPU-scope fence here cost
            // the producer more than the loads themselves)
            ld_acquire_gpu_v2_u64(fl, f0, f1);
            ld_acquire_gpu_v2_u64(fl + 2, f2, f3);
            rotated = f0 == token && f1 == token && f2 == token && f3 == token;
            if (rotated) fence_proxy_async_global();  // ... and before the TMA copy below
          }
          if (!(ok = mbar_wait(bar(kBarKEmpty + s), (use & 1u) ^ 1u, abort_flag))) break;
          if (share && !rotated &&
              FLUX_DBG(it.flags - kflags + static_cast<int64_t>(tj) * 4 + 4 <= n_flag_words,
                       kDbgFlagRead)) {
            // A second look once the ring slot is free: decided early, the
            // first look misses tiles the CTAs that started the head at the
            // same time publish while this one waits (the first item's tiles
            // after its own two).
            const uint64_t *fl = it.flags + static_cast<int64_t>(tj) * 4;
            uint64_t f0, f1, f2, f3;
            ld_acquire_gpu_v2_u64(fl, f0, f1);
            ld_acquire_gpu_v2_u64(fl + 2, f2, f3);
            rotated = f0 == token && f1 == token && f2 == token && f3 == token;
            if (rotated) fence_proxy_async_global();
          }
          const uint32_t dst = sbase + kOffK + s * kTileBytes;
          if (!FLUX_DBG(in_smem(dst, kTileBytes, kOffK, kStages * kTileBytes) && tj >= 0 &&
                            tj < it.n_tiles && krow >= 0 &&
                            krow < (pre ? it.n_pre : it.k_hi) && krow >= (pre ? 0 : it.k_lo) &&
                            h < H && hx < Hl && b < B,
                        kDbgKLoad)) {
            // checked build: no copy; K-full completes without it
            last_k_full |= 1u << s;
            last_k_par = (last_k_par & ~(1u << s)) | ((use & 1u) << s);
            mbar_arrive_n(bar(kBarKFull + s), 4);
          } else if (rotated) {
            // straight to the MMA: the copy completes K-full, whose other
            // three arrivals are made here
            last_k_full |= 1u << s;
            last_k_par = (last_k_par & ~(1u << s)) | ((use & 1u) << s);
            const CUtensorMap *src = pre ? &maps.kpre : &maps.krot;
            const int hs = pre ? h : hx;  // the cache has all H heads
            mbar_arrive_expect_tx(bar(kBarKFull + s), kTileBytes);
            tma_load_4d(dst, src, bar(kBarKFull + s), 0, hs, krow, b);
            tma_load_4d(dst + kBlockBytes, src, bar(kBarKFull + s), 64, hs, krow, b);
            mbar_arrive_n(bar(kBarKFull + s), 3);
          } else {
            const uint32_t par = (raw_par >> s) & 1u;
            raw_par ^= 1u << s;
            last_k_full &= ~(1u << s);
            last_k_par = (last_k_par & ~(1u << s)) | (par << s);
            mbar_arrive_expect_tx(bar(kBarKRaw + s), kTileBytes);
            tma_load_4d(dst, &maps.k, bar(kBarKRaw + s), 0, h, krow, b);
            tma_load_4d(dst + kBlockBytes, &maps.k, bar(kBarKRaw + s), 64, h, krow, b);
            post(kRqK | (static_cast<uint32_t>(s) << 4) | (par << 8) |
                     (static_cast<uint32_t>(tj) << 9),
                 static_cast<uint32_t>(item));
          }
          // after this tile's own copy (and its in-place rotation, if any, is
          // queued ahead of the preparation piece)
          while (share && next < n_items && pieces < kPrepChunks &&
                 (j >= prep_at + gap * pieces || j == n_tiles - 1)) {
            post(kRqPrep | (static_cast<uint32_t>(pieces) << 4), static_cast<uint32_t>(next));
            ++pieces;
          }
          if (!ok) break;
          // the next item's raw Q into L2 a few tiles before it is loaded (with
          // the exchange buffer the RoPE warps have read it long before)
          if (!share && j == (n_tiles > kQPrefetchTiles ? n_tiles - kQPrefetchTiles : 0) &&
              next < n_items) {
            const Item nx = info(next);
            const int nm0 = static_cast<int>(nx.m0);
            for (int t = 0; t < kQTiles && nm0 + t * kBM < S_q; ++t) {
              tma_prefetch_l2_4d(&maps.q, 0, nx.h, nm0 + t * kBM, nx.b);
              tma_prefetch_l2_4d(&maps.q, 64, nx.h, nm0 + t * kBM, nx.b);
            }
          }
        }
      }
      if (ok) post(kRqEnd, 0);
      {  // every copy issued above has landed before the CTA exits (a no-op
         // unless an abort left some unconsumed)
        if (last_q_bar >= 0) drain_wait(bar(last_q_bar), last_q_parity);
        for (int jj = (jt > kStages ? jt - kStages : 0); jj < jt; ++jj) {
          const int sj = jj % kStages;
          drain_wait(bar(((last_k_full >> sj) & 1u) ? kBarKFull + sj : kBarKRaw + sj),
                     (last_k_par >> sj) & 1u);
        }
      }
    } else if (warp == 3 && lane == 0) {
      // ------------------------------------------------------ producer: V
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.vpre);
      int jt = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const Item it = info(item);
        const int b = it.b, h = it.h, n_tiles = it.n_tiles;
        for (int j = 0; j < n_tiles; ++j, ++jt) {
          const int s = jt % kStages;
          const int tj = tile_at(it, j);
          const int vrow = static_cast<int>(tile_row(it, tj));
          const CUtensorMap *src = tj < it.n_main ? &maps.v : &maps.vpre;
          const uint32_t use = static_cast<uint32_t>(jt / kStages);
          if (!(ok = mbar_wait(bar(kBarVEmpty + s), (use & 1u) ^ 1u, abort_flag))) break;
          const uint32_t dst = sbase + kOffV + s * kTileBytes;
          [[maybe_unused]] const bool main_tile = tj < it.n_main;
          if (!FLUX_DBG(in_smem(dst, kTileBytes, kOffV, kStages * kTileBytes) && tj >= 0 &&
                            tj < it.n_tiles && vrow >= (main_tile ? it.k_lo : 0) &&
                            vrow < (main_tile ? it.k_hi : it.n_pre) && h < H && b < B,
                        kDbgVLoad)) {
            mbar_arrive(bar(kBarVFull + s));  // checked build: no copy, the phase completes
            continue;
          }
          mbar_arrive_expect_tx(bar(kBarVFull + s), kTileBytes);
          tma_load_4d(dst, src, bar(kBarVFull + s), 0, h, vrow, b);
          tma_load_4d(dst + kBlockBytes, src, bar(kBarVFull + s), 64, h, vrow, b);
          // the tile two ahead into L2 now, so that its copy does not wait on
          // DRAM when the ring frees up
          if (j + kVPrefetch < n_tiles) {
            const int pj = tile_at(it, j + kVPrefetch);
            const int prow = static_cast<int>(tile_row(it, pj));
            const CUtensorMap *psrc = pj < it.n_main ? &maps.v : &maps.vpre;
            tma_prefetch_l2_4d(psrc, 0, h, prow, b);
            tma_prefetch_l2_4d(psrc, 64, h, prow, b);
          }
        }
      }
      // every copy issued above has landed before the CTA exits (a no-op
      // unless an abort left some unconsumed)
      for (int jj = (jt > kStages ? jt - kStages : 0); jj < jt; ++jj)
        drain_wait(bar(kBarVFull + jj % kStages), static_cast<uint32_t>(jj / kStages) & 1u);
    } else if (warp == 1) {
      // ------------------------------------------------------ MMA issuer
      // The whole warp walks the schedule (its waits are warp-collective);
      // elect.sync picks the lane that issues each tcgen05 instruction.
      // TMEM: S_t at column 128 t, O_t at 256 + 128 t; Q_t at kOffQ + t * kTileBytes
      const uint64_t dq0 = desc_kmajor(sbase + kOffQ, 0);
      const uint64_t dk0 = desc_kmajor(sbase + kOffK, 0);
      const uint64_t dv0 = desc_v(sbase + kOffV, 0);
      // upper descriptor word, the same for Q, K and V (stride and layout)
      const uint32_t desc_hi = static_cast<uint32_t>(dq0 >> 32);
      (void)FLUX_DBG(static_cast<uint32_t>(dk0 >> 32) == desc_hi &&
                         static_cast<uint32_t>(dv0 >> 32) == desc_hi,
                     kDbgMmaS);
      auto issue_s = [&](int t, int sk) {
        if (!FLUX_DBG(t >= 0 && t < kQTiles && sk >= 0 && sk < kStages, kDbgMmaS)) return;
        uint32_t da = static_cast<uint32_t>(desc_advance(dq0, t * kTileBytes));
        uint32_t db = static_cast<uint32_t>(desc_advance(dk0, sk * kTileBytes));
        opaque(da);  // per-MMA descriptors are base + constant, computed here,
        opaque(db);  // not hoisted into registers for every (t, stage, kk)
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kBlockBytes + (kk & 3) * 32) >> 4;
          mma_ss_elect(tmem + t * 128, da + off, db + off, desc_hi, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar(kBarSFull + t));
      };
      int jt = 0;  // first global K/V tile index of the current item
      bool ok = true;
      int k = 0;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++k) {
        const int n_tiles = info(item).n_tiles;
        if (!(ok = mbar_wait_warp(bar(kBarQFull), static_cast<uint32_t>(k) & 1u, abort_flag))) break;
        {
          const int s0 = jt % kStages;
          if (!(ok = mbar_wait_warp(bar(kBarKFull + s0), static_cast<uint32_t>(jt / kStages) & 1u,
                                    abort_flag)))
            break;
          tc_fence_after_sync();
          for (int t = 0; t < kQTiles; ++t) issue_s(t, s0);
          mma_commit_elect(bar(kBarKEmpty + s0));
          if (n_tiles == 1) mma_commit_elect(bar(kBarQFree));
        }
        for (int j = 0; ok && j < n_tiles; ++j) {
          const int g0 = jt + j;  // global tile of this step
          const int sv = g0 % kStages;
          uint32_t dv = static_cast<uint32_t>(desc_advance(dv0, sv * kTileBytes));
          opaque(dv);
          const bool more = j + 1 < n_tiles;
          const int sk = (g0 + 1) % kStages;
          if (!(ok = mbar_wait_warp(bar(kBarVFull + sv), static_cast<uint32_t>(g0 / kStages) & 1u,
                                    abort_flag)))
            break;
          // unrolled: the issuer's own instructions are on the pipe's critical
          // path (its loop overhead cost ~2% when this loop was kept rolled)
#pragma unroll
          for (int t = 0; t < kQTiles; ++t) {
            if (!(ok = mbar_wait_warp(bar(kBarPFull + t), static_cast<uint32_t>(g0) & 1u, abort_flag)))
              break;
            // the previous item's epilogue has read O_t before it is overwritten
            if (j == 0 && k > 0 &&
                !(ok = mbar_wait_warp(bar(kBarOFree + t), static_cast<uint32_t>(k - 1) & 1u,
                                      abort_flag)))
              break;
            tc_fence_after_sync();
            if (FLUX_DBG(t >= 0 && t < kQTiles && sv >= 0 && sv < kStages, kDbgMmaPV)) {
#pragma unroll
              for (int kk = 0; kk < kBN / 16; ++kk)
                mma_ts_elect(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, dv + ((kk * 2048) >> 4),
                             desc_hi, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit_elect(bar(kBarODone + t));
            if (t == kQTiles - 1) mma_commit_elect(bar(kBarVEmpty + sv));
            if (more) {
              if (t == 0 &&
                  !(ok = mbar_wait_warp(bar(kBarKFull + sk),
                                        static_cast<uint32_t>((g0 + 1) / kStages) & 1u, abort_flag)))
                break;
              tc_fence_after_sync();
              issue_s(t, sk);
              if (t == kQTiles - 1) {
                mma_commit_elect(bar(kBarKEmpty + sk));
                if (j + 2 == n_tiles) mma_commit_elect(bar(kBarQFree));  // last S of the item
              }
            }
          }
        }
        jt += n_tiles;
      }
      // drain: every MMA issued above has finished before TMEM is released
      mma_commit_elect(bar(kBarDrain));
      const long long t0 = clock64();
      while (!mbar_try_wait(bar(kBarDrain), 0) && clock64() - t0 < kWaitBudgetCycles) {
      }
      __syncwarp();
    }
  } else if (warp < 12) {
    // ---------------------------------------------------------- softmax
    reg_inc<kRegsSoftmax>();
    const int t = (warp - 4) >> 2;  // Q tile
    const int wq = warp & 3;        // TMEM lane quadrant
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + t * 128 + lane_off;
    const uint32_t tO = tmem + 256 + t * 128 + lane_off;
    const float scale_log2 = 1.4426950408889634f * 0.08838834764831845f;
    bool ok = true;
    int jt = 0;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const Item it = info(item);
      const int b = it.b, h = it.h, n_tiles = it.n_tiles;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_tiles; ++j, ++jt) {
        if (!(ok = mbar_wait_warp(bar(kBarSFull + t), static_cast<uint32_t>(jt) & 1u, abort_flag))) break;
        tc_fence_after_sync();
        uint32_t sr[kBN];
        float mr[kBN / 32];
        if (!FLUX_DBG(in_tmem(tS, kBN, t * 128, t * 128 + 128), kDbgSLoad)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
          tmem_ld32_max(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]), mr[c]);
        tmem_ld_wait();
        const int valid = tile_keys(it, tile_at(it, j));
        float mx = fmax3(mr[0], mr[1], fmaxf(mr[2], mr[3]));
        if (valid < kBN) {
#pragma unroll
          for (int i = 0; i < kBN; ++i)
            if (i >= valid) sr[i] = __float_as_uint(-INFINITY);
          // row max: four independent chains of 3-input max
          float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
#pragma unroll
          for (int i = 0; i < kBN; i += 8) {
            ma = fmax3(ma, __uint_as_float(sr[i]), __uint_as_float(sr[i + 1]));
            mb = fmax3(mb, __uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3]));
            mc = fmax3(mc, __uint_as_float(sr[i + 4]), __uint_as_float(sr[i + 5]));
            md = fmax3(md, __uint_as_float(sr[i + 6]), __uint_as_float(sr[i + 7]));
          }
          mx = fmax3(ma, mb, fmaxf(mc, md));
        }
        mx *= scale_log2;
        float alpha = 1.f;
        float m_use = m_run;
        if (j == 0) {
          m_use = mx;
        } else if (__any_sync(0xffffffffu, mx > m_run + kRescaleThreshold)) {
          m_use = fmaxf(m_run, mx);
          alpha = ex2_approx(m_run - m_use);
          // S_t(j) is complete, hence so is PV_t(j-1): O_t is stable here.
#pragma unroll 1
          for (int c = 0; c < kD / 16; ++c) {
            if (!FLUX_DBG(in_tmem(tO + c * 16, 16, 256 + t * 128, 384 + t * 128), kDbgORescale))
              continue;
            uint32_t o[16];
            tmem_ld16(tO + c * 16, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + c * 16, o);
          }
        }
        // p = 2^(s * scale - m): scale and shift on fp32 pairs, exp2 per lane,
        // row sum in four pair accumulators, P packed to bf16 in four chunks of
        // 32 keys (16 TMEM columns each) to bound registers.
        const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const uint64_t x2 =
                f2_pack(__uint_as_float(sr[c * 32 + i]), __uint_as_float(sr[c * 32 + i + 1]));
            float y0, y1;
            f2_unpack(f2_fma(x2, scale2, negm2), y0, y1);
            const float p0 = ex2_approx(y0);
            const float p1 = ex2_approx(y1);
            acc[(i >> 1) & 3] = f2_add(acc[(i >> 1) & 3], f2_pack(p0, p1));
            pk[i / 2] = pack_bf16x2(p0, p1);
          }
          if (FLUX_DBG(in_tmem(tS + c * 16, 16, t * 128, t * 128 + 64), kDbgPStore))
            tmem_st16(tS + c * 16, pk);
        }
        float sum;
        {
          float a0, a1, b0, b1;
          f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
          f2_unpack(f2_add(acc[2], acc[3]), b0, b1);
          sum = (a0 + a1) + (b0 + b1);
        }
        tmem_st_wait();
        l_run = l_run * alpha + sum;
        m_run = m_use;
        tc_fence_before_sync();
        warp_arrive(bar(kBarPFull + t), lane);
      }
      if (!ok) break;
      // epilogue: wait for the item's last P V, normalise, store bf16 rows
      if (!(ok = mbar_wait_warp(bar(kBarODone + t), static_cast<uint32_t>(jt - 1) & 1u, abort_flag))) break;
      tc_fence_after_sync();
      // Each warp stages its 32 rows, 32 channels at a time, in its own
      // 64-byte-swizzled 2 KB buffer and lane 0 stores them with one TMA copy
      // (rows past the tensor's end are not written). A box that would cross
      // the end of the item's query segment inside the tensor is written row
      // by row instead, rows of the next segment left alone.
      const float inv_l = 1.f / l_run;
      const uint32_t stage = sbase + kOffStage + static_cast<uint32_t>(warp - 4) * kStageWarpBytes;
      const int64_t row0 = it.m0 + t * kBM + wq * 32;
      const bool box_ok = row0 < it.q_hi && (row0 + 32 <= it.q_hi || it.q_hi == S_q);
      const bool row_ok = row0 + lane < it.q_hi;
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t o[32];
        if (!FLUX_DBG(in_tmem(tO + c * 32, 32, 256 + t * 128, 384 + t * 128) &&
                          in_smem(stage, kStageWarpBytes, kOffStage, 8 * kStageWarpBytes),
                      kDbgOLoad))
          continue;
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        if (lane == 0) bulk_wait_read_all();  // the previous copy has read the buffer
        __syncwarp();
        // 16-byte chunk q of row `lane` sits at chunk q ^ ((lane >> 1) & 3)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[8 * q]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
          const uint32_t sa = stage + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4);
          if (box_ok) {
            if (FLUX_DBG(in_smem(sa, 16, kOffStage + (warp - 4) * kStageWarpBytes,
                                 kStageWarpBytes),
                         kDbgStage))
              st_shared_v4(sa, w);
          } else if (row_ok &&
                     FLUX_DBG(b < B && h < H && row0 + lane >= 0 && row0 + lane < S_q,
                              kDbgOutRow)) {
            st_global_v4(outg + ((static_cast<int64_t>(b) * S_q + row0 + lane) * H + h) * kD +
                             c * 32 + q * 8,
                         w);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && box_ok &&
            FLUX_DBG(row0 >= 0 && row0 < S_q && c * 32 < kD && h < H && b < B, kDbgOutTma)) {
          tma_store_4d(&maps.out, stage, c * 32, h, static_cast<int>(row0), b);
          bulk_commit();
        }
      }
      tc_fence_before_sync();
      warp_arrive(bar(kBarOFree + t), lane);
    }
    if (lane == 0) bulk_wait_all();  // every output store is complete
  } else {
    // --------------------------------------------------------- RoPE warps
    reg_dec<kRegsRope>();
    // everything below reads the table: wait for the kernel that writes it
    // when this one was launched to overlap it (a no-op otherwise)
    grid_dep_wait();
    const int u = tid - 384;
    bool ok = true;
    int tuse = 0;   // table-buffer halves consumed so far
    int tload = 0;  // table-buffer loads issued (RoPE warp 0)
    // Table rows [row0, row0 + 64) of the Q-side or K-side table into the
    // shared buffer: RoPE warp 0 loads them once every RoPE warp is done with
    // the previous rows.
    auto load_table = [&](const CUtensorMap *tmap, int64_t row0) {
      if (u < 32) {
        if (!(ok = mbar_wait_warp(bar(kBarTEmpty), (static_cast<uint32_t>(tuse) & 1u) ^ 1u,
                                  abort_flag)))
          return;
        if (lane == 0) {
          // a tile's table rows start inside the sequence or, for the later
          // 64-row pieces of a ragged last 256-row block, up to 192 rows past
          // its end (the copy then reads zeros, as the tile itself does);
          // segment boundaries put the start anywhere
          [[maybe_unused]] const int64_t rows = tmap == &maps.table_q ? S_q : S_k;
          if (FLUX_DBG(row0 >= 0 && row0 < rows + 192 &&
                           (tmap == &maps.table_q || tmap == &maps.table_k),
                       kDbgTableLoad)) {
            mbar_arrive_expect_tx(bar(kBarTFull), kTableBytes);
            tma_load_2d(sbase + kOffT, tmap, bar(kBarTFull), 0, static_cast<int>(row0));
          } else {
            mbar_arrive(bar(kBarTFull));  // checked build: no copy, the phase completes
          }
        }
        __syncwarp();
        ++tload;
      }
    };
    // Rotates a landed tile whose first row is row tok0 of a tensor of
    // n_rows rows in place; with `grow` (K tiles when sharing) the rotated
    // rows also go to the exchange buffer. The table rows of its first half
    // were requested already.
    auto rotate_tile = [&](uint32_t tile, int64_t tok0, int64_t n_rows, uint16_t *grow,
                           const QkNorm &nm, const CUtensorMap *tmap) {
      const int rows_valid =
          static_cast<int>(n_rows - tok0 < kBN ? (n_rows - tok0 > 0 ? n_rows - tok0 : 0) : kBN);
      for (int half = 0; ok && half < 2; ++half) {
        if (!(ok = mbar_wait_warp(bar(kBarTFull), static_cast<uint32_t>(tuse) & 1u, abort_flag)))
          return;
        if (grow != nullptr)
          rotate_half<kNorm, true>(tile, sbase + kOffT, half, u, nm, tok0, rows_valid, grow,
                                   xrow_stride);
        else
          rotate_half<kNorm, false>(tile, sbase + kOffT, half, u, nm, tok0, rows_valid, nullptr, 0);
        warp_arrive(bar(kBarTEmpty), lane);
        ++tuse;
        if (half == 0) load_table(tmap, tok0 + 64);
      }
    };
    // Prepares piece c of the CTA's next item while the current one runs:
    // pieces 0-3 are its Q rows in 64-row blocks, rotated into the exchange
    // buffer; pieces 4-7 the two 64-row halves of its first two K tiles,
    // rotated into the exchange buffer and published (a tile someone already
    // published is rewritten with the same bytes). After the last piece each
    // warp arrives on Q-prep, after which the producer loads the Q rows and
    // the two K tiles without reading flags. Small pieces keep raw K tiles
    // from waiting long behind this work.
    auto prepare_piece = [&](int next, int c) {
      const Item nx = info(next);
      const int kt = (c - 4) >> 1;  // K tile (0 or 1) of pieces 4-7 (none if pre-rotated)
      if (c < 4 || (kt < nx.n_tiles && tile_at(nx, kt) < nx.n_main)) {
        int64_t tok0, n_rows;
        const uint16_t *src;
        uint16_t *dst;
        const uint32_t *tab;
        if (c < 4) {
          tok0 = nx.m0 + c * 64;
          n_rows = S_q;
          src = qg + ((static_cast<int64_t>(nx.b) * S_q + tok0) * H + nx.h) * kD;
          dst = qrot + ((static_cast<int64_t>(nx.b) * S_q + tok0) * Hl + nx.hx) * kD;
          tab = tabq;
        } else {
          tok0 = tile_row(nx, tile_at(nx, kt)) + ((c - 4) & 1) * 64;
          n_rows = S_k;
          src = kg + ((static_cast<int64_t>(nx.b) * S_k + tok0) * H + nx.h) * kD;
          dst = krot + ((static_cast<int64_t>(nx.b) * S_k + tok0) * Hl + nx.hx) * kD;
          tab = tabk;
        }
        const int nrows = static_cast<int>(n_rows - tok0 < 64 ? (n_rows - tok0 > 0 ? n_rows - tok0 : 0) : 64);
        // rows tok0 .. tok0 + nrows - 1 of head h (inputs) / hx (exchange buffer) of batch b
        const bool prep_ok = FLUX_DBG(
            tok0 >= 0 && (nrows == 0 || tok0 + nrows <= n_rows) && nx.b < B && nx.h < H &&
                nx.hx < Hl &&
                (c < 4 || nx.flags - kflags + static_cast<int64_t>(tile_at(nx, kt)) * 4 + 4 <=
                              n_flag_words),
            kDbgPrepare);
        if (nrows > 0 && prep_ok)
          rotate_rows_global<kNorm>(src, dst, tab + tok0 * kPairs, nrows, row_stride, xrow_stride,
                                    u, c < 4 ? qn : kn, tok0);
        fence_proxy_async_global();  // read by TMA copies
        if (c >= 4 && ((c - 4) & 1) == 1 && prep_ok) {
          // publish as the in-place path does: this warp's rows, then its flag
          fence_acq_rel_gpu();
          __syncwarp();
          if (lane == 0) {
            fence_acq_rel_gpu();
            st_relaxed_gpu_u64(nx.flags + static_cast<int64_t>(tile_at(nx, kt)) * 4 + (u >> 5),
                               token);
          }
        }
      }
      if (c == kPrepChunks - 1) warp_arrive(bar(kBarQPrep), lane);
    };
    // Work comes from the producer's queue in issue order; every rotation
    // step, the table ring and each wait are this warp's alone (one arrival
    // per warp on the hand-off barriers), so the warps never wait on each
    // other.
    for (int qi = 0; ok; ++qi) {
      const int e = qi % kRopeQ;
      if (!(ok = mbar_wait_warp(bar(kBarRQFull + e), static_cast<uint32_t>(qi / kRopeQ) & 1u,
                                abort_flag)))
        break;
      uint32_t x, y;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(sbase + kOffRQ + 8 * e)
                   : "memory");
      warp_arrive(bar(kBarRQEmpty + e), lane);  // the slot may be reused
      const uint32_t kind = x & 15u;
      if (kind == kRqEnd) break;
      const int item = static_cast<int>(y);
      if (!FLUX_DBG(kind >= kRqQ && kind <= kRqPrep && item >= 0 && item < n_items &&
                        (kind != kRqPrep || ((x >> 4) & 15u) < static_cast<uint32_t>(kPrepChunks)) &&
                        (kind != kRqK || (((x >> 4) & 15u) < static_cast<uint32_t>(kStages) &&
                                          static_cast<int>(x >> 9) < info(item).n_tiles)),
                    kDbgQueue)) {
        ok = false;
        break;
      }
      if (kind == kRqPrep) {
        prepare_piece(item, static_cast<int>((x >> 4) & 15u));
        continue;
      }
      const uint32_t par = (x >> 8) & 1u;
      const Item it = info(item);
      if (kind == kRqQ) {
        load_table(&maps.table_q, it.m0);
        if (!ok) break;
        if (!(ok = mbar_wait_warp(bar(kBarQRaw), par, abort_flag))) break;
        for (int t = 0; ok && t < kQTiles; ++t) {
          if (t > 0) load_table(&maps.table_q, it.m0 + t * kBM);
          (void)FLUX_DBG(it.m0 >= 0 && it.m0 < S_q, kDbgQRotate);  // rotation stays in smem
          rotate_tile(sbase + kOffQ + t * kTileBytes, it.m0 + t * kBM, S_q, nullptr, qn,
                      &maps.table_q);
        }
        if (!ok) break;
        fence_proxy_async_smem();
        warp_arrive(bar(kBarQFull), lane);
        continue;
      }
      // kind == kRqK: a raw K tile in stage s
      const int s = static_cast<int>((x >> 4) & 15u);
      const int tj = static_cast<int>(x >> 9);
      const int64_t tok0 = tile_row(it, tj);
      load_table(&maps.table_k, tok0);  // in flight while the tile itself lands
      if (!ok) break;
      if (!(ok = mbar_wait_warp(bar(kBarKRaw + s), par, abort_flag))) break;
      // publication: rows tok0 .. of head hx in the exchange buffer and this
      // warp's flag of tile tj
      const bool pub_ok = FLUX_DBG(
          tok0 >= 0 && tok0 < S_k && it.b < B && it.hx < Hl && s < kStages &&
              (!share || it.flags - kflags + static_cast<int64_t>(tj) * 4 + 4 <= n_flag_words),
          kDbgKRotate);
      uint16_t *grow = share && pub_ok
                           ? krot + ((static_cast<int64_t>(it.b) * S_k + tok0) * Hl + it.hx) * kD
                           : nullptr;
      rotate_tile(sbase + kOffK + s * kTileBytes, tok0, S_k, grow, kn, &maps.table_k);
      if (!ok) break;
      fence_proxy_async_smem();
      if (share && pub_ok) {
        // publish this warp's rows of tile tj: each lane's stores, then
        // one flag per warp (release)
        fence_proxy_async_global();
        fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0) {
          fence_acq_rel_gpu();
          st_relaxed_gpu_u64(it.flags + static_cast<int64_t>(tj) * 4 + (u >> 5), token);
        }
      }
      warp_arrive(bar(kBarKFull + s), lane);
    }
    // a table copy still in flight after an abort lands before the CTA exits
    if (u < 32 && tload > tuse) drain_wait(bar(kBarTFull), static_cast<uint32_t>(tload - 1) & 1u);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0 && *abort_flag) {
    grid_dep_wait();  // after the table kernel's clear of the same word
    atomicExch(status, FLUX_ERR_DEVICE_TIMEOUT);
  }
#ifdef FLUX_DEBUG
  if (tid == 0) {  // a failed check outranks the timeout it may have caused
    const int site = atomicAdd(&g_dbg_site, 0);
    if (site != 0) {
      grid_dep_wait();
      atomicExch(status, FLUX_DEBUG_STATUS_BASE - site);
    }
  }
#endif
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// q, k, v or out as a 4-D tensor (D, H, S, B); one box = box_ch channels x
// box_rows tokens of one head, swizzled 128 bytes (64-channel boxes) or 64
// bytes (32-channel boxes); out-of-range tokens read as zeros and are not
// written.
bool make_head_map(CUtensorMap *map, const void *x, int B, int64_t S, int H,
                   uint32_t box_rows = kBN, uint32_t box_ch = 64) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * 2,
                                 static_cast<cuuint64_t>(H) * kD * 2,
                                 static_cast<cuuint64_t>(S) * H * kD * 2};
  const cuuint32_t box[4] = {box_ch, 1, box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(x), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_ch == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The packed table [S, 64] uint32 as a 2-D tensor; one box = 64 tokens.
bool make_table_map(CUtensorMap *map, const uint32_t *table, int64_t S) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kPairs), static_cast<cuuint64_t>(S)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kPairs) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kPairs), kTableRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t *>(table), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// A value no earlier launch in this process used, for the exchange flags: a
// flag equal to it was written during this launch. The counter is mixed
// (splitmix64 finaliser) with a per-process salt so that stale flag words
// left in reused memory, by this or another process, match with
// probability about 2^-64.
uint64_t next_launch_token() {
  static std::atomic<uint64_t> counter{0};
  static const uint64_t salt = [] {
    std::random_device rd;
    return (static_cast<uint64_t>(rd()) << 32) ^ rd() ^
           static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
  }();
  uint64_t z = salt + 0x9E3779B97F4A7C15ull * (counter.fetch_add(1) + 1);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z == 0 ? 1 : z;
}

size_t exchange_bytes(int B, int64_t S_q, int64_t S_k, int H, const AttnSegment *segs,
                      int n_segs) {
  size_t flags = 0;
  for (int r = 0; r < kMaxSegments; ++r)
    for (int g = 0; g < n_segs; ++g)
      if (segs[g].key_range == r) {  // the first segment of each key range sizes its flags
        flags += static_cast<size_t>(B) * H * ((segs[g].k_hi - segs[g].k_lo + kBN - 1) / kBN) * 4;
        break;
      }
  flags = (flags * sizeof(uint64_t) + 255) & ~static_cast<size_t>(255);
  return flags + (static_cast<size_t>(B) * static_cast<size_t>(S_k) * H * kD +
                  static_cast<size_t>(B) * static_cast<size_t>(S_q) * H * kD) * 2;
}

cudaError_t launch_attention_segments(const void *q, const void *k, const void *v, void *out,
                                      const uint32_t *table_q, const uint32_t *table_k,
                                      int *status, int B, int64_t S_q, int64_t S_k, int H,
                                      const AttnSegment *segs, int n_segs,
                                      const PreRotatedKV *pre, void *xbuf,
                                      const QkNormArgs *norm, cudaStream_t stream, bool pdl,
                                      int h0, int Hl) {
  if (n_segs < 1 || n_segs > kMaxSegments) return cudaErrorInvalidValue;
  if (Hl == 0) Hl = H;
  if (h0 < 0 || Hl < 1 || h0 > H - Hl) return cudaErrorInvalidValue;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev], [&] {
    attr_err = cudaFuncSetAttribute(joint_rope_attention_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBytes));
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(joint_rope_attention_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kSmemBytes));
  });
  if (attr_err != cudaSuccess) return attr_err;
  Maps maps;
  if (!make_head_map(&maps.q, q, B, S_q, H) || !make_head_map(&maps.k, k, B, S_k, H) ||
      !make_head_map(&maps.v, v, B, S_k, H) || !make_head_map(&maps.out, out, B, S_q, H, 32, 32) ||
      !make_table_map(&maps.table_q, table_q, S_q) || !make_table_map(&maps.table_k, table_k, S_k))
    return cudaErrorInvalidValue;
  const int64_t S_pre = pre != nullptr ? pre->S : 0;
  if (S_pre < 0 || (S_pre > 0 && (pre->k == nullptr || pre->v == nullptr)))
    return cudaErrorInvalidValue;
  if (S_pre > 0) {
    if (!make_head_map(&maps.kpre, pre->k, B, S_pre, H) ||
        !make_head_map(&maps.vpre, pre->v, B, S_pre, H))
      return cudaErrorInvalidValue;
  } else {
    maps.kpre = maps.k;  // never read
    maps.vpre = maps.v;
  }
  // segments, their items and their key ranges' flag offsets
  Segs sg{};
  sg.n = n_segs;
  int64_t items = 0;
  int64_t range_off[kMaxSegments];
  int64_t off = 0;
  for (int r = 0; r < kMaxSegments; ++r) {
    range_off[r] = -1;
    for (int g = 0; g < n_segs; ++g)
      if (segs[g].key_range == r) {
        range_off[r] = off;
        off += static_cast<int64_t>(B) * Hl * ((segs[g].k_hi - segs[g].k_lo + kBN - 1) / kBN) * 4;
        break;
      }
  }
  for (int g = 0; g < n_segs; ++g) {
    const AttnSegment &a = segs[g];
    if (a.q_lo < 0 || a.q_hi > S_q || a.k_lo < 0 || a.k_hi > S_k || a.k_hi <= a.k_lo ||
        a.key_range < 0 || a.key_range >= kMaxSegments || a.n_pre < 0 || a.n_pre > S_pre)
      return cudaErrorInvalidValue;
    sg.first_item[g] = static_cast<int>(items);
    sg.q_lo[g] = a.q_lo;
    sg.q_hi[g] = a.q_hi;
    sg.k_lo[g] = a.k_lo;
    sg.k_hi[g] = a.k_hi;
    sg.n_rb[g] = static_cast<int>((a.q_hi - a.q_lo + kRowsPerCta - 1) / kRowsPerCta);
    sg.n_main[g] = static_cast<int>((a.k_hi - a.k_lo + kBN - 1) / kBN);
    sg.n_pre[g] = a.n_pre;
    sg.n_tiles[g] = sg.n_main[g] + static_cast<int>((a.n_pre + kBN - 1) / kBN);
    sg.flag_off[g] = range_off[a.key_range];
    items += static_cast<int64_t>(B) * Hl * (a.q_hi > a.q_lo ? sg.n_rb[g] : 0);
    if (items > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  }
  sg.first_item[n_segs] = static_cast<int>(items);
  if (items == 0) return cudaSuccess;
  uint64_t *kflags = nullptr;
  uint16_t *krot = nullptr, *qrot = nullptr;
  if (xbuf != nullptr) {
    const size_t flags = (static_cast<size_t>(off) * sizeof(uint64_t) + 255) & ~static_cast<size_t>(255);
    kflags = static_cast<uint64_t *>(xbuf);
    krot = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(xbuf) + flags);
    qrot = krot + static_cast<size_t>(B) * static_cast<size_t>(S_k) * Hl * kD;
    if (!make_head_map(&maps.krot, krot, B, S_k, Hl) || !make_head_map(&maps.qrot, qrot, B, S_q, Hl))
      return cudaErrorInvalidValue;
  } else {
    maps.krot = maps.k;  // never read
    maps.qrot = maps.q;
  }
  // persistent: one CTA per SM, work items handed out round robin
  const int sms = sm_count_current_device();
  if (sms == 0) return cudaErrorUnknown;
  const unsigned grid = static_cast<unsigned>(items < sms ? items : sms);
  const uint16_t *qg = static_cast<const uint16_t *>(q), *kg = static_cast<const uint16_t *>(k);
  uint16_t *og = static_cast<uint16_t *>(out);
#ifdef FLUX_DEBUG
  {  // checked build: clear the first-failure record; no overlap with the table kernel
    void *site = nullptr;
    e = cudaGetSymbolAddress(&site, g_dbg_site);
    if (e == cudaSuccess) e = cudaMemsetAsync(site, 0, sizeof(int), stream);
    if (e != cudaSuccess) return e;
    pdl = false;
  }
#endif
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const int n_items = static_cast<int>(items);
  const int64_t n_flag_words = xbuf != nullptr ? off : 0;
  const uint64_t token = next_launch_token();
  if (norm != nullptr) {
    const QkNorm qn{norm->q_txt, norm->q_img, norm->s_txt, norm->eps};
    const QkNorm kn{norm->k_txt, norm->k_img, norm->s_txt, norm->eps};
    e = cudaLaunchKernelEx(&cfg, joint_rope_attention_kernel<true>, maps, og, status, sg, B, S_q,
                           S_k, H, h0, Hl, n_items, n_flag_words, kflags, krot, qrot, qg, kg,
                           table_q, table_k, token, qn, kn);
  } else {
    const QkNorm none{nullptr, nullptr, 0, 0.f};
    e = cudaLaunchKernelEx(&cfg, joint_rope_attention_kernel<false>, maps, og, status, sg, B,
                           S_q, S_k, H, h0, Hl, n_items, n_flag_words, kflags, krot, qrot, qg, kg,
                           table_q, table_k, token, none, none);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_joint_attention(const void *q, const void *k, const void *v, void *out,
                                   const uint32_t *table, int *status, int B, int64_t S, int H,
                                   void *krot_scratch, const QkNormArgs *norm,
                                   cudaStream_t stream, bool pdl, int h0, int Hl) {
  const AttnSegment all{0, S, 0, S, 0, 0};
  return launch_attention_segments(q, k, v, out, table, table, status, B, S, S, H, &all, 1,
                                   nullptr, krot_scratch, norm, stream, pdl, h0, Hl);
}

}  // namespace flux
