// lce.cu -- fused linear cross-entropy: per-token NLL, log-sum-exp and target
// logit of z = H W^T without storing the (N, V) logits, and the backward into
// the hidden states and the head (mlx-train-perf 0.5.1 README, "The fused
// cross-entropy loss": the backward recomputes the tiles it needs instead of
// reading a stored logit matrix).
//
// Forward:
// Grid: (token tiles of 128) x (vocabulary splits). A CTA walks its split's
// vocabulary tiles of 256 rows; for each, the tcgen05 tensor cores form the
// 128 x 256 logit tile in TMEM from 64-wide K slices of H and W that TMA
// streams through a 4-stage ring (one CTA per SM), and four epilogue warps
// (one thread per token, reading its TMEM lane) fold the tile into a running
// maximum and sum of exponentials and pick up the target logit when it falls
// in the tile.
// Two TMEM accumulators let the next tile's products run while the epilogue
// reads the previous one. Each CTA writes its split's (max, sum) per token
// and, for tokens whose target lies in its split, the target logit; a merge
// kernel combines the splits.
//
// Roles: warp 0 lane 0 loads (TMA), warp 1 issues the MMAs (lane 0) and owns
// the TMEM allocation, warps 4..7 are the epilogue (warp % 4 = TMEM lane
// quarter). Every wait is bounded (sm103.cuh).
//
// Backward, over the vocabulary in chunks of Vc rows (so that nothing of size
// N x V is ever held): the same kernel, with an epilogue that turns each
// recomputed logit tile into dz = g (exp(z - lse) - [v == target]) in bf16
// and writes it twice, as dz (tokens x Vc) and dz^T (Vc x tokens); then two
// tcgen05 GEMMs, dW[chunk] = dz^T H (written once per chunk) and
// dH += dz W[chunk] (fp32 in the workspace across chunks, in chunk order, so
// the result does not depend on timing; the last chunk writes bf16 dH).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/pa.h"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {
namespace {

// The logit tiles are 128 tokens x 256 vocabulary rows, so every product is
// an N = 256 MMA: those keep the tensor pipe at its full rate while the
// epilogue warps' arithmetic shares the issuing warp's SM sub-partition,
// where N = 128 products fall to about 84 of their 64 cycles.
constexpr int kLceStages = 4;                  // 4 x 48 KB: one CTA per SM
constexpr int kLceTile = 128;                  // tokens per CTA
constexpr int kLceVTile = 256;                 // vocabulary rows per tile
constexpr uint32_t kLceSlice = 128 * 128;      // one 128 x 64 bf16 slice of H (128-byte rows), 16 KB
constexpr uint32_t kLceSliceW = 256 * 128;     // one 256 x 64 bf16 slice of W, 32 KB
constexpr uint32_t kLceStage = kLceSlice + kLceSliceW;
constexpr int kLceThreads = 256;
constexpr uint32_t kLceTmemCols = 512;  // two 256-column fp32 accumulators

struct LceMisc {
  uint64_t full[kLceStages], empty[kLceStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr uint32_t kLceSmem = 1024 /* misc */ + 1024 /* alignment */ + kLceStages * kLceStage;

struct LceParams {
  int N, V, D;
  int vt_per_split;  // vocabulary tiles per split
  const int32_t* targets;
  float* part_m;  // (splits, N): running maximum of the split
  float* part_s;  // (splits, N): sum of exp(z - max) over the split
  float* part_t;  // (splits, N): the target logit, written by the split holding it
  uint32_t* status;
  // backward: vocabulary tiles from vt_base on (one chunk), and dz for them
  int vt_base, vt_end;        // the chunk's vocabulary tiles: vt_base <= vt < vt_end
  const float* lse;           // (N) from the forward
  const float* g;             // (N) upstream gradient dL/dnll
  __nv_bfloat16* dz;          // (N, ld_dz): column v - vt_base * 128
  int ld_dz;
  __nv_bfloat16* dzt;         // (Vc, ld_dzt): row v - vt_base * 128, or null (no dW)
  int ld_dzt;
};

// Token tiles per group of the backward's pair order. The CTAs resident at
// once (one per SM) cover about kLceGroup token tiles of H and
// 152 / kLceGroup vocabulary tiles of W, and a group's H stays in L2 while
// the group walks every vocabulary tile of the chunk. Measured on the
// N = 8192, V = 151,936, D = 4096 backward: 22.15 ms with one token tile
// per group (vocabulary tile fastest), 21.41 / 21.18 / 21.03 / 21.22 /
// 21.74 ms with 8 / 16 / 32 / 48 / 64.
#ifndef PA_LCE_DZ_GROUP
#define PA_LCE_DZ_GROUP 32
#endif
constexpr int kLceGroup = PA_LCE_DZ_GROUP;

// BWD = false: the forward's online log-sum-exp epilogue; the CTA walks the
// vocabulary tiles of split blockIdx.y for token tile blockIdx.x. BWD =
// true: the backward's dz epilogue, which keeps nothing from tile to tile,
// so one CTA per SM takes the chunk's (token tile, vocabulary tile) pairs
// blockIdx.x, blockIdx.x + gridDim.x, ...: pairs run in groups of kLceGroup
// token tiles, token tile fastest inside a group.
template <bool BWD>
__global__ void __launch_bounds__(kLceThreads, 1)
    lce_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW,
               const LceParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  LceMisc& m = *reinterpret_cast<LceMisc*>(smem_raw);
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1024 + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sRing = smem_u32(ring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int VTc = BWD ? p.vt_end - p.vt_base : 0;  // the backward chunk's vocabulary tiles
  int vt0 = 0, nt;                                  // nt >= 1 by construction of the grid
  if (BWD) {
    const int pairs = ((p.N + kLceTile - 1) / kLceTile) * VTc;
    nt = (pairs - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  } else {
    const int VT = (p.V + kLceVTile - 1) / kLceVTile;
    vt0 = blockIdx.y * p.vt_per_split;
    nt = min(vt0 + p.vt_per_split, VT) - vt0;
  }
  // token tile and vocabulary tile of this CTA's tile j (the backward's pair
  // q: group gi of token tiles g0 .. g0 + gs - 1, then its index r inside)
  const int TMc = (p.N + kLceTile - 1) / kLceTile;
  const int VTg = BWD ? VTc : 1;  // the forward never takes pairs
  const auto pair_of = [&](int j) -> int2 {
    const int q = (int)blockIdx.x + j * (int)gridDim.x;
    const int gi = q / (kLceGroup * VTg), r = q - gi * kLceGroup * VTg;
    const int g0 = gi * kLceGroup, gs = min(kLceGroup, TMc - g0);
    return make_int2(g0 + r % gs, p.vt_base + r / gs);
  };
  const auto tile_tm = [&](int j) { return BWD ? pair_of(j).x : (int)blockIdx.x; };
  const auto tile_vt = [&](int j) { return BWD ? pair_of(j).y : vt0 + j; };
  const int KS = p.D / 64;   // K slices per tile
  const Guard g{&m.abort_flag, p.status};

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    for (int s = 0; s < kLceStages; ++s) {
      mbar_init(&m.full[s], 1);
      mbar_init(&m.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&m.acc_full[b], 1);
      mbar_init(&m.acc_empty[b], 128);
    }
    mbar_init(&m.fin, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&m.tmem_base, kLceTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      prefetch_tmap(&tmH);
      prefetch_tmap(&tmW);
      int it = 0;
      bool ok = true;
      for (int j = 0; ok && j < nt; ++j) {
        for (int kc = 0; kc < KS; ++kc, ++it) {
          const int st = it % kLceStages;
          if (!g.wait(&m.empty[st], ((it / kLceStages) & 1) ^ 1, 40)) { ok = false; break; }
          mbar_expect_tx(&m.full[st], kLceStage);
          tma_load_2d(ring + st * kLceStage, &tmH, &m.full[st], kc * 64, tile_tm(j) * kLceTile);
          tma_load_2d(ring + st * kLceStage + kLceSlice, &tmW, &m.full[st], kc * 64, tile_vt(j) * kLceVTile);
        }
      }
      // no copy may still be landing when the CTA exits
      for (int i = (it > kLceStages ? it - kLceStages : 0); i < it; ++i)
        g.drain(&m.full[i % kLceStages], (i / kLceStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = lane == 0;
    constexpr uint32_t idZ = idesc_bf16_f32(128, 256, false, false);
    bool ok = true;
    int it = 0;
    for (int j = 0; ok && j < nt; ++j) {
      const int buf = j & 1;
      // accumulator buf is free once the epilogue has read tile j - 2 from it
      if (j >= 2 && !g.wait_warp(&m.acc_empty[buf], ((j - 2) >> 1) & 1, 41)) { ok = false; break; }
      tc_fence_after();
      for (int kc = 0; kc < KS; ++kc, ++it) {
        const int st = it % kLceStages;
        if (!g.wait_warp(&m.full[st], (it / kLceStages) & 1, 42)) { ok = false; break; }
        tc_fence_after();
        const uint64_t hd = sdesc_sw128(sRing + st * kLceStage, 16, 1024);
        const uint64_t wd = sdesc_sw128(sRing + st * kLceStage + kLceSlice, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (leader)
            umma_bf16(tmem + buf * 256, sdesc_add(hd, kk * 32), sdesc_add(wd, kk * 32), idZ,
                      (kc > 0 || kk > 0) ? 1u : 0u);
        if (leader) umma_commit(&m.empty[st]);
        __syncwarp();
      }
      if (ok && leader) umma_commit(&m.acc_full[buf]);
      __syncwarp();
    }
    if (leader) {
      umma_commit(&m.fin);  // every MMA issued has completed once this arrives
      g.drain(&m.fin, 0);
    }
    __syncwarp();
  } else if (warp >= 4 && BWD) {
    // ------------------------------------------------------------ dz epilogue
    // Thread r owns token row r of the tile: dz = g (2^(z log2e - lse log2e)
    // - [v == target]) for every vocabulary column, zero for an ignored
    // target (outside [0, V)). dz goes out in the token's row (16-byte
    // stores) and, when the head trains, in dz^T, where the 32 lanes of a
    // warp write 32 consecutive tokens of one vocabulary row.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int buf = j & 1;
      const int token = tile_tm(j) * kLceTile + r;
      const bool live = token < p.N;
      const int t = live ? p.targets[token] : -1;
      const bool use = live && t >= 0 && t < p.V;
      const float gl = use ? p.g[token] : 0.f;
      const float l2 = use ? p.lse[token] * 1.4426950408889634f : 0.f;
      ok = g.wait(&m.acc_full[buf], (j >> 1) & 1, 44);
      ok = __all_sync(~0u, ok);
      if (!ok) break;
      tc_fence_after();
      const int v0 = tile_vt(j) * kLceVTile;
      const int c0v = v0 - p.vt_base * kLceVTile;  // column of v0 in the chunk
#pragma unroll 1
      for (int c0 = 0; c0 < kLceVTile; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + buf * 256 + c0, a);
        const int vc = v0 + c0;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          // columns past V (the last tile's tail) are exactly zero
          const float d0 = (use && vc + i < p.V)
                               ? gl * (ex2(fmaf(__uint_as_float(a[i]), 1.4426950408889634f, -l2)) -
                                       (vc + i == t ? 1.f : 0.f))
                               : 0.f;
          const float d1 = (use && vc + i + 1 < p.V)
                               ? gl * (ex2(fmaf(__uint_as_float(a[i + 1]), 1.4426950408889634f, -l2)) -
                                       (vc + i + 1 == t ? 1.f : 0.f))
                               : 0.f;
          w[i >> 1] = pack_bf16x2(d0, d1);
        }
        if (live) {
          // the tile's columns past V are not part of the chunk's output
          __nv_bfloat16* row = p.dz + (size_t)token * p.ld_dz + c0v + c0;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (vc + 8 * u < p.V)
              *reinterpret_cast<uint4*>(row + 8 * u) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          if (p.dzt) {
            __nv_bfloat16* col = p.dzt + (size_t)(c0v + c0) * p.ld_dzt + token;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (vc + i < p.V)
                col[(size_t)i * p.ld_dzt] = __ushort_as_bfloat16((unsigned short)(i & 1 ? w[i >> 1] >> 16 : w[i >> 1] & 0xFFFFu));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&m.acc_empty[buf]);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int token = (int)blockIdx.x * kLceTile + r;
    const int t = token < p.N ? p.targets[token] : -1;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    float m_run = -INFINITY, s_run = 0.f, tgt = 0.f;
    bool have_t = false;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int buf = j & 1;
      ok = g.wait(&m.acc_full[buf], (j >> 1) & 1, 43);
      ok = __all_sync(~0u, ok);
      if (!ok) break;
      tc_fence_after();
      const int v0 = tile_vt(j) * kLceVTile;
#pragma unroll 1
      for (int c0 = 0; c0 < kLceVTile; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + buf * 256 + c0, a);
        const int vc = v0 + c0;
        float cmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (vc + i < p.V) cmax = fmaxf(cmax, __uint_as_float(a[i]));
        if (cmax > -INFINITY) {
          const float m_new = fmaxf(m_run, cmax);
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (vc + i < p.V) acc += expf(__uint_as_float(a[i]) - m_new);
          s_run = s_run * expf(m_run - m_new) + acc;
          m_run = m_new;
        }
        if (t >= vc && t < vc + 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (t == vc + i) tgt = __uint_as_float(a[i]);
          have_t = true;
        }
      }
      tc_fence_before();
      mbar_arrive(&m.acc_empty[buf]);
    }
    if (ok && token < p.N) {
      const size_t o = (size_t)blockIdx.y * p.N + token;
      p.part_m[o] = m_run;
      p.part_s[o] = s_run;
      if (have_t) p.part_t[o] = tgt;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kLceTmemCols);
  }
}

// One thread per token: combine the splits' (max, sum) pairs and look up the
// target logit in the split that holds the target.
__global__ void __launch_bounds__(256) lce_merge_kernel(const LceParams p, int splits, float* __restrict__ nll,
                                                        float* __restrict__ lse, float* __restrict__ tgt_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= p.N) return;
  float M = -INFINITY;
  for (int y = 0; y < splits; ++y) M = fmaxf(M, p.part_m[(size_t)y * p.N + i]);
  float S = 0.f;
  for (int y = 0; y < splits; ++y) {
    const float my = p.part_m[(size_t)y * p.N + i];
    if (my > -INFINITY) S += p.part_s[(size_t)y * p.N + i] * expf(my - M);
  }
  const float l = M + logf(S);
  const int t = p.targets[i];
  float z = 0.f, n = 0.f;
  if (t >= 0 && t < p.V) {
    z = p.part_t[(size_t)(t / kLceVTile / p.vt_per_split) * p.N + i];
    n = l - z;
  }
  lse[i] = l;
  tgt_out[i] = z;
  nll[i] = n;
}

// ------------------------------------------------------------------ GEMM
// C (M x N) from A (M x K, K contiguous) and B (K x N, N contiguous) in
// 128 x 256 output tiles (N = 256 products, which keep their full rate beside
// the epilogue warps' arithmetic). One CTA per SM walks tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... in groups of kGemmGroup row blocks (M tiles
// fastest inside a group, so a group's A panels stay in L2 while it walks
// every N tile), K in steps of 64 through a
// 4-stage TMA ring (A as one 128-row x 64 box, B as four 64-row x 64 boxes,
// all 128-byte swizzled; elements past M, N or K read as zero), tcgen05
// products into two 256-column fp32 TMEM accumulators used by alternate
// tiles, so a tile's epilogue runs beside the next tile's products. The
// epilogue (one thread per output row) stores bf16, or starts / adds to /
// finishes an fp32 accumulator in global memory; each output tile belongs to
// one CTA, so no two threads touch the same element.
constexpr int kGemmStages = 4;
constexpr int kGemmN = 256;                               // output columns per tile
constexpr uint32_t kGemmA = 128 * 128;                    // 128 rows x 64 K, 16 KB
constexpr uint32_t kGemmBHalf = 64 * 128;                 // 64 K rows x 64 N columns, 8 KB
constexpr uint32_t kGemmStage = kGemmA + 4 * kGemmBHalf;  // 48 KB
constexpr int kGemmThreads = 192;
constexpr uint32_t kGemmSmem = 1024 /* misc */ + 1024 /* alignment */ + kGemmStages * kGemmStage;

// Row blocks per group of the tile order. Measured on the N = 8192,
// V = 151,936, D = 4096 backward (38 launches a call), in one run: 20.95,
// 21.01, 20.62 and 20.99 ms with 1 (N tiles fastest), 8, 16 and 32, and
// 21.17 ms with 16 on another box, as with 1 there: the order makes no
// difference beyond the spread between runs. With N tiles fastest a launch
// of 8192 x 4096 x 8192 read 0.60 GB from DRAM against 0.19 GB of operands
// and kept the tensor pipe 78% busy.
#ifndef PA_LCE_GEMM_GROUP
#define PA_LCE_GEMM_GROUP 16
#endif
constexpr int kGemmGroup = PA_LCE_GEMM_GROUP;

enum GemmMode : int { kStoreBf16 = 0, kAccInit = 1, kAccAdd = 2, kAccFinal = 3 };

struct GemmParams {
  int M, N, K;         // N a multiple of 64
  int mode;            // GemmMode
  int m_tiles;         // row blocks of 128
  int n_tiles;         // N tiles of kGemmN per row block
  int tiles;           // M tiles x N tiles
  __nv_bfloat16* c;    // bf16 result (kStoreBf16: the product; kAccFinal: accumulator + product)
  int ldc;
  float* acc;          // fp32 accumulator (kAccInit: set; kAccAdd: add; kAccFinal: read)
  int ldacc;
  uint32_t* status;
};

struct GemmMisc {
  uint64_t full[kGemmStages], empty[kGemmStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin;
  uint32_t tmem_base;
  int abort_flag;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    lce_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  GemmMisc& m = *reinterpret_cast<GemmMisc*>(smem_raw);
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1024 + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sRing = smem_u32(ring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (p.K + 63) / 64;
  // this CTA's tiles: t = blockIdx.x + j * gridDim.x for j < nt (>= 1: the
  // grid is never larger than the tile count)
  const int nt = (p.tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  // first row and column of tile t: group gi holds row blocks g0 .. g0 + gs - 1
  const auto tile_origin = [&](int t) -> int2 {
    const int gi = t / (kGemmGroup * p.n_tiles), r = t - gi * kGemmGroup * p.n_tiles;
    const int g0 = gi * kGemmGroup, gs = min(kGemmGroup, p.m_tiles - g0);
    return make_int2((g0 + r % gs) * 128, (r / gs) * kGemmN);
  };
  const Guard g{&m.abort_flag, p.status};

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&m.full[s], 1);
      mbar_init(&m.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&m.acc_full[b], 1);
      mbar_init(&m.acc_empty[b], 128);
    }
    mbar_init(&m.fin, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&m.tmem_base, 2 * kGemmN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int it = 0;
      bool ok = true;
      for (int j = 0; ok && j < nt; ++j) {
        const int2 o = tile_origin((int)blockIdx.x + j * (int)gridDim.x);
        const int m0 = o.x, n0 = o.y;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int st = it % kGemmStages;
          if (!g.wait(&m.empty[st], ((it / kGemmStages) & 1) ^ 1, 45)) { ok = false; break; }
          uint8_t* sa = ring + st * kGemmStage;
          mbar_expect_tx(&m.full[st], kGemmStage);
          tma_load_2d(sa, &tmA, &m.full[st], kb * 64, m0);
          for (int c = 0; c < kGemmN / 64; ++c)
            tma_load_2d(sa + kGemmA + c * kGemmBHalf, &tmB, &m.full[st], n0 + 64 * c, kb * 64);
        }
      }
      // no copy may still be landing when the CTA exits
      for (int i = (it > kGemmStages ? it - kGemmStages : 0); i < it; ++i)
        g.drain(&m.full[i % kGemmStages], (i / kGemmStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    const bool leader = lane == 0;
    constexpr uint32_t idC = idesc_bf16_f32(128, kGemmN, false, true);
    bool ok = true;
    int it = 0;
    for (int j = 0; ok && j < nt; ++j) {
      const int buf = j & 1;
      // accumulator buf is free once the epilogue has read tile j - 2 from it
      if (j >= 2 && !g.wait_warp(&m.acc_empty[buf], ((j - 2) >> 1) & 1, 48)) { ok = false; break; }
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int st = it % kGemmStages;
        if (!g.wait_warp(&m.full[st], (it / kGemmStages) & 1, 46)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = sRing + st * kGemmStage;
        const uint64_t ad = sdesc_sw128(sa, 16, 1024);
        const uint64_t bd = sdesc_sw128(sa + kGemmA, kGemmBHalf, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          if (leader)
            umma_bf16(tmem + buf * kGemmN, sdesc_add(ad, kk * 32), sdesc_add(bd, kk * 2048), idC,
                      (kb > 0 || kk > 0) ? 1u : 0u);
        if (leader) umma_commit(&m.empty[st]);
        __syncwarp();
      }
      if (ok && leader) umma_commit(&m.acc_full[buf]);
      __syncwarp();
    }
    if (leader) {
      umma_commit(&m.fin);  // every MMA issued has completed once this arrives
      g.drain(&m.fin, 0);
    }
    __syncwarp();
  } else {
    // warps 2..5: TMEM lane quarter warp % 4, one thread per output row
    const int quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    for (int j = 0; j < nt; ++j) {
      const int buf = j & 1;
      const bool ok = __all_sync(~0u, g.wait(&m.acc_full[buf], (j >> 1) & 1, 47));
      if (!ok) break;
      tc_fence_after();
      const int2 o = tile_origin((int)blockIdx.x + j * (int)gridDim.x);
      const int m0 = o.x, n0 = o.y;
      const int row = m0 + quarter * 32 + lane;
#pragma unroll 1
      for (int c0 = 0; c0 < kGemmN; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + buf * kGemmN + c0, a);
        const int col = n0 + c0;
        if (row >= p.M || col >= p.N) continue;  // N is a multiple of 64: 32 columns are all in or all out
        if (p.mode == kAccInit || p.mode == kAccAdd || p.mode == kAccFinal) {
          float4* ac = reinterpret_cast<float4*>(p.acc + (size_t)row * p.ldacc + col);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 v = make_float4(__uint_as_float(a[4 * q]), __uint_as_float(a[4 * q + 1]),
                                   __uint_as_float(a[4 * q + 2]), __uint_as_float(a[4 * q + 3]));
            if (p.mode != kAccInit) {
              const float4 o = ac[q];
              v.x += o.x;
              v.y += o.y;
              v.z += o.z;
              v.w += o.w;
            }
            if (p.mode == kAccFinal) {
              a[4 * q] = __float_as_uint(v.x);
              a[4 * q + 1] = __float_as_uint(v.y);
              a[4 * q + 2] = __float_as_uint(v.z);
              a[4 * q + 3] = __float_as_uint(v.w);
            } else {
              ac[q] = v;
            }
          }
        }
        if (p.mode == kStoreBf16 || p.mode == kAccFinal) {
          uint4* cr = reinterpret_cast<uint4*>(p.c + (size_t)row * p.ldc + col);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            cr[q] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * q]), __uint_as_float(a[8 * q + 1])),
                               pack_bf16x2(__uint_as_float(a[8 * q + 2]), __uint_as_float(a[8 * q + 3])),
                               pack_bf16x2(__uint_as_float(a[8 * q + 4]), __uint_as_float(a[8 * q + 5])),
                               pack_bf16x2(__uint_as_float(a[8 * q + 6]), __uint_as_float(a[8 * q + 7])));
        }
      }
      tc_fence_before();
      mbar_arrive(&m.acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kGemmN);
  }
}

cudaError_t launch_gemm(const CUtensorMap& tA, const CUtensorMap& tB, const GemmParams& gp, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(lce_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  GemmParams q = gp;
  const long long mt = (gp.M + 127) / 128, ntl = (gp.N + kGemmN - 1) / kGemmN;
  if (mt * ntl > (1ll << 30)) return cudaErrorInvalidValue;
  q.m_tiles = (int)mt;
  q.n_tiles = (int)ntl;
  q.tiles = (int)(mt * ntl);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = q.tiles < sms ? q.tiles : sms;
  if (grid < 1) return cudaSuccess;
  lce_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, st>>>(tA, tB, q);
  return cudaGetLastError();
}

}  // namespace

// The vocabulary split of the (token tile x split) grid: the one that makes
// waves x (tiles per CTA + 1) smallest for `slots` resident CTAs, i.e. the
// shortest run once the last wave's idle SMs and each CTA's pipeline fill (about
// one tile) are counted. At most kLceMaxSplits splits (the workspace's partial
// sums are sized for that).
LceSplit lce_split(int N, int V, int slots) {
  const int TT = (N + kLceTile - 1) / kLceTile, VT = (V + kLceVTile - 1) / kLceVTile;
  if (slots < 1) slots = 1;
  LceSplit best{1, VT};
  long long best_cost = -1;
  for (int s = 1; s <= VT && s <= kLceMaxSplits; ++s) {
    const int per = (VT + s - 1) / s, used = (VT + per - 1) / per;
    const long long ctas = (long long)TT * used, waves = (ctas + slots - 1) / slots;
    const long long cost = waves * (per + 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = LceSplit{used, per};
    }
  }
  return best;
}

int lce_slots() {
  // one resident CTA per SM: 4 x 48 KB stages and all 512 TMEM columns
  static_assert(kLceSmem <= 232448, "shared memory");
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    sms = 148;
  return sms;
}

cudaError_t launch_lce_fwd(int N, int V, int D, const void* hidden, const void* head, const int32_t* targets,
                           float* nll, float* lse, float* target_logit, float* part, uint32_t* status,
                           cudaStream_t st) {
  const LceSplit sp = lce_split(N, V, lce_slots());
  CUtensorMap tH, tW;
  if (!tmap_bf16_2d_sw128(&tH, hidden, D, N, kLceTile) || !tmap_bf16_2d_sw128(&tW, head, D, V, kLceVTile))
    return cudaErrorInvalidValue;
  LceParams p{};
  p.N = N;
  p.V = V;
  p.D = D;
  p.vt_per_split = sp.per;
  p.targets = targets;
  p.part_m = part;
  p.part_s = part + (size_t)sp.splits * N;
  p.part_t = part + (size_t)2 * sp.splits * N;
  p.status = status;
  cudaError_t e = cudaFuncSetAttribute(lce_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLceSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((N + kLceTile - 1) / kLceTile, sp.splits);
  lce_kernel<false><<<grid, kLceThreads, kLceSmem, st>>>(tH, tW, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  lce_merge_kernel<<<(N + 255) / 256, 256, 0, st>>>(p, sp.splits, nll, lse, target_logit);
  return cudaGetLastError();
}

}  // namespace pa

namespace pa {

int lce_bwd_chunk(int N, int V) {
  // dz and dz^T of one chunk together take 4 N Vc bytes: at most 512 MiB
  // (chunks are whole vocabulary tiles)
  long long vc = ((1ll << 27) / (N > 0 ? N : 1)) / kLceVTile * kLceVTile;
  const long long vmax = (long long)(V + kLceVTile - 1) / kLceVTile * kLceVTile;
  if (vc > 8192) vc = 8192;
  if (vc > vmax) vc = vmax;
  if (vc < kLceVTile) vc = kLceVTile;
  return (int)vc;
}

LceBwdLayout lce_bwd_layout(int N, int V, int D) {
  LceBwdLayout L;
  L.vc = lce_bwd_chunk(N, V);
  L.chunks = (V + L.vc - 1) / L.vc;
  L.ld_dzt = (N + 63) / 64 * 64;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  L.acc = 256;
  L.dz = L.acc + (L.chunks > 1 ? up((size_t)N * D * 4) : 0);
  L.dzt = L.dz + up((size_t)N * L.vc * 2);
  L.bytes = L.dzt + up((size_t)L.vc * L.ld_dzt * 2);
  return L;
}

cudaError_t launch_lce_bwd(int N, int V, int D, const void* hidden, const void* head, const int32_t* targets,
                           const float* lse, const float* g, void* dhidden, void* dhead, void* ws, uint32_t* status,
                           cudaStream_t st) {
  const LceBwdLayout L = lce_bwd_layout(N, V, D);
  uint8_t* w = static_cast<uint8_t*>(ws);
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(w + L.dz);
  __nv_bfloat16* dzt = reinterpret_cast<__nv_bfloat16*>(w + L.dzt);
  float* acc = reinterpret_cast<float*>(w + L.acc);
  CUtensorMap tH, tW, tHb;
  if (!tmap_bf16_2d_sw128(&tH, hidden, D, N, kLceTile) || !tmap_bf16_2d_sw128(&tW, head, D, V, kLceVTile) ||
      !tmap_bf16_2d_sw128(&tHb, hidden, D, N, 64))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(lce_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLceSmem);
  if (e != cudaSuccess) return e;
  for (int c = 0; c < L.chunks; ++c) {
    const int cv0 = c * L.vc, kc = (V - cv0 < L.vc) ? V - cv0 : L.vc;  // the chunk's vocabulary rows
    // dz (and dz^T) of the chunk: one CTA per SM over its (token tile,
    // vocabulary tile) pairs
    LceParams p{};
    p.N = N;
    p.V = V;
    p.D = D;
    p.vt_per_split = 0;
    p.targets = targets;
    p.status = status;
    p.vt_base = cv0 / kLceVTile;
    p.vt_end = (cv0 + kc + kLceVTile - 1) / kLceVTile;
    p.lse = lse;
    p.g = g;
    p.dz = dz;
    p.ld_dz = L.vc;
    p.dzt = dhead ? dzt : nullptr;
    p.ld_dzt = L.ld_dzt;
    const int pairs = ((N + kLceTile - 1) / kLceTile) * (p.vt_end - p.vt_base);
    lce_kernel<true><<<pairs < lce_slots() ? pairs : lce_slots(), kLceThreads, kLceSmem, st>>>(tH, tW, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // dW rows of the chunk = dz^T H (tokens are the contraction)
    if (dhead) {
      CUtensorMap tA;
      if (!tmap_bf16_2d_sw128_pitch(&tA, dzt, N, kc, L.ld_dzt, 128)) return cudaErrorInvalidValue;
      GemmParams gp{};
      gp.M = kc;
      gp.N = D;
      gp.K = N;
      gp.mode = kStoreBf16;
      gp.c = static_cast<__nv_bfloat16*>(dhead) + (size_t)cv0 * D;
      gp.ldc = D;
      gp.status = status;
      if ((e = launch_gemm(tA, tHb, gp, st)) != cudaSuccess) return e;
    }
    // dH += dz W[chunk] (the chunk's vocabulary rows are the contraction)
    CUtensorMap tA, tB;
    if (!tmap_bf16_2d_sw128_pitch(&tA, dz, kc, N, L.vc, 128) ||
        !tmap_bf16_2d_sw128(&tB, static_cast<const __nv_bfloat16*>(head) + (size_t)cv0 * D, D, kc, 64))
      return cudaErrorInvalidValue;
    GemmParams gp{};
    gp.M = N;
    gp.N = D;
    gp.K = kc;
    gp.mode = L.chunks == 1 ? kStoreBf16 : c == 0 ? kAccInit : c == L.chunks - 1 ? kAccFinal : kAccAdd;
    gp.c = static_cast<__nv_bfloat16*>(dhidden);
    gp.ldc = D;
    gp.acc = acc;
    gp.ldacc = D;
    gp.status = status;
    if ((e = launch_gemm(tA, tB, gp, st)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pa
