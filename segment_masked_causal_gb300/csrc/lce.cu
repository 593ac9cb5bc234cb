// lce.cu -- fused linear cross-entropy forward: per-token NLL, log-sum-exp and
// target logit of z = H W^T without storing the (N, V) logits
// (mlx-train-perf 0.5.1 README, "The fused cross-entropy loss").
//
// Grid: (token tiles of 128) x (vocabulary splits). A CTA walks its split's
// vocabulary tiles of 128 rows; for each, the tcgen05 tensor cores form the
// 128 x 128 logit tile in TMEM from 64-wide K slices of H and W that TMA
// streams through a 4-stage ring, and four epilogue warps (one thread per
// token, reading its TMEM lane) fold the tile into a running maximum and sum
// of exponentials and pick up the target logit when it falls in the tile.
// Two TMEM accumulators let the next tile's products run while the epilogue
// reads the previous one. Each CTA writes its split's (max, sum) per token
// and, for tokens whose target lies in its split, the target logit; a merge
// kernel combines the splits.
//
// Roles: warp 0 lane 0 loads (TMA), warp 1 issues the MMAs (lane 0) and owns
// the TMEM allocation, warps 4..7 are the epilogue (warp % 4 = TMEM lane
// quarter). Every wait is bounded (sm103.cuh).
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

constexpr int kLceStages = 4;
constexpr int kLceTile = 128;                  // tokens per CTA and vocabulary rows per tile
constexpr uint32_t kLceSlice = 128 * 128;      // one 128 x 64 bf16 slice (128-byte rows), 16 KB
constexpr uint32_t kLceStage = 2 * kLceSlice;  // H slice + W slice
constexpr int kLceThreads = 256;
constexpr uint32_t kLceTmemCols = 256;  // two 128-column fp32 accumulators

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
};

__global__ void __launch_bounds__(kLceThreads, 1)
    lce_fwd_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW,
                   const LceParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  LceMisc& m = *reinterpret_cast<LceMisc*>(smem_raw);
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1024 + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sRing = smem_u32(ring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tm = blockIdx.x;
  const int VT = (p.V + kLceTile - 1) / kLceTile;
  const int vt0 = blockIdx.y * p.vt_per_split;
  const int vt1 = min(vt0 + p.vt_per_split, VT);
  const int nt = vt1 - vt0;  // >= 1 by construction of the grid
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
          tma_load_2d(ring + st * kLceStage, &tmH, &m.full[st], kc * 64, tm * kLceTile);
          tma_load_2d(ring + st * kLceStage + kLceSlice, &tmW, &m.full[st], kc * 64, (vt0 + j) * kLceTile);
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
    constexpr uint32_t idZ = idesc_bf16_f32(128, 128, false, false);
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
            umma_bf16(tmem + buf * 128, sdesc_add(hd, kk * 32), sdesc_add(wd, kk * 32), idZ,
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
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int token = tm * kLceTile + r;
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
      const int v0 = (vt0 + j) * kLceTile;
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + buf * 128 + c0, a);
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
    z = p.part_t[(size_t)(t / kLceTile / p.vt_per_split) * p.N + i];
    n = l - z;
  }
  lse[i] = l;
  tgt_out[i] = z;
  nll[i] = n;
}

}  // namespace

LceSplit lce_split(int N, int V) {
  const int TT = (N + kLceTile - 1) / kLceTile, VT = (V + kLceTile - 1) / kLceTile;
  int splits = (2 * 148 + TT - 1) / TT;
  if (splits < 1) splits = 1;
  if (splits > VT) splits = VT;
  const int per = (VT + splits - 1) / splits;
  return LceSplit{(VT + per - 1) / per, per};
}

cudaError_t launch_lce_fwd(int N, int V, int D, const void* hidden, const void* head, const int32_t* targets,
                           float* nll, float* lse, float* target_logit, float* part, uint32_t* status,
                           cudaStream_t st) {
  const LceSplit sp = lce_split(N, V);
  CUtensorMap tH, tW;
  if (!tmap_bf16_2d_sw128(&tH, hidden, D, N, kLceTile) || !tmap_bf16_2d_sw128(&tW, head, D, V, kLceTile))
    return cudaErrorInvalidValue;
  LceParams p{N, V, D, sp.per, targets, part, part + (size_t)sp.splits * N, part + (size_t)2 * sp.splits * N,
              status};
  cudaError_t e = cudaFuncSetAttribute(lce_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLceSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((N + kLceTile - 1) / kLceTile, sp.splits);
  lce_fwd_kernel<<<grid, kLceThreads, kLceSmem, st>>>(tH, tW, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  lce_merge_kernel<<<(N + 255) / 256, 256, 0, st>>>(p, sp.splits, nll, lse, target_logit);
  return cudaGetLastError();
}

}  // namespace pa
