// bwd_dq.cu -- packed attention backward, dQ pass, for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row); it visits the
// same key tiles as the forward (the changelog's PACKED dQ kernel: cross-
// segment blocks skipped). Every key tile is processed as two 64-column
// halves ("steps"):
//   S  = Q K^T   (TMEM, 64 columns)   P  = exp(scale * S - lse)
//   dP = dO V^T  (TMEM, 64 columns)   dS = P * (dP - delta)   (bf16, over S)
//   dQ += dS K   (TMEM accumulator, dS read straight from TMEM)
// and finally dQ *= scale. The probabilities are recomputed from the saved
// log-sum-exp (mlx-train-perf 0.5.1 README, "Flash-attention training path":
// the backward recomputes the tiles it needs from O(N) saved state).
//
// Q and dO stay in TMEM for the whole CTA (each row thread stores its own row
// once), so the S and dP MMAs read only K and V from shared memory. S/dP of
// consecutive steps alternate between two TMEM buffers: the MMA issuer starts
// step i+1 while the softmax warps work on step i.
//
// Warp roles: warp 0 TMA producer (K/V tiles, 3-stage ring), warp 1 MMA
// issuer and TMEM owner, warps 2..9 two threads per query row, 32 key columns
// each.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct DqLayout {
  static constexpr int NS = 3;
  static constexpr uint32_t KV_BYTES = 128 * D * 2;
  static constexpr uint32_t KV_CHUNK = 128 * 128;  // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + NS * KV_BYTES;
  static constexpr uint32_t TILE_BYTES = OFF_V + NS * KV_BYTES;
  static constexpr uint32_t MISC_BYTES = 2048;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: Q and dO as bf16 (D/2 columns each), dQ accumulator, two step buffers
  // of 128 columns whose 64-column halves hold S and dP and swap roles on every use
  static constexpr uint32_t TM_Q = 0, TM_DO = D / 2, TM_DQ = D, TM_BUF = 2 * D, TMEM_COLS = 512;
};

struct DqMisc {
  uint64_t kv_full[3], kv_empty[3];
  uint64_t qdo_ready, s_full[2], ds_full[2], dq_done[2], mma_final;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) int32_t segkv[3][128];
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __nv_bfloat16* __restrict__ q, const AttnParams p) {
  using L = DqLayout<D>;
  constexpr int NS = L::NS;
  static_assert(sizeof(DqMisc) <= L::MISC_BYTES, "misc region");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DqMisc& m = *reinterpret_cast<DqMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(DqMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // longest causal rows first, across all heads and batch rows
  const int per_tile = p.Hq * p.B;
  const int tq = p.T - 1 - (int)blockIdx.x / per_tile;
  const int h = (int)blockIdx.x % p.Hq, b = ((int)blockIdx.x / p.Hq) % p.B, hk = h / p.G;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&m.kv_full[s], 1);
      mbar_init(&m.kv_empty[s], 1);
    }
    mbar_init(&m.qdo_ready, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.ds_full[s], 256);
      mbar_init(&m.dq_done[s], 1);
    }
    mbar_init(&m.mma_final, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&m.tmem_base, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;
  const KvWalk walk(trow, tq);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int krow0 = (b * p.Hkv + hk) * p.N;
      int j = 0;
      for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS;
        if (!g.wait(&m.kv_empty[st], ((j / NS) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&m.kv_full[st], 2 * L::KV_BYTES + (p.seg ? 512 : 0));
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(base + L::OFF_K + st * L::KV_BYTES + c * L::KV_CHUNK, &tmK, &m.kv_full[st], c * 64,
                      krow0 + tk * kTile);
          tma_load_2d(base + L::OFF_V + st * L::KV_BYTES + c * L::KV_CHUNK, &tmV, &m.kv_full[st], c * 64,
                      krow0 + tk * kTile);
        }
        if (p.seg) bulk_load(m.segkv[st], p.seg + (size_t)b * p.N + tk * kTile, 512, &m.kv_full[st]);
      }
      for (int i = (j > NS ? j - NS : 0); i < j; ++i) g.drain(&m.kv_full[i % NS], (i / NS) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idQ = idesc_bf16_f32(128, D, false, true);
      // dQ += dS_i K_half(i): dS from TMEM, K rows of the half as the K dimension
      auto issue_dq = [&](int i) -> bool {
        const int bb = i & 1, st = (i >> 1) % NS, half = i & 1;
        if (!g.wait(&m.ds_full[bb], (i >> 1) & 1, 2)) return false;
        tc_fence_after();
        const uint32_t buf = tmem + L::TM_BUF + bb * 128 + (((i >> 1) & 1) ? 64 : 0);  // step i's S half
        const uint64_t kd = sdesc_sw128(sK + st * L::KV_BYTES + half * 64 * 128, L::KV_CHUNK, 1024);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ta(tmem + L::TM_DQ, buf + (kk >> 1) * 32 + (kk & 1) * 8, sdesc_add(kd, kk * 2048), idQ,
                       kk > 0 ? 1u : acc0);
        umma_commit(&m.dq_done[bb]);
        if (half == 1) umma_commit(&m.kv_empty[st]);
        return true;
      };
      bool ok = g.wait(&m.qdo_ready, 0, 3);
      tc_fence_after();
      int i = 0, j = 0;
      for (int tk = walk.first(); ok && tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS;
        if (!g.wait(&m.kv_full[st], (j / NS) & 1, 4)) { ok = false; break; }
        for (int half = 0; half < 2; ++half, ++i) {
          const int bb = i & 1;
          // Buffer bb's halves swap roles on every use: S of step i goes where
          // dP of step i-2 was (free once that softmax read it), dP where step
          // i-2's dS was (free once its dQ MMAs ran).
          const uint32_t buf = tmem + L::TM_BUF + bb * 128;
          const uint32_t sO = ((i >> 1) & 1) ? 64 : 0, dO_ = 64 - sO;
          const uint64_t kd = sdesc_sw128(sK + st * L::KV_BYTES + half * 64 * 128, 16, 1024);
          const uint64_t vd = sdesc_sw128(sV + st * L::KV_BYTES + half * 64 * 128, 16, 1024);
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32;
            umma_bf16_ta(buf + sO, tmem + L::TM_Q + kk * 8, sdesc_add(kd, ko), idS, kk > 0 ? 1u : 0u);
          }
          // only now wait for step i-2's dQ MMAs: S of step i is queued behind them
          if (i >= 2 && !g.wait(&m.dq_done[bb], ((i - 2) >> 1) & 1, 5)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32;
            umma_bf16_ta(buf + dO_, tmem + L::TM_DO + kk * 8, sdesc_add(vd, ko), idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&m.s_full[bb]);
          if (i > 0 && !issue_dq(i - 1)) { ok = false; break; }
        }
      }
      if (ok && i > 0) issue_dq(i - 1);
      umma_commit(&m.mma_final);
      g.drain(&m.mma_final, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int hsel = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int qidx = tq * kTile + r;
    const size_t row = (size_t)(b * p.Hq + h) * p.N + qidx;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const float lse2 = p.lse_in[row] * 1.4426950408889634f;
    const float dlt = p.delta[row];
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    // this thread's half of its Q and dO rows into TMEM, as bf16 pairs
    {
      const uint32_t* qsrc = reinterpret_cast<const uint32_t*>(q + row * D) + hsel * (D / 4);
      const uint32_t* dsrc = reinterpret_cast<const uint32_t*>(p.dout + row * D) + hsel * (D / 4);
#pragma unroll
      for (int c0 = 0; c0 < D / 4; c0 += 16) {
        uint32_t a[16], d[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const uint4 x = __ldg(reinterpret_cast<const uint4*>(qsrc + c0 + e));
          const uint4 y = __ldg(reinterpret_cast<const uint4*>(dsrc + c0 + e));
          a[e] = x.x; a[e + 1] = x.y; a[e + 2] = x.z; a[e + 3] = x.w;
          d[e] = y.x; d[e + 1] = y.y; d[e + 2] = y.z; d[e + 3] = y.w;
        }
        tmem_st16(tmem + lane_base + L::TM_Q + hsel * (D / 4) + c0, a);
        tmem_st16(tmem + lane_base + L::TM_DO + hsel * (D / 4) + c0, d);
      }
      tc_fence_before();
      mbar_arrive(&m.qdo_ready);
    }
    bool ok = true;
    int i = 0, j = 0;
    for (int tk = walk.first(); ok && tk <= tq; tk = walk.next(tk), ++j) {
      const int st = j % NS;
      const bool masked = !tile_pair_full(tq, walk.qt, tk, trow[tk]);
      if (masked && p.seg) {  // segment ids of this key tile arrived with it
        ok = g.wait(&m.kv_full[st], (j / NS) & 1, 6);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      for (int half = 0; half < 2; ++half, ++i) {
        const int bb = i & 1;
        ok = g.wait(&m.s_full[bb], (i >> 1) & 1, 7);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sO = ((i >> 1) & 1) ? 64 : 0;
        const uint32_t buf = tmem + lane_base + L::TM_BUF + bb * 128 + sO + hsel * 32;
        uint32_t sv[32], dp[32];
        tmem_ld32x2(buf, tmem + lane_base + L::TM_BUF + bb * 128 + (64 - sO) + hsel * 32, sv, dp);
        const int c0 = half * 64 + hsel * 32;  // key column within the tile
        const int k0 = tk * kTile + c0;
        uint32_t dw[16];
        float sz[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) sz[e] = __uint_as_float(sv[e]);
        if (masked) {
          const int4* g4 = reinterpret_cast<const int4*>(&m.segkv[st][c0]);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int4 gv = p.seg ? g4[e4] : make_int4(0, 0, 0, 0);
            const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = e4 * 4 + e;
              sz[c] = (k0 + c <= qidx && gz[e] == segq) ? sz[c] : -INFINITY;
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2(fmaf(sz[e], sl2, -lse2)), p1 = ex2(fmaf(sz[e + 1], sl2, -lse2));
          dw[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - dlt), p1 * (__uint_as_float(dp[e + 1]) - dlt));
        }
        tmem_st16(buf, dw);  // dS over this thread's own S columns
        tc_fence_before();
        mbar_arrive(&m.ds_full[bb]);
      }
    }
    if (ok && i > 0) {
      ok = g.wait(&m.dq_done[(i - 1) & 1], ((i - 1) >> 1) & 1, 10);
      ok = __all_sync(~0u, ok);
    }
    if (ok && i > 0) {
      tc_fence_after();
      uint4* drow = reinterpret_cast<uint4*>(p.dq + row * D);
      const float sc = p.scale;
#pragma unroll
      for (int c0 = hsel * (D / 2); c0 < (hsel + 1) * (D / 2); c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_DQ + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * sc, __uint_as_float(v[q4 * 8 + 1]) * sc);
          w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * sc, __uint_as_float(v[q4 * 8 + 3]) * sc);
          w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * sc, __uint_as_float(v[q4 * 8 + 5]) * sc);
          w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * sc, __uint_as_float(v[q4 * 8 + 7]) * sc);
          drow[(c0 >> 3) + q4] = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_dq_d(const AttnParams& p, const void* q, const void* k, const void* v, const void* dout,
                        cudaStream_t st) {
  using L = DqLayout<D>;
  CUtensorMap tk, tv;
  const uint64_t krows = (uint64_t)p.B * p.Hkv * p.N;
  if (!tmap_bf16_2d_sw128(&tk, k, D, krows, 128) || !tmap_bf16_2d_sw128(&tv, v, D, krows, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  AttnParams pp = p;
  pp.dout = static_cast<const __nv_bfloat16*>(dout);
  dim3 grid(p.T * p.Hq * p.B);
  dq_kernel<D><<<grid, 320, L::SMEM, st>>>(tk, tv, static_cast<const __nv_bfloat16*>(q), pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                          const void* dout, cudaStream_t st) {
  return D == 128 ? launch_dq_d<128>(p, q, k, v, dout, st) : launch_dq_d<64>(p, q, k, v, dout, st);
}

}  // namespace pa
