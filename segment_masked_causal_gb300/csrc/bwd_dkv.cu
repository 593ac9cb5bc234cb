// bwd_dkv.cu -- packed attention backward, dK/dV pass, for sm_103a.
//
// One CTA per (key tile of 128 rows, kv head, batch row). It walks every query
// head of its group and, for each, the query tiles from the diagonal up to
// the last tile whose segment range overlaps the key tile's -- the query walk
// ends at the key block's segment end instead of masking the rest
// (mlx-train-perf 0.5.1 README, "Sequence packing", the 0.5.0 dK/dV change).
// Per visited (query head, query tile) "step", with K and V resident in
// shared memory:
//   S^T  = K Q^T   (TMEM, 128 columns)   P^T  = exp(scale * S^T - lse)
//   dP^T = V dO^T  (TMEM, 128 columns)   dS^T = P^T * (dP^T - delta)
//   dV += P^T dO   dK += dS^T Q          (TMEM accumulators; P^T and dS^T are
//                                         written back as bf16 over S^T and fed
//                                         to the MMA straight from TMEM)
// and finally dK *= scale. The group's heads are summed inside the CTA in a
// fixed order, so dK/dV need no atomics and are deterministic.
//
// Every MMA is 128 x 128 (or 128 x D) x 16, wide enough that the one issuing
// thread keeps the tensor pipe busy. Besides dV and dK, TMEM holds two
// 128-column regions that swap roles every step: S^T of step i goes where dP^T
// of step i-1 was (released by the softmax warps as soon as they have read
// it), dP^T where step i-1's P^T/dS^T were (free once its gradient MMAs ran).
//
// Warp roles: warp 0 TMA producer (Q and dO tiles plus the query tile's lse,
// delta and segment ids through a 2-stage ring), warp 1 MMA issuer and TMEM
// owner, warps 2..9 softmax: two threads per key row, 64 query columns each.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct DkvLayout {
  static constexpr int NS = 2;                   // Q/dO stages
  static constexpr uint32_t TB = 128 * D * 2;    // one 128-row tile of K, V, Q or dO
  static constexpr uint32_t CHUNK = 128 * 128;   // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TB;
  static constexpr uint32_t OFF_Q = OFF_V + TB;
  static constexpr uint32_t OFF_DO = OFF_Q + NS * TB;
  static constexpr uint32_t TILE_BYTES = OFF_DO + NS * TB;
  static constexpr uint32_t MISC_BYTES = 4096;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: dV, dK accumulators (D columns each), then two 128-column regions
  static constexpr uint32_t TM_DV = 0, TM_DK = D, TM_X = 256, TM_Y = 384, TMEM_COLS = 512;
};

struct DkvMisc {
  uint64_t kv_full, q_full[2], q_empty[2];
  uint64_t s_full[2], dp_free[2], pds_full[2], grad_done[2], mma_final;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float lse[2][128];
  alignas(16) float dl[2][128];
  alignas(16) int32_t segq[2][128];
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const AttnParams p) {
  using L = DkvLayout<D>;
  constexpr int NS = L::NS;
  static_assert(sizeof(DkvMisc) <= L::MISC_BYTES, "misc region");
  static_assert(L::SMEM <= 232448, "shared memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DkvMisc& m = *reinterpret_cast<DkvMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(DkvMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sDO = smem_u32(base + L::OFF_DO);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest causal walks (smallest key tile index) first, across all heads
  const int per_tile = p.Hkv * p.B;
  const int tk = (int)blockIdx.x / per_tile;
  const int hk = (int)blockIdx.x % p.Hkv, b = ((int)blockIdx.x / p.Hkv) % p.B;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};
  const QWalk walk(trow, tk);
  const int h0 = hk * p.G, h1 = h0 + p.G;

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    mbar_init(&m.kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&m.q_full[s], 1);
      mbar_init(&m.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.dp_free[s], 256);
      mbar_init(&m.pds_full[s], 256);
      mbar_init(&m.grad_done[s], 1);
    }
    mbar_init(&m.mma_final, 1);
    fence_mbar_init();
  }
  if (!p.seg)  // every token in one segment: the query-tile ids are all 0
    for (int x = threadIdx.x; x < NS * 128; x += blockDim.x) (&m.segq[0][0])[x] = 0;
  if (warp == 1) {
    tmem_alloc(&m.tmem_base, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int krow = (b * p.Hkv + hk) * p.N + tk * kTile;
      mbar_expect_tx(&m.kv_full, 2 * L::TB);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(base + L::OFF_K + c * L::CHUNK, &tmK, &m.kv_full, c * 64, krow);
        tma_load_2d(base + L::OFF_V + c * L::CHUNK, &tmV, &m.kv_full, c * 64, krow);
      }
      const uint32_t qbytes = 2 * L::TB + 1024 + (p.seg ? 512 : 0);
      int i = 0;
      bool ok = true;
      for (int hq = h0; ok && hq < h1; ++hq) {
        for (int tq = walk.first(); tq < walk.end(); tq = walk.next(tq), ++i) {
          const int st = i % NS;
          if (!g.wait(&m.q_empty[st], ((i / NS) & 1) ^ 1, 1)) { ok = false; break; }
          const int qrow = (b * p.Hq + hq) * p.N + tq * kTile;
          mbar_expect_tx(&m.q_full[st], qbytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(base + L::OFF_Q + st * L::TB + c * L::CHUNK, &tmQ, &m.q_full[st], c * 64, qrow);
            tma_load_2d(base + L::OFF_DO + st * L::TB + c * L::CHUNK, &tmDO, &m.q_full[st], c * 64, qrow);
          }
          bulk_load(m.lse[st], p.lse_in + qrow, 512, &m.q_full[st]);
          bulk_load(m.dl[st], p.delta + qrow, 512, &m.q_full[st]);
          if (p.seg) bulk_load(m.segq[st], p.seg + (size_t)b * p.N + tq * kTile, 512, &m.q_full[st]);
        }
      }
      g.drain(&m.kv_full, 0);
      for (int k = (i > NS ? i - NS : 0); k < i; ++k) g.drain(&m.q_full[k % NS], (k / NS) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idG = idesc_bf16_f32(128, D, false, true);
      const uint64_t kd = sdesc_sw128(sK, 16, 1024), vd = sdesc_sw128(sV, 16, 1024);
      // dV += P^T dO, dK += dS^T Q for step i: thread-half h keeps P^T of its 64
      // query columns in region columns 64h..64h+31 and dS^T in 64h+32..64h+63
      auto issue_grad = [&](int i) -> bool {
        const int bb = i & 1, st = i % NS;
        if (!g.wait(&m.pds_full[bb], (i >> 1) & 1, 2)) return false;
        tc_fence_after();
        const uint32_t sreg = tmem + (bb ? L::TM_Y : L::TM_X);
        const uint64_t gq = sdesc_sw128(sQ + st * L::TB, L::CHUNK, 1024);
        const uint64_t gd = sdesc_sw128(sDO + st * L::TB, L::CHUNK, 1024);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t pcol = sreg + (kk >> 2) * 64 + (kk & 3) * 8;
          const uint32_t acc = kk > 0 ? 1u : acc0;
          umma_bf16_ta(tmem + L::TM_DV, pcol, sdesc_add(gd, kk * 2048), idG, acc);
          umma_bf16_ta(tmem + L::TM_DK, pcol + 32, sdesc_add(gq, kk * 2048), idG, acc);
        }
        umma_commit(&m.grad_done[bb]);
        umma_commit(&m.q_empty[st]);
        return true;
      };
      bool ok = g.wait(&m.kv_full, 0, 3);
      int i = 0;
      for (int hq = h0; ok && hq < h1; ++hq) {
        for (int tq = walk.first(); tq < walk.end(); tq = walk.next(tq), ++i) {
          const int bb = i & 1, st = i % NS;
          const uint32_t sreg = tmem + (bb ? L::TM_Y : L::TM_X), dreg = tmem + (bb ? L::TM_X : L::TM_Y);
          if (!g.wait(&m.q_full[st], (i / NS) & 1, 4)) { ok = false; break; }
          // S^T_i where dP^T_{i-1} was: free once that softmax has read it
          if (i >= 1 && !g.wait(&m.dp_free[(i - 1) & 1], ((i - 1) >> 1) & 1, 5)) { ok = false; break; }
          tc_fence_after();
          const uint64_t qd = sdesc_sw128(sQ + st * L::TB, 16, 1024);
          const uint64_t dod = sdesc_sw128(sDO + st * L::TB, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
            umma_bf16(sreg, sdesc_add(kd, ko), sdesc_add(qd, ko), idS, kk > 0 ? 1u : 0u);
          }
          if (i >= 1) {
            // gradient MMAs of step i-1, then dP^T_i into the region they read
            if (!issue_grad(i - 1)) { ok = false; break; }
            if (!g.wait(&m.grad_done[(i - 1) & 1], ((i - 1) >> 1) & 1, 6)) { ok = false; break; }
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
            umma_bf16(dreg, sdesc_add(vd, ko), sdesc_add(dod, ko), idS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&m.s_full[bb]);
        }
      }
      if (ok && i > 0) issue_grad(i - 1);
      umma_commit(&m.mma_final);
      g.drain(&m.mma_final, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int hsel = (warp - 2) >> 2;  // which 64 query columns of every step
    const int r = quarter * 32 + lane;
    const int kvidx = tk * kTile + r;
    const int32_t segk = p.seg ? p.seg[(size_t)b * p.N + kvidx] : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const int4 kt = trow[tk];
    bool ok = true;
    int i = 0;
    for (int hq = h0; ok && hq < h1; ++hq) {
      for (int tq = walk.first(); tq < walk.end(); tq = walk.next(tq), ++i) {
        const int bb = i & 1, st = i % NS;
        ok = g.wait(&m.q_full[st], (i / NS) & 1, 7);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        ok = g.wait(&m.s_full[bb], (i >> 1) & 1, 8);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sreg = tmem + lane_base + (bb ? L::TM_Y : L::TM_X) + hsel * 64;
        const uint32_t dreg = tmem + lane_base + (bb ? L::TM_X : L::TM_Y) + hsel * 64;
        const bool masked = !tile_pair_full(tq, trow[tq], tk, kt);
        uint32_t sv[2][32];
        tmem_ld32x2(sreg, sreg + 32, sv[0], sv[1]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dp[32];
          tmem_ld32(dreg + 32 * c, dp);
          if (c == 1) {  // dP^T fully read: the region may take the next step's S^T
            tc_fence_before();
            mbar_arrive(&m.dp_free[bb]);
          }
          const int c0 = hsel * 64 + 32 * c;  // query column within the tile
          const int q0 = tq * kTile + c0;
          const float4* l4 = reinterpret_cast<const float4*>(&m.lse[st][c0]);
          const float4* d4 = reinterpret_cast<const float4*>(&m.dl[st][c0]);
          const int4* g4 = reinterpret_cast<const int4*>(&m.segq[st][c0]);
          uint32_t pw[16], dw[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 lv = l4[e4], dv = d4[e4];
            const float lz[4] = {lv.x, lv.y, lv.z, lv.w}, dz[4] = {dv.x, dv.y, dv.z, dv.w};
            float sz[4], pz[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) sz[e] = __uint_as_float(sv[c][e4 * 4 + e]);
            if (masked) {
              const int4 gv = g4[e4];
              const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                sz[e] = (q0 + e4 * 4 + e >= kvidx && gz[e] == segk) ? sz[e] : -INFINITY;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) pz[e] = ex2(fmaf(sz[e], sl2, -lz[e] * 1.4426950408889634f));
            pw[e4 * 2] = pack_bf16x2(pz[0], pz[1]);
            pw[e4 * 2 + 1] = pack_bf16x2(pz[2], pz[3]);
            dw[e4 * 2] = pack_bf16x2(pz[0] * (__uint_as_float(dp[e4 * 4]) - dz[0]),
                                     pz[1] * (__uint_as_float(dp[e4 * 4 + 1]) - dz[1]));
            dw[e4 * 2 + 1] = pack_bf16x2(pz[2] * (__uint_as_float(dp[e4 * 4 + 2]) - dz[2]),
                                         pz[3] * (__uint_as_float(dp[e4 * 4 + 3]) - dz[3]));
          }
          // P^T and dS^T over this thread's own S^T columns (all read above)
          tmem_st16x2(sreg + 16 * c, sreg + 32 + 16 * c, pw, dw);
        }
        tc_fence_before();
        mbar_arrive(&m.pds_full[bb]);
      }
    }
    if (ok && i > 0) {
      ok = g.wait(&m.grad_done[(i - 1) & 1], ((i - 1) >> 1) & 1, 9);
      ok = __all_sync(~0u, ok);
    }
    if (ok && i > 0) {
      tc_fence_after();
      const size_t row = (size_t)(b * p.Hkv + hk) * p.N + kvidx;
      uint4* vrow = reinterpret_cast<uint4*>(p.dv + row * D);
      uint4* krow = reinterpret_cast<uint4*>(p.dk + row * D);
      const float sc = p.scale;
#pragma unroll
      for (int c0 = hsel * (D / 2); c0 < (hsel + 1) * (D / 2); c0 += 32) {
        uint32_t v[32], k[32];
        tmem_ld32x2(tmem + lane_base + L::TM_DV + c0, tmem + lane_base + L::TM_DK + c0, v, k);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 wv, wk;
          wv.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]), __uint_as_float(v[q4 * 8 + 1]));
          wv.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]), __uint_as_float(v[q4 * 8 + 3]));
          wv.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]), __uint_as_float(v[q4 * 8 + 5]));
          wv.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]), __uint_as_float(v[q4 * 8 + 7]));
          wk.x = pack_bf16x2(__uint_as_float(k[q4 * 8 + 0]) * sc, __uint_as_float(k[q4 * 8 + 1]) * sc);
          wk.y = pack_bf16x2(__uint_as_float(k[q4 * 8 + 2]) * sc, __uint_as_float(k[q4 * 8 + 3]) * sc);
          wk.z = pack_bf16x2(__uint_as_float(k[q4 * 8 + 4]) * sc, __uint_as_float(k[q4 * 8 + 5]) * sc);
          wk.w = pack_bf16x2(__uint_as_float(k[q4 * 8 + 6]) * sc, __uint_as_float(k[q4 * 8 + 7]) * sc);
          vrow[(c0 >> 3) + q4] = wv;
          krow[(c0 >> 3) + q4] = wk;
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
cudaError_t launch_dkv_d(const AttnParams& p, const void* q, const void* k, const void* v, const void* dout,
                         cudaStream_t st) {
  using L = DkvLayout<D>;
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t qrows = (uint64_t)p.B * p.Hq * p.N, krows = (uint64_t)p.B * p.Hkv * p.N;
  if (!tmap_bf16_2d_sw128(&tq, q, D, qrows, 128) || !tmap_bf16_2d_sw128(&tdo, dout, D, qrows, 128) ||
      !tmap_bf16_2d_sw128(&tk, k, D, krows, 128) || !tmap_bf16_2d_sw128(&tv, v, D, krows, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dkv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * p.Hkv * p.B);
  dkv_kernel<D><<<grid, 320, L::SMEM, st>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkv(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                           const void* dout, cudaStream_t st) {
  return D == 128 ? launch_dkv_d<128>(p, q, k, v, dout, st) : launch_dkv_d<64>(p, q, k, v, dout, st);
}

}  // namespace pa
