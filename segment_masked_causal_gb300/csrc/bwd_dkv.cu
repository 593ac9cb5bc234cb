// bwd_dkv.cu -- packed attention backward, dK/dV pass, for sm_103a.
//
// One CTA per (key tile of 128 rows, kv head, batch row). It walks every query
// head of its group and, for each, the query tiles from the diagonal up to
// the last tile whose segment range overlaps the key tile's -- the query walk
// ends at the key block's segment end instead of masking the rest
// (mlx-train-perf 0.5.1 README, "Sequence packing", the 0.5.0 dK/dV change).
// Every query tile is processed as two 64-row halves ("steps"). Per step, with
// K and V resident in shared memory:
//   S^T  = K Q^T   (TMEM, 64 columns)   P^T  = exp(scale * S^T - lse)
//   dP^T = V dO^T  (TMEM, 64 columns)   dS^T = P^T * (dP^T - delta)
//   dV += P^T dO   dK += dS^T Q         (TMEM accumulators; P^T and dS^T are
//                                        written back as bf16 over S^T and fed
//                                        to the MMA straight from TMEM)
// and finally dK *= scale. The group's heads are summed inside the CTA in a
// fixed order, so dK/dV need no atomics and are deterministic.
//
// Pipelining: S^T/dP^T of a step live in one of two TMEM buffers, so the MMA
// issuer starts step i+1's S^T and dP^T before step i's gradient MMAs and the
// tensor core runs while the softmax warps work on step i. Within a buffer the
// S^T and dP^T halves swap roles on every use, so a step's S^T never waits and
// its dP^T waits only for gradient MMAs already queued ahead of that S^T: the
// single MMA-issuing thread never stalls on work it has just issued.
//
// Warp roles: warp 0 TMA producer (Q, dO halves plus their lse, delta and
// segment ids through a 4-stage ring), warp 1 MMA issuer and TMEM owner,
// warps 2..9 softmax: two threads per key row, 32 query columns each.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct DkvLayout {
  static constexpr int NS = 4;                           // Q/dO half-tile stages
  static constexpr uint32_t KV_BYTES = 128 * D * 2;      // one K or V tile
  static constexpr uint32_t QH_BYTES = 64 * D * 2;       // one 64-row half tile of Q or dO
  static constexpr uint32_t KV_CHUNK = 128 * 128;        // one 64-column chunk of a 128-row tile
  static constexpr uint32_t QH_CHUNK = 64 * 128;         // one 64-column chunk of a 64-row tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;
  static constexpr uint32_t OFF_DO = OFF_Q + NS * QH_BYTES;
  static constexpr uint32_t TILE_BYTES = OFF_DO + NS * QH_BYTES;
  static constexpr uint32_t MISC_BYTES = 4096;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: dV, dK accumulators, then two step buffers of 128 columns each;
  // a buffer's 64-column halves hold S^T and dP^T and swap roles on every use
  static constexpr uint32_t TM_DV = 0, TM_DK = D, TM_BUF = 2 * D, TMEM_COLS = 512;
};

struct DkvMisc {
  uint64_t kv_full, q_full[4], q_empty[4];
  uint64_t s_full[2], pds_full[2], grad_done[2], mma_final;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float lse[4][64];
  alignas(16) float dl[4][64];
  alignas(16) int32_t segq[4][64];
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const AttnParams p) {
  using L = DkvLayout<D>;
  constexpr int NS = L::NS;
  static_assert(sizeof(DkvMisc) <= L::MISC_BYTES, "misc region");
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
      mbar_init(&m.pds_full[s], 256);
      mbar_init(&m.grad_done[s], 1);
    }
    mbar_init(&m.mma_final, 1);
    fence_mbar_init();
  }
  if (!p.seg)  // every token in one segment: the query-tile ids are all 0
    for (int x = threadIdx.x; x < NS * 64; x += blockDim.x) (&m.segq[0][0])[x] = 0;
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
      mbar_expect_tx(&m.kv_full, 2 * L::KV_BYTES);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(base + L::OFF_K + c * L::KV_CHUNK, &tmK, &m.kv_full, c * 64, krow);
        tma_load_2d(base + L::OFF_V + c * L::KV_CHUNK, &tmV, &m.kv_full, c * 64, krow);
      }
      const uint32_t qbytes = 2 * L::QH_BYTES + 512 + (p.seg ? 256 : 0);
      int i = 0;
      bool ok = true;
      for (int hq = h0; ok && hq < h1; ++hq) {
        for (int tq = walk.first(); ok && tq < walk.end(); tq = walk.next(tq)) {
          for (int half = 0; half < 2; ++half, ++i) {
            const int st = i % NS;
            if (!g.wait(&m.q_empty[st], ((i / NS) & 1) ^ 1, 1)) { ok = false; break; }
            const int qrow = (b * p.Hq + hq) * p.N + tq * kTile + half * 64;
            mbar_expect_tx(&m.q_full[st], qbytes);
            for (int c = 0; c < D / 64; ++c) {
              tma_load_2d(base + L::OFF_Q + st * L::QH_BYTES + c * L::QH_CHUNK, &tmQ, &m.q_full[st], c * 64, qrow);
              tma_load_2d(base + L::OFF_DO + st * L::QH_BYTES + c * L::QH_CHUNK, &tmDO, &m.q_full[st], c * 64,
                          qrow);
            }
            bulk_load(m.lse[st], p.lse_in + qrow, 256, &m.q_full[st]);
            bulk_load(m.dl[st], p.delta + qrow, 256, &m.q_full[st]);
            if (p.seg) bulk_load(m.segq[st], p.seg + (size_t)b * p.N + tq * kTile + half * 64, 256, &m.q_full[st]);
          }
        }
      }
      g.drain(&m.kv_full, 0);
      for (int k = (i > NS ? i - NS : 0); k < i; ++k) g.drain(&m.q_full[k % NS], (k / NS) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idG = idesc_bf16_f32(128, D, false, true);
      auto issue_grad = [&](int i) -> bool {
        const int bb = i & 1, st = i % NS;
        if (!g.wait(&m.pds_full[bb], (i >> 1) & 1, 2)) return false;
        tc_fence_after();
        const uint32_t buf = tmem + L::TM_BUF + bb * 128 + (((i >> 1) & 1) ? 64 : 0);  // step i's S^T half
        const uint64_t gq = sdesc_sw128(sQ + st * L::QH_BYTES, L::QH_CHUNK, 1024);
        const uint64_t gd = sdesc_sw128(sDO + st * L::QH_BYTES, L::QH_CHUNK, 1024);
        const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // thread-half kk>>1 keeps P^T in its columns [0,16) and dS^T in [16,32)
          const uint32_t pcol = buf + (kk >> 1) * 32 + (kk & 1) * 8;
          const uint32_t acc = kk > 0 ? 1u : acc0;
          umma_bf16_ta(tmem + L::TM_DV, pcol, sdesc_add(gd, kk * 2048), idG, acc);
          umma_bf16_ta(tmem + L::TM_DK, pcol + 16, sdesc_add(gq, kk * 2048), idG, acc);
        }
        umma_commit(&m.grad_done[bb]);
        umma_commit(&m.q_empty[st]);
        return true;
      };
      const uint64_t dk0 = sdesc_sw128(sK, 16, 1024), dv0 = sdesc_sw128(sV, 16, 1024);
      bool ok = g.wait(&m.kv_full, 0, 3);
      int i = 0;
      for (int hq = h0; ok && hq < h1; ++hq) {
        for (int tq = walk.first(); ok && tq < walk.end(); tq = walk.next(tq)) {
          for (int half = 0; half < 2; ++half, ++i) {
            const int bb = i & 1, st = i % NS;
            if (!g.wait(&m.q_full[st], (i / NS) & 1, 4)) { ok = false; break; }
            // Buffer bb's two halves swap roles on every use: S^T of step i goes
            // where dP^T of step i-2 was (free once that softmax read it), dP^T
            // where step i-2's P^T/dS^T was (free once its gradient MMAs ran).
            const uint32_t buf = tmem + L::TM_BUF + bb * 128;
            const uint32_t sO = ((i >> 1) & 1) ? 64 : 0, dO_ = 64 - sO;
            const uint64_t dq0 = sdesc_sw128(sQ + st * L::QH_BYTES, 16, 1024);
            const uint64_t do0 = sdesc_sw128(sDO + st * L::QH_BYTES, 16, 1024);
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t ko = (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32;
              const uint32_t qo = (kk >> 2) * L::QH_CHUNK + (kk & 3) * 32;
              umma_bf16(buf + sO, sdesc_add(dk0, ko), sdesc_add(dq0, qo), idS, kk > 0 ? 1u : 0u);
            }
            // only now wait for step i-2's gradient MMAs: S^T of step i is queued behind them
            if (i >= 2 && !g.wait(&m.grad_done[bb], ((i - 2) >> 1) & 1, 5)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t ko = (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32;
              const uint32_t qo = (kk >> 2) * L::QH_CHUNK + (kk & 3) * 32;
              umma_bf16(buf + dO_, sdesc_add(dv0, ko), sdesc_add(do0, qo), idS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&m.s_full[bb]);
            if (i > 0 && !issue_grad(i - 1)) { ok = false; break; }
          }
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
    const int hsel = (warp - 2) >> 2;  // which 32 of the step's 64 query columns
    const int r = quarter * 32 + lane;
    const int kvidx = tk * kTile + r;
    const int32_t segk = p.seg ? p.seg[(size_t)b * p.N + kvidx] : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const int4 kt = trow[tk];
    bool ok = true;
    int i = 0;
    for (int hq = h0; ok && hq < h1; ++hq) {
      for (int tq = walk.first(); ok && tq < walk.end(); tq = walk.next(tq)) {
        const bool masked = !tile_pair_full(tq, trow[tq], tk, kt);
        for (int half = 0; half < 2; ++half, ++i) {
          const int bb = i & 1, st = i % NS;
          ok = g.wait(&m.q_full[st], (i / NS) & 1, 6);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          ok = g.wait(&m.s_full[bb], (i >> 1) & 1, 7);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sO = ((i >> 1) & 1) ? 64 : 0;
          const uint32_t buf = tmem + lane_base + L::TM_BUF + bb * 128 + sO + hsel * 32;
          const uint32_t dbuf = tmem + lane_base + L::TM_BUF + bb * 128 + (64 - sO) + hsel * 32;
          uint32_t sv[32], dp[32];
          tmem_ld32x2(buf, dbuf, sv, dp);  // this thread's S^T and dP^T columns
          const int c0 = hsel * 32;
          const int q0 = tq * kTile + half * 64 + c0;
          const float4* l4 = reinterpret_cast<const float4*>(&m.lse[st][c0]);
          const float4* d4 = reinterpret_cast<const float4*>(&m.dl[st][c0]);
          const int4* g4 = reinterpret_cast<const int4*>(&m.segq[st][c0]);
          uint32_t pw[16], dw[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 lv = l4[e4], dv = d4[e4];
            const float lz[4] = {lv.x, lv.y, lv.z, lv.w}, dz[4] = {dv.x, dv.y, dv.z, dv.w};
            float pz[4], sz[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) sz[e] = __uint_as_float(sv[e4 * 4 + e]);
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
          // P^T and dS^T go over this thread's own S^T columns
          tmem_st16x2(buf, buf + 16, pw, dw);
          tc_fence_before();
          mbar_arrive(&m.pds_full[bb]);
        }
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
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_DV + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]), __uint_as_float(v[q4 * 8 + 1]));
          w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]), __uint_as_float(v[q4 * 8 + 3]));
          w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]), __uint_as_float(v[q4 * 8 + 5]));
          w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]), __uint_as_float(v[q4 * 8 + 7]));
          vrow[(c0 >> 3) + q4] = w;
        }
        tmem_ld32(tmem + lane_base + L::TM_DK + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * sc, __uint_as_float(v[q4 * 8 + 1]) * sc);
          w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * sc, __uint_as_float(v[q4 * 8 + 3]) * sc);
          w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * sc, __uint_as_float(v[q4 * 8 + 5]) * sc);
          w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * sc, __uint_as_float(v[q4 * 8 + 7]) * sc);
          krow[(c0 >> 3) + q4] = w;
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
  if (!tmap_bf16_2d_sw128(&tq, q, D, qrows, 64) || !tmap_bf16_2d_sw128(&tdo, dout, D, qrows, 64) ||
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
