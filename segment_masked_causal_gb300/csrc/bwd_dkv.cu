// bwd_dkv.cu -- packed attention backward, dK/dV pass, for sm_103a.
//
// One CTA per (key tile of 128 rows, kv head, batch row). It walks every query
// head of its group and, for each, the query tiles from the diagonal up to
// the last tile whose segment range overlaps the key tile's -- the query walk
// ends at the key block's segment end instead of masking the rest
// (mlx-train-perf 0.5.1 README, "Sequence packing", the 0.5.0 dK/dV change).
// Per visited (query head, query tile), with K and V resident:
//   S^T  = K Q^T   (TMEM)        P^T  = exp(scale * S^T - lse)      (bf16 smem)
//   dP^T = V dO^T  (TMEM)        dS^T = P^T * (dP^T - delta)         (bf16 smem)
//   dV += P^T dO   dK += dS^T Q  (TMEM accumulators)
// and finally dK *= scale. The group's heads are summed inside the CTA in a
// fixed order, so dK/dV need no atomics and are deterministic.
//
// Warp roles: warp 0 TMA producer (Q, dO tiles plus the query tile's lse,
// delta and segment ids), warp 1 MMA issuer and TMEM owner, warps 2..5 one
// key row per thread.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct DkvLayout {
  static constexpr int NSQ = (D == 128) ? 1 : 2;
  static constexpr uint32_t KV_BYTES = 128 * D * 2;
  static constexpr uint32_t Q_BYTES = 128 * D * 2;
  static constexpr uint32_t PT_BYTES = 128 * 128 * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + KV_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + KV_BYTES;
  static constexpr uint32_t OFF_DO = OFF_Q + NSQ * Q_BYTES;
  static constexpr uint32_t OFF_P = OFF_DO + NSQ * Q_BYTES;
  static constexpr uint32_t OFF_DS = OFF_P + PT_BYTES;
  static constexpr uint32_t TILE_BYTES = OFF_DS + PT_BYTES;
  static constexpr uint32_t MISC_BYTES = 4096;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TMEM_COLS = 512;
};

struct DkvMisc {
  uint64_t kv_full, q_full[2], q_empty[2];
  uint64_t s_full, s_empty, pds_full, grad_done, mma_final;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float lse[2][128];
  alignas(16) float dl[2][128];
  alignas(16) int32_t segq[2][128];
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const AttnParams p) {
  using L = DkvLayout<D>;
  constexpr int NSQ = L::NSQ;
  static_assert(sizeof(DkvMisc) <= L::MISC_BYTES, "misc region");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DkvMisc& m = *reinterpret_cast<DkvMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(DkvMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sDO = smem_u32(base + L::OFF_DO);
  const uint32_t sP = smem_u32(base + L::OFF_P), sDS = smem_u32(base + L::OFF_DS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // key tiles near the end of a row have the shortest causal walks: start the
  // longest ones first
  const int tk = (int)blockIdx.x;
  const int hk = blockIdx.y, b = blockIdx.z;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};
  const QWalk walk(trow, tk);
  const int h0 = hk * p.G, h1 = h0 + p.G;

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    mbar_init(&m.kv_full, 1);
    for (int s = 0; s < NSQ; ++s) {
      mbar_init(&m.q_full[s], 1);
      mbar_init(&m.q_empty[s], 1);
    }
    mbar_init(&m.s_full, 1);
    mbar_init(&m.s_empty, 128);
    mbar_init(&m.pds_full, 128);
    mbar_init(&m.grad_done, 1);
    mbar_init(&m.mma_final, 1);
    fence_mbar_init();
  }
  if (!p.seg)  // every token in one segment: the query-tile ids are all 0
    for (int x = threadIdx.x; x < 2 * 128; x += blockDim.x) (&m.segq[0][0])[x] = 0;
  if (warp == 1) {
    tmem_alloc(&m.tmem_base, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int krow = (b * p.Hkv + hk) * p.N + tk * kTile;
      mbar_expect_tx(&m.kv_full, 2 * L::KV_BYTES);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(base + L::OFF_K + c * 16384, &tmK, &m.kv_full, c * 64, krow);
        tma_load_2d(base + L::OFF_V + c * 16384, &tmV, &m.kv_full, c * 64, krow);
      }
      const uint32_t qbytes = 2 * L::Q_BYTES + 1024 + (p.seg ? 512 : 0);
      int i = 0;
      bool ok = true;
      for (int hq = h0; ok && hq < h1; ++hq) {
        for (int tq = walk.first(); tq < walk.end(); tq = walk.next(tq), ++i) {
          const int st = i % NSQ;
          if (!g.wait(&m.q_empty[st], ((i / NSQ) & 1) ^ 1, 1)) { ok = false; break; }
          const int qrow = (b * p.Hq + hq) * p.N + tq * kTile;
          mbar_expect_tx(&m.q_full[st], qbytes);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_2d(base + L::OFF_Q + st * L::Q_BYTES + c * 16384, &tmQ, &m.q_full[st], c * 64, qrow);
            tma_load_2d(base + L::OFF_DO + st * L::Q_BYTES + c * 16384, &tmDO, &m.q_full[st], c * 64, qrow);
          }
          bulk_load(m.lse[st], p.lse_in + qrow, 512, &m.q_full[st]);
          bulk_load(m.dl[st], p.delta + qrow, 512, &m.q_full[st]);
          if (p.seg) bulk_load(m.segq[st], p.seg + (size_t)b * p.N + tq * kTile, 512, &m.q_full[st]);
        }
      }
      g.drain(&m.kv_full, 0);
      for (int k = (i > NSQ ? i - NSQ : 0); k < i; ++k) g.drain(&m.q_full[k % NSQ], (k / NSQ) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idG = idesc_bf16_f32(128, D, false, true);
      auto issue_grad = [&](int i) -> bool {
        const int st = i % NSQ;
        if (!g.wait(&m.pds_full, i & 1, 2)) return false;
        tc_fence_after();
        const uint32_t qa = sQ + st * L::Q_BYTES, da = sDO + st * L::Q_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          umma_bf16(tmem + L::TM_DV, sdesc_sw128(sP + aoff, 16, 1024), sdesc_sw128(da + kk * 2048, 16384, 1024),
                    idG, acc);
          umma_bf16(tmem + L::TM_DK, sdesc_sw128(sDS + aoff, 16, 1024), sdesc_sw128(qa + kk * 2048, 16384, 1024),
                    idG, acc);
        }
        umma_commit(&m.grad_done);
        umma_commit(&m.q_empty[st]);
        return true;
      };
      bool ok = g.wait(&m.kv_full, 0, 3);
      int i = 0;
      for (int hq = h0; ok && hq < h1; ++hq) {
        for (int tq = walk.first(); tq < walk.end(); tq = walk.next(tq), ++i) {
          const int st = i % NSQ;
          if (NSQ == 1 && i > 0 && !issue_grad(i - 1)) { ok = false; break; }
          if (!g.wait(&m.q_full[st], (i / NSQ) & 1, 4) || !g.wait(&m.s_empty, (i & 1) ^ 1, 5)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qa = sQ + st * L::Q_BYTES, da = sDO + st * L::Q_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tmem + L::TM_S, sdesc_sw128(sK + koff, 16, 1024), sdesc_sw128(qa + koff, 16, 1024), idS,
                      kk > 0 ? 1u : 0u);
            umma_bf16(tmem + L::TM_DP, sdesc_sw128(sV + koff, 16, 1024), sdesc_sw128(da + koff, 16, 1024), idS,
                      kk > 0 ? 1u : 0u);
          }
          umma_commit(&m.s_full);
          if (NSQ > 1 && i > 0 && !issue_grad(i - 1)) { ok = false; break; }
        }
      }
      if (ok && i > 0) issue_grad(i - 1);
      umma_commit(&m.mma_final);
      g.drain(&m.mma_final, 0);
    }
    __syncwarp();
  } else {
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int kvidx = tk * kTile + r;
    const int32_t segk = p.seg ? p.seg[(size_t)b * p.N + kvidx] : 0;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    const int4 kt = trow[tk];
    bool ok = true;
    int i = 0;
    for (int hq = h0; ok && hq < h1; ++hq) {
      for (int tq = walk.first(); tq < walk.end(); tq = walk.next(tq), ++i) {
        const int st = i % NSQ;
        ok = g.wait(&m.q_full[st], (i / NSQ) & 1, 6);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        ok = g.wait(&m.s_full, i & 1, 7);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        tc_fence_after();
        const bool masked = !tile_pair_full(tq, trow[tq], tk, kt);
        const int qbase = tq * kTile;
        float pr[128];
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + L::TM_S + c0, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = c0 + e;
            float s = __uint_as_float(v[e]);
            if (masked) {
              const bool vis = (qbase + c >= kvidx) && (m.segq[st][c] == segk);
              s = vis ? s : -INFINITY;
            }
            pr[c] = ex2(fmaf(s, sl2, -m.lse[st][c] * 1.4426950408889634f));
          }
        }
        // P^T / dS^T tiles are free once the previous step's gradient MMAs finished
        if (i > 0) ok = g.wait(&m.grad_done, (i - 1) & 1, 8);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
#pragma unroll
        for (int c8 = 0; c8 < 128; c8 += 8)
          st_shared_v4(sP + sw128_offset(r, c8), pack_bf16x2(pr[c8], pr[c8 + 1]), pack_bf16x2(pr[c8 + 2], pr[c8 + 3]),
                       pack_bf16x2(pr[c8 + 4], pr[c8 + 5]), pack_bf16x2(pr[c8 + 6], pr[c8 + 7]));
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + L::TM_DP + c0, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) pr[c0 + e] = pr[c0 + e] * (__uint_as_float(v[e]) - m.dl[st][c0 + e]);
#pragma unroll
          for (int c8 = c0; c8 < c0 + 32; c8 += 8)
            st_shared_v4(sDS + sw128_offset(r, c8), pack_bf16x2(pr[c8], pr[c8 + 1]),
                         pack_bf16x2(pr[c8 + 2], pr[c8 + 3]), pack_bf16x2(pr[c8 + 4], pr[c8 + 5]),
                         pack_bf16x2(pr[c8 + 6], pr[c8 + 7]));
        }
        tc_fence_before();
        mbar_arrive(&m.s_empty);
        fence_async_smem();
        mbar_arrive(&m.pds_full);
      }
    }
    if (ok && i > 0) {
      ok = g.wait(&m.grad_done, (i - 1) & 1, 9);
      ok = __all_sync(~0u, ok);
    }
    if (ok && i > 0) {
      tc_fence_after();
      const size_t row = (size_t)(b * p.Hkv + hk) * p.N + kvidx;
      uint4* vrow = reinterpret_cast<uint4*>(p.dv + row * D);
      uint4* krow = reinterpret_cast<uint4*>(p.dk + row * D);
      const float sc = p.scale;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
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
  if (!tmap_bf16_2d_sw128(&tq, q, D, qrows, 128) || !tmap_bf16_2d_sw128(&tdo, dout, D, qrows, 128) ||
      !tmap_bf16_2d_sw128(&tk, k, D, krows, 128) || !tmap_bf16_2d_sw128(&tv, v, D, krows, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dkv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T, p.Hkv, p.B);
  dkv_kernel<D><<<grid, 192, L::SMEM, st>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkv(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                           const void* dout, cudaStream_t st) {
  return D == 128 ? launch_dkv_d<128>(p, q, k, v, dout, st) : launch_dkv_d<64>(p, q, k, v, dout, st);
}

}  // namespace pa
