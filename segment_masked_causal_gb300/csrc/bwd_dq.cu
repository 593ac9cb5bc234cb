// bwd_dq.cu -- packed attention backward, dQ pass, for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row); it visits the
// same key tiles as the forward (the changelog's PACKED dQ kernel: cross-
// segment blocks skipped). Per key tile:
//   S  = Q K^T           (TMEM)     P  = exp(scale * S - lse)
//   dP = dO V^T          (TMEM)     dS = P * (dP - delta)      (bf16, smem)
//   dQ += dS K           (TMEM accumulator)
// and finally dQ *= scale. The probabilities are recomputed from the saved
// log-sum-exp (mlx-train-perf 0.5.1 README, "Flash-attention training path":
// the backward recomputes the tiles it needs from O(N) saved state).
//
// Warp roles as in the forward: warp 0 TMA producer, warp 1 MMA issuer and
// TMEM owner, warps 2..5 one query row per thread.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct DqLayout {
  static constexpr int NS = (D == 128) ? 2 : 3;
  static constexpr uint32_t Q_BYTES = 128 * D * 2;
  static constexpr uint32_t KV_BYTES = 128 * D * 2;
  static constexpr uint32_t DS_BYTES = 128 * 128 * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_K = OFF_DO + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NS * KV_BYTES;
  static constexpr uint32_t OFF_DS = OFF_V + NS * KV_BYTES;
  static constexpr uint32_t TILE_BYTES = OFF_DS + DS_BYTES;
  static constexpr uint32_t MISC_BYTES = 2048;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DQ = 256, TMEM_COLS = 512;
};

struct DqMisc {
  uint64_t q_full;
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full, s_empty, ds_full, dq_done, seg_ready[2];
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
  int32_t segkv[2][128];
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const AttnParams p) {
  using L = DqLayout<D>;
  constexpr int NS = L::NS;
  static_assert(sizeof(DqMisc) <= L::MISC_BYTES, "misc region");
  extern __shared__ uint8_t smem_raw[];
  DqMisc& m = *reinterpret_cast<DqMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(DqMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sDO = smem_u32(base + L::OFF_DO);
  const uint32_t sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);
  const uint32_t sDS = smem_u32(base + L::OFF_DS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tq = p.T - 1 - (int)blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z, hk = h / p.G;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    mbar_init(&m.q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&m.kv_full[s], 1);
      mbar_init(&m.kv_empty[s], 1);
    }
    mbar_init(&m.s_full, 1);
    mbar_init(&m.s_empty, 128);
    mbar_init(&m.ds_full, 128);
    mbar_init(&m.dq_done, 1);
    mbar_init(&m.seg_ready[0], 128);
    mbar_init(&m.seg_ready[1], 128);
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
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int qrow = (b * p.Hq + h) * p.N + tq * kTile;
      const int krow0 = (b * p.Hkv + hk) * p.N;
      mbar_expect_tx(&m.q_full, 2 * L::Q_BYTES);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_2d(base + L::OFF_Q + c * 16384, &tmQ, &m.q_full, c * 64, qrow);
        tma_load_2d(base + L::OFF_DO + c * 16384, &tmDO, &m.q_full, c * 64, qrow);
      }
      int j = 0;
      for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS;
        if (!g.wait(&m.kv_empty[st], ((j / NS) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&m.kv_full[st], 2 * L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_2d(base + L::OFF_K + st * L::KV_BYTES + c * 16384, &tmK, &m.kv_full[st], c * 64,
                      krow0 + tk * kTile);
          tma_load_2d(base + L::OFF_V + st * L::KV_BYTES + c * 16384, &tmV, &m.kv_full[st], c * 64,
                      krow0 + tk * kTile);
        }
      }
      g.drain(&m.q_full, 0);
      for (int i = (j > NS ? j - NS : 0); i < j; ++i) g.drain(&m.kv_full[i % NS], (i / NS) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idQ = idesc_bf16_f32(128, D, false, true);
      auto issue_dq = [&](int i) -> bool {
        const int st = i % NS;
        if (!g.wait(&m.ds_full, i & 1, 2)) return false;
        tc_fence_after();
        const uint32_t ka = sK + st * L::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + L::TM_DQ, sdesc_sw128(sDS + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(ka + kk * 2048, 16384, 1024), idQ, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&m.dq_done);
        umma_commit(&m.kv_empty[st]);
        return true;
      };
      bool ok = g.wait(&m.q_full, 0, 3);
      int j = 0;
      for (int tk = walk.first(); ok && tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS;
        ok = g.wait(&m.kv_full[st], (j / NS) & 1, 4) && g.wait(&m.s_empty, (j & 1) ^ 1, 5);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = sK + st * L::KV_BYTES, va = sV + st * L::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16(tmem + L::TM_S, sdesc_sw128(sQ + koff, 16, 1024), sdesc_sw128(ka + koff, 16, 1024), idS,
                    kk > 0 ? 1u : 0u);
          umma_bf16(tmem + L::TM_DP, sdesc_sw128(sDO + koff, 16, 1024), sdesc_sw128(va + koff, 16, 1024), idS,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(&m.s_full);
        if (j > 0) ok = issue_dq(j - 1);
      }
      if (ok && j > 0) issue_dq(j - 1);
      umma_commit(&m.mma_final);
      g.drain(&m.mma_final, 0);
    }
    __syncwarp();
  } else {
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int qidx = tq * kTile + r;
    const size_t row = (size_t)(b * p.Hq + h) * p.N + qidx;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const float lse2 = p.lse_in[row] * 1.4426950408889634f;
    const float dlt = p.delta[row];
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int j = 0;
    uint32_t nseg0 = 0, nseg1 = 0;
    for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++j) {
      const int sb = j & 1;
      // segkv[sb] was last read in tile j-2; this thread already saw dq_done
      // for tile j-2 (before writing dS in tile j-1), and that MMA needed the
      // ds_full arrivals every thread made after its tile j-2 mask reads.
      const bool masked = !tile_pair_full(tq, walk.qt, tk, trow[tk]);
      if (masked) {
        m.segkv[sb][r] = p.seg ? p.seg[(size_t)b * p.N + tk * kTile + r] : 0;
        mbar_arrive(&m.seg_ready[sb]);
        const uint32_t use = sb ? nseg1++ : nseg0++;
        ok = g.wait(&m.seg_ready[sb], use & 1, 7);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      ok = g.wait(&m.s_full, j & 1, 8);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      tc_fence_after();
      float pr[128];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_S + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = c0 + i;
          float s = __uint_as_float(v[i]);
          if (masked) {
            const bool vis = (tk * kTile + c <= qidx) && (m.segkv[sb][c] == segq);
            s = vis ? s : -INFINITY;
          }
          pr[c] = ex2(fmaf(s, sl2, -lse2));
        }
      }
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_DP + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) pr[c0 + i] = pr[c0 + i] * (__uint_as_float(v[i]) - dlt);
      }
      tc_fence_before();
      mbar_arrive(&m.s_empty);
      // the dS tile is free once the previous dQ MMA has read it
      if (j >= 1) ok = g.wait(&m.dq_done, (j - 1) & 1, 9);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
#pragma unroll
      for (int c8 = 0; c8 < 128; c8 += 8)
        st_shared_v4(sDS + sw128_offset(r, c8), pack_bf16x2(pr[c8], pr[c8 + 1]), pack_bf16x2(pr[c8 + 2], pr[c8 + 3]),
                     pack_bf16x2(pr[c8 + 4], pr[c8 + 5]), pack_bf16x2(pr[c8 + 6], pr[c8 + 7]));
      fence_async_smem();
      mbar_arrive(&m.ds_full);
    }
    if (ok && j > 0) {
      ok = g.wait(&m.dq_done, (j - 1) & 1, 10);
      ok = __all_sync(~0u, ok);
    }
    if (ok && j > 0) {
      tc_fence_after();
      uint4* drow = reinterpret_cast<uint4*>(p.dq + row * D);
      const float sc = p.scale;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
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
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t qrows = (uint64_t)p.B * p.Hq * p.N, krows = (uint64_t)p.B * p.Hkv * p.N;
  if (!tmap_bf16_2d_sw128(&tq, q, D, qrows, 128) || !tmap_bf16_2d_sw128(&tdo, dout, D, qrows, 128) ||
      !tmap_bf16_2d_sw128(&tk, k, D, krows, 128) || !tmap_bf16_2d_sw128(&tv, v, D, krows, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T, p.Hq, p.B);
  dq_kernel<D><<<grid, 192, L::SMEM, st>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                          const void* dout, cudaStream_t st) {
  return D == 128 ? launch_dq_d<128>(p, q, k, v, dout, st) : launch_dq_d<64>(p, q, k, v, dout, st);
}

}  // namespace pa
