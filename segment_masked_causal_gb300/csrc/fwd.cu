// fwd.cu -- packed (block-diagonal causal) attention forward for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row). Warp roles:
//   warp 0      TMA producer: Q once, then K/V tiles through an NS-deep ring
//   warp 1      MMA issuer (one thread): S = Q K^T into TMEM (double-buffered),
//               O += P V into a TMEM accumulator; owns the TMEM allocation
//   warps 2..5  softmax: one query row per thread, read from TMEM lane
//               32*(warp%4)+lane; online softmax in the log2 domain; P is
//               written as bf16 into a swizzled shared-memory tile that the
//               next MMA reads; epilogue O / l -> bf16, lse -> fp32
//
// The kernel visits only key tiles whose segment-id range overlaps the query
// tile's (the changelog's PACKED forward: cross-segment blocks are skipped,
// not masked) and applies the element mask (j <= i and seg[i] == seg[j]) only
// on tile pairs that are not entirely visible. The saved state is O and its
// log-sum-exp (mlx-train-perf 0.5.1 README, "Flash-attention training path").
//
// Online softmax keeps a running maximum m (log2 units of the scaled score)
// and rescales the O accumulator only when a new tile raises m by more than 8
// (a factor 256), so most tiles leave O untouched; P is always computed
// against the m in use, so O and l stay consistent and O / l is exact.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct FwdLayout {
  static constexpr int NS = (D == 128) ? 2 : 3;
  static constexpr uint32_t Q_BYTES = 128 * D * 2;
  static constexpr uint32_t KV_BYTES = 128 * D * 2;
  static constexpr uint32_t P_BYTES = 128 * 128 * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + NS * KV_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + NS * KV_BYTES;
  static constexpr uint32_t TILE_BYTES = OFF_P + 2 * P_BYTES;
  static constexpr uint32_t MISC_BYTES = 2048;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  static constexpr uint32_t TM_S0 = 0, TM_O = 256, TMEM_COLS = 512;
};

struct FwdMisc {
  uint64_t q_full;
  uint64_t k_full[3], v_full[3], kv_empty[3];
  uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
  uint64_t seg_ready[2];
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort_flag;
  int32_t segkv[2][128];
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using L = FwdLayout<D>;
  constexpr int NS = L::NS;
  static_assert(sizeof(FwdMisc) <= L::MISC_BYTES, "misc region");
  extern __shared__ uint8_t smem_raw[];
  FwdMisc& m = *reinterpret_cast<FwdMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(FwdMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sK = smem_u32(base + L::OFF_K);
  const uint32_t sV = smem_u32(base + L::OFF_V), sP = smem_u32(base + L::OFF_P);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tq = p.T - 1 - (int)blockIdx.x;  // longest causal rows first
  const int h = blockIdx.y, b = blockIdx.z, hk = h / p.G;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    mbar_init(&m.q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&m.k_full[s], 1);
      mbar_init(&m.v_full[s], 1);
      mbar_init(&m.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.s_empty[s], 128);
      mbar_init(&m.p_full[s], 128);
      mbar_init(&m.pv_done[s], 1);
      mbar_init(&m.seg_ready[s], 128);
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
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      const int qrow = (b * p.Hq + h) * p.N + tq * kTile;
      const int krow0 = (b * p.Hkv + hk) * p.N;
      mbar_expect_tx(&m.q_full, L::Q_BYTES);
      for (int c = 0; c < D / 64; ++c) tma_load_2d(base + L::OFF_Q + c * 16384, &tmQ, &m.q_full, c * 64, qrow);
      int j = 0;
      for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS;
        if (!g.wait(&m.kv_empty[st], ((j / NS) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&m.k_full[st], L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(base + L::OFF_K + st * L::KV_BYTES + c * 16384, &tmK, &m.k_full[st], c * 64,
                      krow0 + tk * kTile);
        mbar_expect_tx(&m.v_full[st], L::KV_BYTES);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(base + L::OFF_V + st * L::KV_BYTES + c * 16384, &tmV, &m.v_full[st], c * 64,
                      krow0 + tk * kTile);
      }
      // no copy may still be landing when the CTA exits
      g.drain(&m.q_full, 0);
      for (int i = (j > NS ? j - NS : 0); i < j; ++i) {
        g.drain(&m.k_full[i % NS], (i / NS) & 1);
        g.drain(&m.v_full[i % NS], (i / NS) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      auto issue_pv = [&](int i) -> bool {
        const int st = i % NS, pb = i & 1;
        if (!g.wait(&m.p_full[pb], (i >> 1) & 1, 2)) return false;
        if (!g.wait(&m.v_full[st], (i / NS) & 1, 3)) return false;
        tc_fence_after();
        const uint32_t pa = sP + pb * L::P_BYTES, va = sV + st * L::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16(tmem + L::TM_O, sdesc_sw128(pa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(va + kk * 2048, 16384, 1024), idO, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&m.pv_done[pb]);
        umma_commit(&m.kv_empty[st]);
        return true;
      };
      bool ok = g.wait(&m.q_full, 0, 4);
      int j = 0;
      for (int tk = walk.first(); ok && tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS, sb = j & 1;
        ok = g.wait(&m.k_full[st], (j / NS) & 1, 5) && g.wait(&m.s_empty[sb], ((j >> 1) & 1) ^ 1, 6);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ka = sK + st * L::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_bf16(tmem + L::TM_S0 + sb * 128, sdesc_sw128(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(ka + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), idS, kk > 0 ? 1u : 0u);
        umma_commit(&m.s_full[sb]);
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok && j > 0) issue_pv(j - 1);
      umma_commit(&m.mma_final);
      g.drain(&m.mma_final, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int qidx = tq * kTile + r;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f, lr = 0.f;
    bool ok = true;
    int j = 0;
    uint32_t nseg0 = 0, nseg1 = 0;  // completed uses of seg_ready[0/1]
    for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++j) {
      const int sb = j & 1;
      // P buffer sb (and segkv[sb]) are free once PV of tile j-2 completed
      if (j >= 2) ok = g.wait(&m.pv_done[sb], ((j - 2) >> 1) & 1, 7);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      const bool masked = !tile_pair_full(tq, walk.qt, tk, trow[tk]);
      if (masked) {
        m.segkv[sb][r] = p.seg ? p.seg[(size_t)b * p.N + tk * kTile + r] : 0;
        mbar_arrive(&m.seg_ready[sb]);
        const uint32_t use = sb ? nseg1++ : nseg0++;
        ok = g.wait(&m.seg_ready[sb], use & 1, 11);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      ok = g.wait(&m.s_full[sb], (j >> 1) & 1, 8);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_S0 + sb * 128 + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c0 + i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      mbar_arrive(&m.s_empty[sb]);
      if (masked) {
        const int kbase = tk * kTile;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const bool vis = (kbase + c <= qidx) && (m.segkv[sb][c] == segq);
          s[c] = vis ? s[c] : -INFINITY;
        }
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) mt = fmaxf(mt, s[c]);
      const float ms = mt * sl2;
      const bool need = ms > m_used + 8.f;
      if (__any_sync(~0u, need)) {
        const float m_new = fmaxf(m_used, ms);
        const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
        if (j > 0) {
          ok = g.wait(&m.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, 9);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + L::TM_O + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(tmem + lane_base + L::TM_O + c0, v);
          }
        }
        l *= alpha;
        lr *= alpha;
        m_used = m_new;
      }
      const float moff = (m_used == -INFINITY) ? 0.f : m_used;
      const uint32_t pbase = sP + sb * L::P_BYTES;
      // l sums the exact fp32 weights (for lse); lr sums the bf16-rounded
      // weights the PV product actually uses, so O / lr is a true convex
      // combination of the value rows
      float lsum = 0.f, lrsum = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < 128; c8 += 8) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float e0 = ex2(fmaf(s[c8 + 2 * i], sl2, -moff));
          const float e1 = ex2(fmaf(s[c8 + 2 * i + 1], sl2, -moff));
          lsum += e0 + e1;
          w[i] = pack_bf16x2(e0, e1);
          lrsum += __uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xFFFF0000u);
        }
        st_shared_v4(pbase + sw128_offset(r, c8), w[0], w[1], w[2], w[3]);
      }
      l += lsum;
      lr += lrsum;
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&m.p_full[sb]);
    }
    if (ok && j > 0) {
      ok = g.wait(&m.pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, 10);
      ok = __all_sync(~0u, ok);
    }
    if (ok && j > 0) {
      tc_fence_after();
      const float inv_l = 1.f / lr;
      const size_t row = (size_t)(b * p.Hq + h) * p.N + qidx;
      uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_O + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * inv_l, __uint_as_float(v[q4 * 8 + 1]) * inv_l);
          w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * inv_l, __uint_as_float(v[q4 * 8 + 3]) * inv_l);
          w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * inv_l, __uint_as_float(v[q4 * 8 + 5]) * inv_l);
          w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * inv_l, __uint_as_float(v[q4 * 8 + 7]) * inv_l);
          orow[(c0 >> 3) + q4] = w;
        }
      }
      p.lse[row] = m_used * 0.6931471805599453f + logf(l);
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
cudaError_t launch_fwd_d(const AttnParams& p, const void* q, const void* k, const void* v, cudaStream_t st) {
  using L = FwdLayout<D>;
  CUtensorMap tq, tk, tv;
  if (!tmap_bf16_2d_sw128(&tq, q, D, (uint64_t)p.B * p.Hq * p.N, 128) ||
      !tmap_bf16_2d_sw128(&tk, k, D, (uint64_t)p.B * p.Hkv * p.N, 128) ||
      !tmap_bf16_2d_sw128(&tv, v, D, (uint64_t)p.B * p.Hkv * p.N, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T, p.Hq, p.B);
  fwd_kernel<D><<<grid, 192, L::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                       cudaStream_t st) {
  return D == 128 ? launch_fwd_d<128>(p, q, k, v, st) : launch_fwd_d<64>(p, q, k, v, st);
}

}  // namespace pa
