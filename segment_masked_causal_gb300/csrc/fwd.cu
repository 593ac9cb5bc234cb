// fwd.cu -- packed (block-diagonal causal) attention forward for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row). It visits only
// key tiles whose segment-id range overlaps the query tile's (the changelog's
// PACKED forward: cross-segment blocks are skipped, not masked) and applies
// the element mask (j <= i and seg[i] == seg[j]) only on tile pairs that are
// not entirely visible. The saved state is O and its log-sum-exp
// (mlx-train-perf 0.5.1 README, "Flash-attention training path").
//
// The visited key tiles alternate between two softmax warpgroups: warpgroup w
// takes tiles w, w+2, w+4, ... and keeps its own S buffer, running maximum,
// sums and O accumulator in TMEM; the two partial results are combined once
// at the end:
//   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)).
// Per tile: S = Q K^T (128 x 128, Q and K in shared memory), P = 2^(S log2e
// scale - m) written back as bf16 over S and fed to O += P V straight from
// TMEM. Every MMA is at least 128 x D x 16. Each warpgroup has its own
// MMA-issuing warp, so while one warpgroup computes its P the tensor core
// runs the other warpgroup's PV and S.
//
// Online softmax works in log2 units of the scaled score and rescales an O
// accumulator only when its running maximum rises by more than 8 (a factor
// 256); P is always computed against the maximum in use, so O and l stay
// consistent and O / l is exact in real arithmetic.
//
// Warp roles: warp 0 TMA producer (Q once; K through a 3-stage ring, V and
// the key tile's segment ids through a 2-stage ring), warps 1 and 2 the MMA
// issuers of warpgroups 0 and 1 (warp 1 also owns TMEM), warps 3..6
// warpgroup 0 and warps 7..10 warpgroup 1 (one query row per thread in each;
// TMEM lane quarter = warp index mod 4).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct FwdLayout {
  static constexpr int NSK = 3, NSV = 2;
  static constexpr uint32_t TB = 128 * D * 2;   // one 128-row tile of Q, K or V
  static constexpr uint32_t CHUNK = 128 * 128;  // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TB;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TB;
  static constexpr uint32_t TILE_BYTES = OFF_V + NSV * TB;
  static constexpr uint32_t MISC_BYTES = 8192;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: S_0, S_1 (128 columns each), O_0 at 256, O_1 at 384 (D columns each)
  static constexpr uint32_t TM_S = 0, TM_O = 256, TMEM_COLS = 512;
};

struct FwdMisc {
  uint64_t q_full, k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], comb_ready, mma_final[2];
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) int32_t segkv[2][128];
  float mst[2][128], lst[2][128], lrst[2][128];  // per-warpgroup row statistics for the final combine
};

template <int D>
__global__ void __launch_bounds__(352, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using L = FwdLayout<D>;
  constexpr int NSK = L::NSK, NSV = L::NSV;
  static_assert(sizeof(FwdMisc) <= L::MISC_BYTES, "misc region");
  static_assert(L::SMEM <= 232448, "shared memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  FwdMisc& m = *reinterpret_cast<FwdMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(FwdMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // longest causal rows first, across all heads and batch rows
  const int per_tile = p.Hq * p.B;
  const int tq = p.T - 1 - (int)blockIdx.x / per_tile;
  const int h = (int)blockIdx.x % p.Hq, b = ((int)blockIdx.x / p.Hq) % p.B, hk = h / p.G;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    mbar_init(&m.q_full, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&m.k_full[s], 1);
      mbar_init(&m.k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&m.v_full[s], 1);
      mbar_init(&m.v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.p_full[s], 128);
      mbar_init(&m.pv_done[s], 1);
    }
    mbar_init(&m.comb_ready, 256);
    mbar_init(&m.mma_final[0], 1);
    mbar_init(&m.mma_final[1], 1);
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
      mbar_expect_tx(&m.q_full, L::TB);
      for (int c = 0; c < D / 64; ++c) tma_load_2d(base + L::OFF_Q + c * L::CHUNK, &tmQ, &m.q_full, c * 64, qrow);
      int jk = 0, jv = 0;
      for (int tk = walk.first(); tk <= tq; tk = walk.next(tk)) {
        const int sk = jk % NSK, sv = jv % NSV;
        if (!g.wait(&m.k_empty[sk], ((jk / NSK) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&m.k_full[sk], L::TB);
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(base + L::OFF_K + sk * L::TB + c * L::CHUNK, &tmK, &m.k_full[sk], c * 64, krow0 + tk * kTile);
        ++jk;
        if (!g.wait(&m.v_empty[sv], ((jv / NSV) & 1) ^ 1, 2)) break;
        mbar_expect_tx(&m.v_full[sv], L::TB + (p.seg ? 512 : 0));
        for (int c = 0; c < D / 64; ++c)
          tma_load_2d(base + L::OFF_V + sv * L::TB + c * L::CHUNK, &tmV, &m.v_full[sv], c * 64, krow0 + tk * kTile);
        if (p.seg) bulk_load(m.segkv[sv], p.seg + (size_t)b * p.N + tk * kTile, 512, &m.v_full[sv]);
        ++jv;
      }
      // no copy may still be landing when the CTA exits
      g.drain(&m.q_full, 0);
      for (int i = (jk > NSK ? jk - NSK : 0); i < jk; ++i) g.drain(&m.k_full[i % NSK], (i / NSK) & 1);
      for (int i = (jv > NSV ? jv - NSV : 0); i < jv; ++i) g.drain(&m.v_full[i % NSV], (i / NSV) & 1);
    }
    __syncwarp();
  } else if (warp <= 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues warpgroup 0's tiles and warp 2 warpgroup 1's, each in its
    // own order: while one waits for its PV to finish reading P before the
    // next S may overwrite that buffer, the other keeps the tensor pipe fed.
    // The whole warp runs the issue loop and every wait; lane 0 alone issues
    // the tcgen05 instructions.
    const int w = warp - 1;
    const bool leader = lane == 0;
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
    const uint64_t qd = sdesc_sw128(sQ, 16, 1024);
    const int n = walk.count();
    // S_j = Q K_j^T into this warpgroup's S buffer
    auto issue_s = [&](int j) -> bool {
      const int sk = j % NSK;
      if (!g.wait_warp(&m.k_full[sk], (j / NSK) & 1, 3)) return false;
      tc_fence_after();
      const uint64_t kd = sdesc_sw128(sK + sk * L::TB, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
        if (leader) umma_bf16(tmem + L::TM_S + w * 128, sdesc_add(qd, ko), sdesc_add(kd, ko), idS, kk > 0 ? 1u : 0u);
      }
      if (leader) {
        umma_commit(&m.s_full[w]);
        umma_commit(&m.k_empty[sk]);
      }
      __syncwarp();
      return true;
    };
    bool ok = g.wait_warp(&m.q_full, 0, 4);
    if (ok && w < n) ok = issue_s(w);
    for (int j = w; ok && j < n; j += 2) {
      const int sv = j % NSV;  // == w: each warpgroup has its own V stage
      // O_w += P_j V_j, P_j read from this warpgroup's S buffer
      if (!g.wait_warp(&m.p_full[w], (j >> 1) & 1, 5) || !g.wait_warp(&m.v_full[sv], (j / NSV) & 1, 6)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t vd = sdesc_sw128(sV + sv * L::TB, L::CHUNK, 1024);
      const uint32_t acc0 = j >= 2 ? 1u : 0u;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (leader)
          umma_bf16_ta(tmem + L::TM_O + w * 128, tmem + L::TM_S + w * 128 + kk * 8, sdesc_add(vd, kk * 2048), idO,
                       kk > 0 ? 1u : acc0);
      if (leader) {
        umma_commit(&m.pv_done[w]);
        umma_commit(&m.v_empty[sv]);
      }
      __syncwarp();
      // S_{j+2} reuses this S buffer: wait for the PV just queued to read P_j
      if (j + 2 < n) {
        if (!g.wait_warp(&m.pv_done[w], (j >> 1) & 1, 7)) { ok = false; break; }
        ok = issue_s(j + 2);
      }
    }
    if (leader) {
      umma_commit(&m.mma_final[w]);
      g.drain(&m.mma_final[w], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int w = (warp - 3) >> 2;  // warpgroup: takes every other visited key tile
    const int r = quarter * 32 + lane;
    const int qidx = tq * kTile + r;
    const size_t row = (size_t)(b * p.Hq + h) * p.N + qidx;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + lane_base + L::TM_S + w * 128;
    const uint32_t tO = tmem + lane_base + L::TM_O + w * 128;
    const float sl2 = p.scale_log2;
    const int n = walk.count();
    float m_used = -INFINITY, l = 0.f, lr = 0.f;
    bool ok = true;
    int jj = 0, mine = 0, jlast = -1;
    for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++jj) {
      if ((jj & 1) != w) continue;
      const bool masked = !tile_pair_full(tq, walk.qt, tk, trow[tk]);
      if (masked && p.seg) {  // segment ids of this key tile arrived with V
        ok = g.wait(&m.v_full[jj % NSV], (jj / NSV) & 1, 8);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      ok = g.wait(&m.s_full[w], (jj >> 1) & 1, 9);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      tc_fence_after();
      // Two passes over S in TMEM (the row never sits in registers whole):
      // pass 1 finds the row maximum, pass 2 forms P. Both walk the 128 keys
      // as four 32-column chunks in rolled loops: instruction fetch, not
      // arithmetic, limits these warps, so the code must stay small.
      const int k0 = tk * kTile;
      const int4* g4 = reinterpret_cast<const int4*>(&m.segkv[jj % NSV][0]);
      auto load32 = [&](int c, uint32_t (&x)[32]) {
        tmem_ld32(tS + 32 * c, x);
        if (masked) {
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int4 gv = p.seg ? g4[c * 8 + e4] : make_int4(0, 0, 0, 0);
            const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = e4 * 4 + e;
              x[cc] = (k0 + 32 * c + cc <= qidx && gz[e] == segq) ? x[cc] : __float_as_uint(-INFINITY);
            }
          }
        }
      };
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t x[32];
        load32(c, x);
#pragma unroll
        for (int e = 0; e < 32; ++e) mx4[e & 3] = fmaxf(mx4[e & 3], __uint_as_float(x[e]));
      }
      const float ms = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * sl2;
      if (__any_sync(~0u, ms > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, ms);
        const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
        if (mine > 0) {  // O_w holds earlier tiles: rescale it once their PV is done
          ok = g.wait(&m.pv_done[w], ((jj - 2) >> 1) & 1, 10);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tO + c0, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st32(tO + c0, v);
          }
        }
        l *= alpha;
        lr *= alpha;
        m_used = m_new;
      }
      const float moff = (m_used == -INFINITY) ? 0.f : m_used;
      // l sums the exact fp32 weights (for lse); lr sums the bf16-rounded
      // weights the PV product uses, so O / lr is a convex combination
      float ls4[4] = {0.f, 0.f, 0.f, 0.f}, lr4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {  // 32 keys -> 16 packed columns, over S columns already read
        uint32_t x[32];
        load32(c, x);
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float e0 = ex2(fmaf(__uint_as_float(x[e]), sl2, -moff));
          const float e1 = ex2(fmaf(__uint_as_float(x[e + 1]), sl2, -moff));
          const uint32_t y = pack_bf16x2(e0, e1);
          ls4[(e >> 1) & 3] += e0 + e1;
          lr4[(e >> 1) & 3] += __uint_as_float(y << 16) + __uint_as_float(y & 0xFFFF0000u);
          pw[e >> 1] = y;
        }
        tmem_st16_nowait(tS + 16 * c, pw);
      }
      tmem_wait_st();
      l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      lr += (lr4[0] + lr4[1]) + (lr4[2] + lr4[3]);
      tc_fence_before();
      mbar_arrive(&m.p_full[w]);
      ++mine;
      jlast = jj;
    }
    // ------------------------------------------------------------ combine + epilogue
    if (ok && mine > 0) {
      ok = g.wait(&m.pv_done[w], (jlast >> 1) & 1, 11);
      ok = __all_sync(~0u, ok);
    }
    if (ok) {
      m.mst[w][r] = m_used;
      m.lst[w][r] = l;
      m.lrst[w][r] = lr;
      mbar_arrive(&m.comb_ready);
      ok = g.wait(&m.comb_ready, 0, 12);
      ok = __all_sync(~0u, ok);
    }
    if (ok) {
      tc_fence_after();
      const bool has1 = n > 1;  // warpgroup 1 saw at least one tile
      // both threads of a row evaluate the same expressions in the same order
      const float m0 = m.mst[0][r], m1 = has1 ? m.mst[1][r] : -INFINITY;
      const float mx = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mx);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mx);
      const float l0 = m.lst[0][r], l1 = has1 ? m.lst[1][r] : 0.f;
      const float r0 = m.lrst[0][r], r1 = has1 ? m.lrst[1][r] : 0.f;
      const float lsum = l0 * f0 + l1 * f1;
      const float inv = 1.f / (r0 * f0 + r1 * f1);
      const float g0 = f0 * inv, g1 = f1 * inv;
      uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
      const uint32_t tO0 = tmem + lane_base + L::TM_O, tO1 = tO0 + 128;
#pragma unroll
      for (int c0 = w * (D / 2); c0 < (w + 1) * (D / 2); c0 += 32) {
        uint32_t a[32], bb[32];
        if (has1) {
          tmem_ld32x2(tO0 + c0, tO1 + c0, a, bb);
        } else {
          tmem_ld32(tO0 + c0, a);
#pragma unroll
          for (int e = 0; e < 32; ++e) bb[e] = 0u;
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = __uint_as_float(a[q4 * 8 + e]) * g0 + __uint_as_float(bb[q4 * 8 + e]) * g1;
          uint4 x;
          x.x = pack_bf16x2(o[0], o[1]);
          x.y = pack_bf16x2(o[2], o[3]);
          x.z = pack_bf16x2(o[4], o[5]);
          x.w = pack_bf16x2(o[6], o[7]);
          orow[(c0 >> 3) + q4] = x;
        }
      }
      if (w == 0) p.lse[row] = mx * 0.6931471805599453f + logf(lsum);
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
  const uint64_t qrows = (uint64_t)p.B * p.Hq * p.N, krows = (uint64_t)p.B * p.Hkv * p.N;
  if (!tmap_bf16_2d_sw128(&tq, q, D, qrows, 128) || !tmap_bf16_2d_sw128(&tk, k, D, krows, 128) ||
      !tmap_bf16_2d_sw128(&tv, v, D, krows, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * p.Hq * p.B);
  fwd_kernel<D><<<grid, 352, L::SMEM, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                       cudaStream_t st) {
  return D == 128 ? launch_fwd_d<128>(p, q, k, v, st) : launch_fwd_d<64>(p, q, k, v, st);
}

}  // namespace pa
