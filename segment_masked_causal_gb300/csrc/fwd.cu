// fwd.cu -- packed (block-diagonal causal) attention forward for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row). It visits only
// key tiles whose segment-id range overlaps the query tile's (the changelog's
// PACKED forward: cross-segment blocks are skipped, not masked) and applies
// the element mask (j <= i and seg[i] == seg[j]) only on tile pairs that are
// not entirely visible. The saved state is O and its log-sum-exp
// (mlx-train-perf 0.5.1 README, "Flash-attention training path").
//
// Every key tile is split into two 64-key halves ("steps"; step i = 2 * tile +
// half). Half h of every tile goes to softmax warpgroup h, which keeps its own running maximum, sums and O
// accumulator (TMEM); the two partial results are combined once at the end:
//   O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)).
// Per half:  S_h = Q K_h^T (TMEM, 64 columns; Q resident in TMEM as the A
// operand), P_h = 2^(S_h log2e scale - m) written back as bf16 over S_h and
// fed to O_h += P_h V_h straight from TMEM. Shared memory carries only the
// K/V ring. S buffers rotate over three 64-column slots and the MMA issuer
// queues S_{i+1} before PV_i, so a slot it must wait for was freed by a PV
// issued two groups earlier and the tensor pipe never drains.
//
// Online softmax works in log2 units of the scaled score and rescales an O
// accumulator only when its running maximum rises by more than 8 (a factor
// 256); P is always computed against the maximum in use, so O and l stay
// consistent and O / l is exact in real arithmetic.
//
// Warp roles: warp 0 TMA producer (K/V ring), warp 1 MMA issuer and TMEM
// owner, warps 2..5 warpgroup 0 and warps 6..9 warpgroup 1 (one query row per
// thread in each).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct FwdLayout {
  static constexpr int NS = (D == 128) ? 3 : 4;   // K/V stages
  static constexpr uint32_t KV_BYTES = 128 * D * 2;
  static constexpr uint32_t KV_CHUNK = 128 * 128;  // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + NS * KV_BYTES;
  static constexpr uint32_t TILE_BYTES = OFF_V + NS * KV_BYTES;
  static constexpr uint32_t MISC_BYTES = 8192;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: three rotating 64-column S buffers, Q as bf16 (D/2 columns), O_0, O_1
  static constexpr uint32_t TM_S = 0, TM_Q = 192, TM_O = 256, TMEM_COLS = 512;
};

struct FwdMisc {
  uint64_t kv_full[4], kv_empty[4];
  uint64_t q_ready, s_full[3], p_full[3], pv_done[3], comb_ready, mma_final;
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) int32_t segkv[4][128];
  float mst[2][128], lst[2][128], lrst[2][128];  // per-warpgroup row statistics for the final combine
};

template <int D>
__global__ void __launch_bounds__(320, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __nv_bfloat16* __restrict__ q, const AttnParams p) {
  using L = FwdLayout<D>;
  constexpr int NS = L::NS;
  static_assert(sizeof(FwdMisc) <= L::MISC_BYTES, "misc region");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  FwdMisc& m = *reinterpret_cast<FwdMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(FwdMisc) + 1023) & ~uintptr_t(1023));
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
    mbar_init(&m.q_ready, 256);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.p_full[s], 128);
      mbar_init(&m.pv_done[s], 1);
    }
    mbar_init(&m.comb_ready, 256);
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
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      // O_w += P_w V_half for step i = 2 * tile + half (warpgroup w = half);
      // P_w sits in S slot i % 3
      auto issue_pv = [&](int i) -> bool {
        const int w = i & 1, st = (i >> 1) % NS, bi = i % 3;
        if (!g.wait(&m.p_full[bi], (i / 3) & 1, 2)) return false;
        tc_fence_after();
        const uint64_t vd = sdesc_sw128(sV + st * L::KV_BYTES + w * 64 * 128, L::KV_CHUNK, 1024);
        const uint32_t acc0 = i >= 2 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ta(tmem + L::TM_O + w * D, tmem + L::TM_S + bi * 64 + kk * 8, sdesc_add(vd, kk * 2048), idO,
                       kk > 0 ? 1u : acc0);
        umma_commit(&m.pv_done[bi]);
        if (w == 1) umma_commit(&m.kv_empty[st]);
        return true;
      };
      bool ok = g.wait(&m.q_ready, 0, 3);
      tc_fence_after();
      int i = 0, j = 0;
      for (int tk = walk.first(); ok && tk <= tq; tk = walk.next(tk), ++j) {
        const int st = j % NS;
        if (!g.wait(&m.kv_full[st], (j / NS) & 1, 4)) { ok = false; break; }
        for (int w = 0; w < 2; ++w, ++i) {
          const int bi = i % 3;
          // slot bi is free once the PV of step i-3 has read the P it held
          if (i >= 3 && !g.wait(&m.pv_done[bi], ((i - 3) / 3) & 1, 5)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kd = sdesc_sw128(sK + st * L::KV_BYTES + w * 64 * 128, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_bf16_ta(tmem + L::TM_S + bi * 64, tmem + L::TM_Q + kk * 8,
                         sdesc_add(kd, (kk >> 2) * L::KV_CHUNK + (kk & 3) * 32), idS, kk > 0 ? 1u : 0u);
          umma_commit(&m.s_full[bi]);
          // PV one step behind S: the slot S_{i+1} needs was freed by PV_{i-2},
          // issued two groups earlier, so the issuer never waits on the group
          // it has just queued
          if (i >= 1 && !issue_pv(i - 1)) { ok = false; break; }
        }
      }
      if (ok && i >= 1) ok = issue_pv(i - 1);
      umma_commit(&m.mma_final);
      g.drain(&m.mma_final, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int w = (warp - 2) >> 2;  // warpgroup: which 64-key half of every tile
    const int r = quarter * 32 + lane;
    const int qidx = tq * kTile + r;
    const size_t row = (size_t)(b * p.Hq + h) * p.N + qidx;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tO = tmem + lane_base + L::TM_O + w * D;
    const float sl2 = p.scale_log2;
    // this warpgroup's half of the query row into TMEM, as bf16 pairs
    {
      const uint32_t* qsrc = reinterpret_cast<const uint32_t*>(q + row * D) + w * (D / 4);
#pragma unroll
      for (int c0 = 0; c0 < D / 4; c0 += 16) {
        uint32_t a[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const uint4 x = __ldg(reinterpret_cast<const uint4*>(qsrc + c0 + e));
          a[e] = x.x; a[e + 1] = x.y; a[e + 2] = x.z; a[e + 3] = x.w;
        }
        tmem_st16(tmem + lane_base + L::TM_Q + w * (D / 4) + c0, a);
      }
      tc_fence_before();
      mbar_arrive(&m.q_ready);
    }
    float m_used = -INFINITY, l = 0.f, lr = 0.f;
    bool ok = true;
    int j = 0;
    for (int tk = walk.first(); tk <= tq; tk = walk.next(tk), ++j) {
      const int st = j % NS;
      const bool masked = !tile_pair_full(tq, walk.qt, tk, trow[tk]);
      if (masked && p.seg) {  // segment ids of this key tile arrived with it
        ok = g.wait(&m.kv_full[st], (j / NS) & 1, 6);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      const int i = 2 * j + w, bi = i % 3;
      const uint32_t tS = tmem + lane_base + L::TM_S + bi * 64;
      ok = g.wait(&m.s_full[bi], (i / 3) & 1, 7);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      tc_fence_after();
      float s[64];
      {
        uint32_t v0[32], v1[32];
        tmem_ld32x2(tS, tS + 32, v0, v1);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          s[e] = __uint_as_float(v0[e]);
          s[32 + e] = __uint_as_float(v1[e]);
        }
      }
      if (masked) {
        const int k0 = tk * kTile + w * 64;
        const int4* g4 = reinterpret_cast<const int4*>(&m.segkv[st][w * 64]);
#pragma unroll
        for (int e4 = 0; e4 < 16; ++e4) {
          const int4 gv = p.seg ? g4[e4] : make_int4(0, 0, 0, 0);
          const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = e4 * 4 + e;
            s[c] = (k0 + c <= qidx && gz[e] == segq) ? s[c] : -INFINITY;
          }
        }
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < 64; ++e) mx4[e & 3] = fmaxf(mx4[e & 3], s[e]);
      const float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float ms = mt * sl2;
      if (__any_sync(~0u, ms > m_used + 8.f)) {
        const float m_new = fmaxf(m_used, ms);
        const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
        if (j > 0) {  // O_w holds earlier tiles: rescale it once their PV is done
          ok = g.wait(&m.pv_done[(i - 2) % 3], ((i - 2) / 3) & 1, 8);
          if (!__all_sync(~0u, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
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
      uint32_t lo[16], hi[16];
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        const float e0 = ex2(fmaf(s[e], sl2, -moff));
        const float e1 = ex2(fmaf(s[e + 1], sl2, -moff));
        const uint32_t x = pack_bf16x2(e0, e1);
        ls4[(e >> 1) & 3] += e0 + e1;
        lr4[(e >> 1) & 3] += __uint_as_float(x << 16) + __uint_as_float(x & 0xFFFF0000u);
        if (e < 32) lo[e >> 1] = x; else hi[(e - 32) >> 1] = x;
      }
      l += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      lr += (lr4[0] + lr4[1]) + (lr4[2] + lr4[3]);
      tmem_st16x2(tS, tS + 16, lo, hi);  // P_w over the first 32 columns of this row's S slot
      tc_fence_before();
      mbar_arrive(&m.p_full[bi]);
    }
    // ------------------------------------------------------------ combine + epilogue
    if (ok && j > 0) {
      const int il = 2 * (j - 1) + w;
      ok = g.wait(&m.pv_done[il % 3], (il / 3) & 1, 9);
      ok = __all_sync(~0u, ok);
    }
    if (ok) {
      m.mst[w][r] = m_used;
      m.lst[w][r] = l;
      m.lrst[w][r] = lr;
      mbar_arrive(&m.comb_ready);
      ok = g.wait(&m.comb_ready, 0, 10);
      ok = __all_sync(~0u, ok);
    }
    if (ok && j > 0) {
      tc_fence_after();
      // both threads of a row evaluate the same expressions in the same order
      const float m0 = m.mst[0][r], m1 = m.mst[1][r];
      const float mx = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mx);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mx);
      const float lsum = m.lst[0][r] * f0 + m.lst[1][r] * f1;
      const float inv = 1.f / (m.lrst[0][r] * f0 + m.lrst[1][r] * f1);
      const float g0 = f0 * inv, g1 = f1 * inv;
      uint4* orow = reinterpret_cast<uint4*>(p.out + row * D);
      const uint32_t tO0 = tmem + lane_base + L::TM_O, tO1 = tO0 + D;
#pragma unroll
      for (int c0 = w * (D / 2); c0 < (w + 1) * (D / 2); c0 += 32) {
        uint32_t a[32], bb[32];
        tmem_ld32(tO0 + c0, a);
        tmem_ld32(tO1 + c0, bb);
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
  CUtensorMap tk, tv;
  const uint64_t krows = (uint64_t)p.B * p.Hkv * p.N;
  if (!tmap_bf16_2d_sw128(&tk, k, D, krows, 128) || !tmap_bf16_2d_sw128(&tv, v, D, krows, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * p.Hq * p.B);
  fwd_kernel<D><<<grid, 320, L::SMEM, st>>>(tk, tv, static_cast<const __nv_bfloat16*>(q), p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                       cudaStream_t st) {
  return D == 128 ? launch_fwd_d<128>(p, q, k, v, st) : launch_fwd_d<64>(p, q, k, v, st);
}

}  // namespace pa
