// bwd_dq.cu -- packed attention backward, dQ pass, for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row); it visits the
// same key tiles as the forward (the changelog's PACKED dQ kernel: cross-
// segment blocks skipped). Per key tile j:
//   S  = Q K^T   (TMEM, 128 columns)   P  = exp(scale * S - lse)
//   dP = dO V^T  (TMEM, 128 columns)   dS = P * (dP - delta)   (bf16, over S)
//   dQ += dS K   (TMEM accumulator, dS read straight from TMEM)
// and finally dQ *= scale. The probabilities are recomputed from the saved
// log-sum-exp (mlx-train-perf 0.5.1 README, "Flash-attention training path":
// the backward recomputes the tiles it needs from O(N) saved state).
//
// Every MMA is 128 x 128 (or 128 x D) with K = 16. Two warps issue them: one
// issues dP and S, the other dQ as soon as each tile's dS is ready, so neither
// waits behind the other's dependencies. TMEM holds dQ, one S region and two
// dP regions used by alternate key tiles; dS is written over its tile's dP.
// The softmax warps release the S region as soon as they have loaded it, and
// a dP region is needed again only two tiles later, so the next tile's S and
// dP run on the tensor core while this tile's dS is being formed. The key
// tiles' segment ids ride the K ring; a K stage is released only after dQ,
// which follows the softmax's use of them. dQ leaves through the Q tile's
// shared memory and a TMA store.
//
// Warp roles: warp 0 TMA producer (Q and dO once; K through a 3-stage ring,
// V through a 2-stage ring), warp 1 dP/S issuer and TMEM owner, warp 2 dQ
// issuer, warps 3..10 softmax: two threads per query row (TMEM lane quarter
// = warp index mod 4), 64 key columns each.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct DqLayout {
  static constexpr int NSK = 3, NSV = 2;
  static constexpr uint32_t TB = 128 * D * 2;     // one 128-row tile of Q, dO, K or V
  static constexpr uint32_t CHUNK = 128 * 128;    // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = OFF_Q + TB;
  static constexpr uint32_t OFF_K = OFF_DO + TB;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TB;
  static constexpr uint32_t TILE_BYTES = OFF_V + NSV * TB;
  static constexpr uint32_t MISC_BYTES = 2048;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: dQ accumulator, one S region, and two dP regions (128 columns each)
  // used by alternate tiles; dS is written over its tile's dP
  static constexpr uint32_t TM_DQ = 0, TM_S = 128, TM_P0 = 256, TM_P1 = 384, TMEM_COLS = 512;
  static __device__ __forceinline__ uint32_t reg_p(int j) { return (j & 1) ? TM_P1 : TM_P0; }
};

struct DqMisc {
  uint64_t q_full, k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full, s_free, ds_full[2], dq_done[2], mma_final[2];
  uint64_t o_staged;  // dQ rows written to shared memory by all softmax threads
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) int32_t segkv[3][128];
};

template <int D, int DM, bool T4>
__global__ void __launch_bounds__(352, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const __grid_constant__ CUtensorMap tmDQ, const AttnParams p) {
  using L = DqLayout<D>;
  constexpr int NSK = L::NSK, NSV = L::NSV;
  static_assert(sizeof(DqMisc) <= L::MISC_BYTES, "misc region");
  static_assert(L::SMEM <= 232448, "shared memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  DqMisc& m = *reinterpret_cast<DqMisc*>(smem_raw);
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + sizeof(DqMisc) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sDO = smem_u32(base + L::OFF_DO);
  const uint32_t sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the prologue's work list: the same order as the forward: longest key walks first, all heads of a tile together
  const int ent = p.work_q[(int)blockIdx.x / p.Hq];
  const int tq = ent % p.T, b = ent / p.T;
  const int h = (int)blockIdx.x % p.Hq, hk = h / p.G;
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
    mbar_init(&m.s_full, 1);
    mbar_init(&m.s_free, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.ds_full[s], 256);
      mbar_init(&m.dq_done[s], 1);
    }
    mbar_init(&m.mma_final[0], 1);
    mbar_init(&m.mma_final[1], 1);
    mbar_init(&m.o_staged, 256);
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
    // Lane 0 loads Q, dO and the K ring (with the key tiles' segment ids),
    // lane 1 the V ring: each ring refills as soon as its own stage is released.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmK);
      mbar_expect_tx(&m.q_full, 2 * L::TB);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_rows(base + L::OFF_Q + c * L::CHUNK, &tmQ, &m.q_full, c * 64, tq * kTile, h, b, p.Hq, p.N, T4);
        tma_load_rows(base + L::OFF_DO + c * L::CHUNK, &tmDO, &m.q_full, c * 64, tq * kTile, h, b, p.Hq, p.N, T4);
      }
      int jk = 0;
      int4 te, te_next;  // table entries of this and the next visited key tile
      for (int tk = walk.first(te), tk_next; tk <= tq; tk = tk_next, te = te_next, ++jk) {
        tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
        const int sk = jk % NSK;
        if (!g.wait(&m.k_empty[sk], ((jk / NSK) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&m.k_full[sk], L::TB + (p.seg ? 512 : 0));
        for (int c = 0; c < D / 64; ++c)
          tma_load_rows(base + L::OFF_K + sk * L::TB + c * L::CHUNK, &tmK, &m.k_full[sk], c * 64,
                        tk * kTile, hk, b, p.Hkv, p.N, T4);
        if (p.seg) bulk_load(m.segkv[sk], p.seg + (size_t)b * p.N + tk * kTile, 512, &m.k_full[sk]);
      }
      // no copy may still be landing when the CTA exits
      g.drain(&m.q_full, 0);
      for (int i = (jk > NSK ? jk - NSK : 0); i < jk; ++i) g.drain(&m.k_full[i % NSK], (i / NSK) & 1);
    } else if (lane == 1) {
      prefetch_tmap(&tmV);
      int jv = 0;
      int4 te, te_next;  // table entries of this and the next visited key tile
      for (int tk = walk.first(te), tk_next; tk <= tq; tk = tk_next, te = te_next, ++jv) {
        tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
        const int sv = jv % NSV;
        if (!g.wait(&m.v_empty[sv], ((jv / NSV) & 1) ^ 1, 2)) break;
        mbar_expect_tx(&m.v_full[sv], L::TB);
        for (int c = 0; c < D / 64; ++c)
          tma_load_rows(base + L::OFF_V + sv * L::TB + c * L::CHUNK, &tmV, &m.v_full[sv], c * 64,
                        tk * kTile, hk, b, p.Hkv, p.N, T4);
      }
      for (int i = (jv > NSV ? jv - NSV : 0); i < jv; ++i) g.drain(&m.v_full[i % NSV], (i / NSV) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ dP / S issuer
    // Per tile j: dP_j, then S_j. S_j reuses the S region that dQ_{j-2} read;
    // with dP_j issued in between, that wait never empties the tensor pipe.
    // The whole warp runs the issue loop and every wait; lane 0 alone issues
    // the tcgen05 instructions.
    const bool leader = lane == 0;
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint64_t qd = sdesc_sw128(sQ, 16, 1024), dod = sdesc_sw128(sDO, 16, 1024);
    bool ok = g.wait_warp(&m.q_full, 0, 4);
    int j = 0;
    int4 te, te_next;  // table entries of this and the next visited key tile
    for (int tk = walk.first(te), tk_next; ok && tk <= tq; tk = tk_next, te = te_next, ++j) {
      tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
      const int rs = j & 1, sk = j % NSK, sv = j % NSV;
      // dP_j into dP region rs once dQ_{j-2} has read the dS that was there
      if (!g.wait_warp(&m.v_full[sv], (j / NSV) & 1, 7)) { ok = false; break; }
      if (j >= 2 && !g.wait_warp(&m.dq_done[rs], ((j - 2) >> 1) & 1, 8)) { ok = false; break; }
      tc_fence_after();
      const uint64_t vd = sdesc_sw128(sV + sv * L::TB, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < DM / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
        if (leader) umma_bf16(tmem + L::reg_p(j), sdesc_add(dod, ko), sdesc_add(vd, ko), idS, kk > 0 ? 1u : 0u);
      }
      if (leader) umma_commit(&m.v_empty[sv]);
      __syncwarp();
      // S_j into the S region once the softmax has read S_{j-1}
      if (!g.wait_warp(&m.k_full[sk], (j / NSK) & 1, 5)) { ok = false; break; }
      if (j >= 1 && !g.wait_warp(&m.s_free, (j - 1) & 1, 6)) { ok = false; break; }
      tc_fence_after();
      const uint64_t kd = sdesc_sw128(sK + sk * L::TB, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < DM / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
        if (leader) umma_bf16(tmem + L::TM_S, sdesc_add(qd, ko), sdesc_add(kd, ko), idS, kk > 0 ? 1u : 0u);
      }
      if (leader) umma_commit(&m.s_full);  // also covers dP_j, issued before
      __syncwarp();
    }
    if (leader) {
      umma_commit(&m.mma_final[0]);
      g.drain(&m.mma_final[0], 0);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ dQ issuer
    // dQ += dS_j K_j as soon as dS_j is in TMEM: thread-half h keeps the dS of
    // its 64 key columns in columns 64h..64h+31 of the tile's dP region; K is
    // the MN-major B operand.
    const bool leader = lane == 0;
    constexpr uint32_t idQ = idesc_bf16_f32(128, DM, false, true);
    bool ok = true;
    int j = 0;
    int4 te, te_next;  // table entries of this and the next visited key tile
    for (int tk = walk.first(te), tk_next; ok && tk <= tq; tk = tk_next, te = te_next, ++j) {
      tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
      const int rs = j & 1, sk = j % NSK;
      if (!g.wait_warp(&m.k_full[sk], (j / NSK) & 1, 2)) { ok = false; break; }
      if (!g.wait_warp(&m.ds_full[rs], (j >> 1) & 1, 3)) { ok = false; break; }
      tc_fence_after();
      const uint32_t preg = tmem + L::reg_p(j);
      const uint64_t kmn = sdesc_sw128(sK + sk * L::TB, L::CHUNK, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (leader)
          umma_bf16_ta(tmem + L::TM_DQ, preg + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_add(kmn, kk * 2048), idQ,
                       (j > 0 || kk > 0) ? 1u : 0u);
      if (leader) {
        umma_commit(&m.dq_done[rs]);
        umma_commit(&m.k_empty[sk]);
      }
      __syncwarp();
    }
    if (leader) {
      umma_commit(&m.mma_final[1]);
      g.drain(&m.mma_final[1], 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int hsel = (warp - 3) >> 2;  // which 64 key columns of every tile
    const int r = quarter * 32 + lane;
    const int qidx = tq * kTile + r;
    const size_t row = (size_t)(b * p.Hq + h) * p.N + qidx;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const float lse2 = p.lse2[row];  // lse * log2(e), from the delta step
    const float dlt = p.delta[row];
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int j = 0;
    int4 te, te_next;  // table entries of this and the next visited key tile
    for (int tk = walk.first(te), tk_next; tk <= tq; tk = tk_next, te = te_next, ++j) {
      tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
      const int rs = j & 1, sk = j % NSK;
      const bool masked = !tile_pair_full(tq, walk.qt, tk, te);
      if (masked && p.seg) {  // segment ids of this key tile arrived with K
        ok = g.wait(&m.k_full[sk], (j / NSK) & 1, 9);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      ok = g.wait(&m.s_full, j & 1, 10);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      tc_fence_after();
      const uint32_t sreg = tmem + lane_base + L::TM_S + hsel * 64;
      const uint32_t preg = tmem + lane_base + L::reg_p(j) + hsel * 64;
      const int c0 = hsel * 64;
      // S (64 columns) and the first dP chunk first, so the S region is
      // released before any arithmetic; dS goes over this thread's own dP
      // columns, which have been read by then.
      uint32_t sa[32], sb[32], dpa[32];
      tmem_ld32x3(sreg, sreg + 32, preg, sa, sb, dpa);
      tc_fence_before();
      mbar_arrive(&m.s_free);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dpb[32];
        if (c == 1) tmem_ld32(preg + 32, dpb);
        uint32_t* sv = c ? sb : sa;
        const uint32_t* dp = c ? dpb : dpa;
        const int k0 = tk * kTile + c0 + 32 * c;
        if (masked) {
          const int4* g4 = reinterpret_cast<const int4*>(&m.segkv[sk][c0 + 32 * c]);
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const int4 gv = p.seg ? g4[e4] : make_int4(0, 0, 0, 0);
            const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int cc = e4 * 4 + e;
              sv[cc] = (k0 + cc <= qidx && gz[e] == segq) ? sv[cc] : __float_as_uint(-INFINITY);
            }
          }
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(sv[e]), sl2, -lse2));
          const float p1 = ex2(fmaf(__uint_as_float(sv[e + 1]), sl2, -lse2));
          w[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - dlt), p1 * (__uint_as_float(dp[e + 1]) - dlt));
        }
        tmem_st16_nowait(preg + 16 * c, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&m.ds_full[rs]);
    }
    if (ok && j > 0) {
      ok = g.wait(&m.dq_done[(j - 1) & 1], ((j - 1) >> 1) & 1, 11);
      ok = __all_sync(~0u, ok);
    }
    if (ok && j > 0) {
      tc_fence_after();
      // This thread's half of the dQ row goes into the Q tile's shared memory
      // (free: every MMA has completed), in the 128-byte-swizzled layout a TMA
      // store reads; one thread then stores the whole tile, so the writes to
      // global memory are whole 128-byte rows.
      uint8_t* so = base + L::OFF_Q;
      const float sc = p.scale;
#pragma unroll
      for (int c0 = hsel * (D / 2); c0 < (hsel + 1) * (D / 2); c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + L::TM_DQ + c0, v);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col = c0 + 8 * q4;  // first of the 8 columns in this 16-byte unit
          const uint32_t off = (col >> 6) * L::CHUNK + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4);
          st_shared_v4(smem_u32(so + off),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * sc, __uint_as_float(v[q4 * 8 + 1]) * sc),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * sc, __uint_as_float(v[q4 * 8 + 3]) * sc),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * sc, __uint_as_float(v[q4 * 8 + 5]) * sc),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * sc, __uint_as_float(v[q4 * 8 + 7]) * sc));
        }
      }
      fence_async_smem();  // these writes are read by the TMA store
      mbar_arrive(&m.o_staged);
      if (warp == 3 && lane == 0 && g.wait(&m.o_staged, 0, 12)) {
        for (int c = 0; c < D / 64; ++c) tma_store_rows(&tmDQ, so + c * L::CHUNK, c * 64, tq * kTile,
                                                        h, b, p.Hq, p.N, T4);
        bulk_commit();
        bulk_wait_all();  // the store has read shared memory (and completed) before the CTA exits
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

template <int D, int DM = D>
cudaError_t launch_dq_d(const AttnParams& p, int Dio, const RowStrides& rs, const void* q, const void* k, const void* v,
                        const void* dout, cudaStream_t st) {
  using L = DqLayout<D>;
  CUtensorMap tq, tdo, tk, tv, tdq;
  // contiguous tensors: 2-D maps over their rows (cheaper for TMA than the
  // 4-D form, which strided tensors need)
  AttnParams pp = p;
  pp.tma4 = (p.Nr == p.N && is_contiguous(rs, p.Hq, p.Hkv, p.N, Dio)) ? 0 : 1;
  const auto qmap = [&](CUtensorMap* m, const void* t) {
    return pp.tma4 ? tmap_bf16_bhnd_sw128(m, t, Dio, p.Nr, p.Hq, p.B, rs.q_n, rs.q_h, rs.q_b)
                   : tmap_bf16_2d_sw128(m, t, Dio, (uint64_t)p.B * p.Hq * p.N, 128);
  };
  const auto kmap = [&](CUtensorMap* m, const void* t) {
    return pp.tma4 ? tmap_bf16_bhnd_sw128(m, t, Dio, p.Nr, p.Hkv, p.B, rs.k_n, rs.k_h, rs.k_b)
                   : tmap_bf16_2d_sw128(m, t, Dio, (uint64_t)p.B * p.Hkv * p.N, 128);
  };
  if (!qmap(&tq, q) || !qmap(&tdo, dout) || !kmap(&tk, k) || !kmap(&tv, v) || !qmap(&tdq, p.dq))
    return cudaErrorInvalidValue;
  // the tensor maps' form is fixed at compile time: the contiguous case runs
  // exactly the 2-D code
  const auto kfn = pp.tma4 ? dq_kernel<D, DM, true> : dq_kernel<D, DM, false>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * p.Hq * p.B);
  kfn<<<grid, 352, L::SMEM, st>>>(tq, tdo, tk, tv, tdq, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k,
                          const void* v, const void* dout, cudaStream_t st) {
  // head dim 96 runs the 128-wide tile layout: its tensor maps are 96
  // elements wide, so TMA fills columns 96..127 of every loaded tile with
  // zeros and drops them from every store; the MMAs contract over 96 (six
  // K-steps) and produce 96 columns (N = 96), so no work is spent on them.
  if (D == 64) return launch_dq_d<64>(p, 64, rs, q, k, v, dout, st);
  if (D == 96) return launch_dq_d<128, 96>(p, 96, rs, q, k, v, dout, st);
  return launch_dq_d<128>(p, 128, rs, q, k, v, dout, st);
}

}  // namespace pa
