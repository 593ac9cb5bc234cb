// bwd_dkv.cu -- packed attention backward, dK/dV pass, for sm_103a.
//
// One CTA per (key tile of 128 rows, kv head, batch row). It walks every query
// head of its group and, for each, the query tiles from the diagonal up to
// the last tile whose segment range overlaps the key tile's -- the query walk
// ends at the key block's segment end instead of masking the rest
// (mlx-train-perf 0.5.1 README, "Sequence packing", the 0.5.0 dK/dV change).
// Per visited (query head, query tile) step i, with K and V resident in
// shared memory:
//   S^T_i  = K Q_i^T   (TMEM)   P^T_i  = exp(scale * S^T_i - lse)   (rounded to bf16)
//   dP^T_i = V dO_i^T  (TMEM)   dS^T_i = P^T_i * (dP^T_i - delta)
//   dV += P^T_i dO_i   dK += dS^T_i Q_i
// and finally dK *= scale. P^T_i and dS^T_i are written back as bf16 over
// S^T_i and fed to the gradient MMAs straight from TMEM. The group's heads are
// summed inside the CTA in a fixed order, so dK/dV need no atomics and are
// deterministic.
//
// Thread slice h of a key row keeps P^T of its 32 query columns in packed
// columns 32h..32h+15 of step i's S region and dS^T in 32h+16..32h+31.
//
// TMEM holds the dV and dK accumulators and two 128-column regions whose roles
// swap every step: S^T_{i+1} goes where dP^T_i was as soon as the softmax
// warps have read dP^T_i, and dP^T_{i+1} goes where P^T_i/dS^T_i were once
// the gradient MMAs of step i have read them.
//
// Two warps issue MMAs, each in its own order, so neither waits behind the
// other's dependencies: one issues S^T_i and dP^T_i (looking ahead), the
// other dV_i as soon as P^T_i is ready and dK_i once dS^T_i is. The
// softmax warps run each step in two phases: phase A turns S^T_i into P^T_i,
// phase B reads dP^T_i (releasing its region) and forms dS^T_i. Q rides a
// 3-stage ring (with the step's lse) because each Q tile is read twice a step
// apart (by S^T_i and by dK_i); dO rides a 2-stage ring with the step's
// delta vector, and a dO stage is released by the dP^T and dV products and by
// the softmax once phase B has read delta. dK and dV leave through the K and
// V tiles' shared memory and TMA stores.
//
// Warp roles: warp 0 TMA producer (lane 0 the Q ring, lane 1 the dO ring),
// warp 1 issues S^T/dP^T and owns TMEM, warp 2 issues dV/dK, warps 3..18
// softmax: four threads per key row (TMEM lane quarter = warp index mod 4),
// 32 query columns each. Nothing in a step reduces along a row, so the
// columns split freely; sixteen warps hide the TMEM-load, exponential and
// barrier latencies of the two phases better than eight did.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

constexpr int kDkvThreads = 608;  // warps 3..18 softmax: four threads per key row
constexpr int kQStages = 3, kDoStages = 2;

struct DkvMisc {
  uint64_t kv_full;
  uint64_t q_full[kQStages], q_empty[kQStages];
  uint64_t do_full[kDoStages], do_empty[kDoStages];
  uint64_t s_full[2], dp_full[2], p_full[2], dp_free[2], ds_full[2], grad_done[2];
  uint64_t final_sd, final_grad;
  uint64_t o_staged;  // dK and dV rows written to shared memory by all softmax threads
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) float lse[kQStages][128];
  alignas(16) float dl[kDoStages][128];
};

template <int D>
struct DkvLayout {
  static constexpr uint32_t TB = 128 * D * 2;    // one 128-row tile of K, V, Q or dO
  static constexpr uint32_t CHUNK = 128 * 128;   // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TB;
  static constexpr uint32_t OFF_Q = OFF_V + TB;
  static constexpr uint32_t OFF_DO = OFF_Q + kQStages * TB;
  static constexpr uint32_t OFF_MISC = OFF_DO + kDoStages * TB;
  static constexpr uint32_t SMEM = OFF_MISC + (uint32_t)((sizeof(DkvMisc) + 127) & ~size_t(127));
  // TMEM: dV, dK accumulators (D columns each), then the two step regions
  static constexpr uint32_t TM_DV = 0, TM_DK = D, TM_X = 256, TM_Y = 384, TMEM_COLS = 512;
  // region holding S^T_i (then P^T_i and dS^T_i), and the one holding dP^T_i
  static __device__ __forceinline__ uint32_t reg_s(int i) { return (i & 1) ? TM_Y : TM_X; }
  static __device__ __forceinline__ uint32_t reg_dp(int i) { return (i & 1) ? TM_X : TM_Y; }
};

template <int D, int DM, bool T4>
__global__ void __launch_bounds__(kDkvThreads, 1)
    dkv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
               const AttnParams p) {
  using L = DkvLayout<D>;
  static_assert(L::SMEM <= 232448, "shared memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The 128-byte-swizzled tiles sit at fixed offsets from the start of dynamic
  // shared memory, which must therefore be 1 KiB aligned; otherwise do nothing.
  if (smem_u32_runtime(smem_raw) & 1023u) {
    if (threadIdx.x == 0 && p.status) atomicOr(p.status, PA_DEVERR_SMEM);
    return;
  }
  uint8_t* base = smem_raw;
  DkvMisc& m = *reinterpret_cast<DkvMisc*>(base + L::OFF_MISC);
  const uint32_t sK = smem_u32(base + L::OFF_K), sV = smem_u32(base + L::OFF_V);
  const uint32_t sQ = smem_u32(base + L::OFF_Q), sDO = smem_u32(base + L::OFF_DO);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the prologue's work list: longest query walks first, all kv heads of a tile together
  const int ent = p.work_k[(int)blockIdx.x / p.Hkv];
  const int tk = ent % p.T, b = ent / p.T;
  const int hk = (int)blockIdx.x % p.Hkv;
  const int4* trow = p.tiles + (size_t)b * p.T;
  const Guard g{&m.abort_flag, p.status};
  const QWalk walk(trow, tk);
  const int h0 = hk * p.G, h1 = h0 + p.G;

  if (threadIdx.x == 0) {
    m.abort_flag = 0;
    mbar_init(&m.kv_full, 1);
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(&m.q_full[s], 1);
      mbar_init(&m.q_empty[s], 1);
    }
    for (int s = 0; s < kDoStages; ++s) {
      mbar_init(&m.do_full[s], 1);
      // released by the dP^T and dV MMAs and by the softmax threads once
      // phase B has read the stage's delta vector
      mbar_init(&m.do_empty[s], 2 + 512);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.dp_full[s], 1);
      mbar_init(&m.p_full[s], 512);
      mbar_init(&m.dp_free[s], 512);
      mbar_init(&m.ds_full[s], 512);
      mbar_init(&m.grad_done[s], 1);
    }
    mbar_init(&m.final_sd, 1);
    mbar_init(&m.final_grad, 1);
    mbar_init(&m.o_staged, 512);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 loads K, V and the Q ring (with lse), lane 1 the dO ring (with
    // delta): each ring refills as soon as its own stage is released.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_expect_tx(&m.kv_full, 2 * L::TB);
      for (int c = 0; c < D / 64; ++c) {
        tma_load_rows(base + L::OFF_K + c * L::CHUNK, &tmK, &m.kv_full, c * 64, tk * kTile, hk, b, p.Hkv, p.N, T4);
        tma_load_rows(base + L::OFF_V + c * L::CHUNK, &tmV, &m.kv_full, c * 64, tk * kTile, hk, b, p.Hkv, p.N, T4);
      }
      int i = 0;
      bool ok = true;
      for (int hq = h0; ok && hq < h1; ++hq) {
        int4 te = walk.kt, te_next;  // table entries of this and the next visited query tile
        for (int tq = walk.first(), tq_next; tq < walk.end(); tq = tq_next, te = te_next, ++i) {
          tq_next = walk.next(tq, te_next);  // loaded now, used after this tile's work
          const int qs = i % kQStages;
          const int qrow = (b * p.Hq + hq) * p.N + tq * kTile;
          if (!g.wait(&m.q_empty[qs], ((i / kQStages) & 1) ^ 1, 1)) { ok = false; break; }
          mbar_expect_tx(&m.q_full[qs], L::TB + 512);
          for (int c = 0; c < D / 64; ++c)
            tma_load_rows(base + L::OFF_Q + qs * L::TB + c * L::CHUNK, &tmQ, &m.q_full[qs], c * 64,
                          tq * kTile, hq, b, p.Hq, p.N, T4);
          bulk_load(m.lse[qs], p.lse2 + qrow, 512, &m.q_full[qs]);  // lse * log2(e), from the delta step
        }
      }
      // no copy may still be landing when the CTA exits
      g.drain(&m.kv_full, 0);
      for (int k = (i > kQStages ? i - kQStages : 0); k < i; ++k) g.drain(&m.q_full[k % kQStages], (k / kQStages) & 1);
    } else if (lane == 1) {
      prefetch_tmap(&tmDO);
      int i = 0;
      bool ok = true;
      for (int hq = h0; ok && hq < h1; ++hq) {
        int4 te = walk.kt, te_next;  // table entries of this and the next visited query tile
        for (int tq = walk.first(), tq_next; tq < walk.end(); tq = tq_next, te = te_next, ++i) {
          tq_next = walk.next(tq, te_next);  // loaded now, used after this tile's work
          const int ds = i % kDoStages;
          const int qrow = (b * p.Hq + hq) * p.N + tq * kTile;
          if (!g.wait(&m.do_empty[ds], ((i / kDoStages) & 1) ^ 1, 2)) { ok = false; break; }
          mbar_expect_tx(&m.do_full[ds], L::TB + 512);
          for (int c = 0; c < D / 64; ++c)
            tma_load_rows(base + L::OFF_DO + ds * L::TB + c * L::CHUNK, &tmDO, &m.do_full[ds], c * 64,
                          tq * kTile, hq, b, p.Hq, p.N, T4);
          bulk_load(m.dl[ds], p.delta + qrow, 512, &m.do_full[ds]);
        }
      }
      for (int k = (i > kDoStages ? i - kDoStages : 0); k < i; ++k)
        g.drain(&m.do_full[k % kDoStages], (k / kDoStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ S^T / dP^T issuer
    // The whole warp runs the issue loop and every wait; lane 0 alone issues
    // the tcgen05 instructions.
    const bool leader = lane == 0;
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint64_t kd = sdesc_sw128(sK, 16, 1024), vd = sdesc_sw128(sV, 16, 1024);
    bool ok = g.wait_warp(&m.kv_full, 0, 3);
    int i = 0;
    for (int hq = h0; ok && hq < h1; ++hq) {
      int4 te = walk.kt, te_next;  // table entries of this and the next visited query tile
      for (int tq = walk.first(), tq_next; tq < walk.end(); tq = tq_next, te = te_next, ++i) {
        tq_next = walk.next(tq, te_next);  // loaded now, used after this tile's work
        const int qs = i % kQStages, ds = i % kDoStages;
        if (!g.wait_warp(&m.q_full[qs], (i / kQStages) & 1, 4)) { ok = false; break; }
        // S^T_i where dP^T_{i-1} was: free once the softmax has read it
        if (i >= 1 && !g.wait_warp(&m.dp_free[(i - 1) & 1], ((i - 1) >> 1) & 1, 5)) { ok = false; break; }
        tc_fence_after();
        const uint64_t qd = sdesc_sw128(sQ + qs * L::TB, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DM / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
          if (leader) umma_bf16(tmem + L::reg_s(i), sdesc_add(kd, ko), sdesc_add(qd, ko), idS, kk > 0 ? 1u : 0u);
        }
        if (leader) umma_commit(&m.s_full[i & 1]);
        __syncwarp();
        // dP^T_i where P^T_{i-1}/dS^T_{i-1} were: free once their MMAs ran
        if (!g.wait_warp(&m.do_full[ds], (i / kDoStages) & 1, 6)) { ok = false; break; }
        if (i >= 1 && !g.wait_warp(&m.grad_done[(i - 1) & 1], ((i - 1) >> 1) & 1, 7)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dod = sdesc_sw128(sDO + ds * L::TB, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DM / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
          if (leader) umma_bf16(tmem + L::reg_dp(i), sdesc_add(vd, ko), sdesc_add(dod, ko), idS, kk > 0 ? 1u : 0u);
        }
        if (leader) {
          umma_commit(&m.dp_full[i & 1]);
          umma_commit(&m.do_empty[ds]);
        }
        __syncwarp();
      }
    }
    if (leader) {
      umma_commit(&m.final_sd);
      g.drain(&m.final_sd, 0);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ dV / dK issuer
    // thread slice h keeps P^T of its 32 query columns in columns 32h..32h+15
    // of step j's S region and dS^T in columns 32h+16..32h+31
    const bool leader = lane == 0;
    constexpr uint32_t idG = idesc_bf16_f32(128, DM, false, true);
    bool ok = true;
    int j = 0;
    for (int hq = h0; ok && hq < h1; ++hq) {
      int4 te = walk.kt, te_next;  // table entries of this and the next visited query tile
      for (int tq = walk.first(), tq_next; tq < walk.end(); tq = tq_next, te = te_next, ++j) {
        tq_next = walk.next(tq, te_next);  // loaded now, used after this tile's work
        const int qs = j % kQStages, ds = j % kDoStages;
        const uint32_t sreg = tmem + L::reg_s(j);
        // dV_j as soon as P^T_j is in place, dK_j once dS^T_j is: dP^T_{j+1}
        // waits for both, and only dK_j then stands between the end of the
        // softmax and the next dP^T
        if (!g.wait_warp(&m.do_full[ds], (j / kDoStages) & 1, 8)) { ok = false; break; }
        if (!g.wait_warp(&m.p_full[j & 1], (j >> 1) & 1, 9)) { ok = false; break; }
        tc_fence_after();
        const uint64_t gd = sdesc_sw128(sDO + ds * L::TB, L::CHUNK, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (leader)
            umma_bf16_ta(tmem + L::TM_DV, sreg + (kk >> 1) * 32 + (kk & 1) * 8, sdesc_add(gd, kk * 2048), idG,
                         (j > 0 || kk > 0) ? 1u : 0u);
        if (leader) umma_commit(&m.do_empty[ds]);
        __syncwarp();
        if (!g.wait_warp(&m.q_full[qs], (j / kQStages) & 1, 10)) { ok = false; break; }
        if (!g.wait_warp(&m.ds_full[j & 1], (j >> 1) & 1, 11)) { ok = false; break; }
        tc_fence_after();
        const uint64_t gq = sdesc_sw128(sQ + qs * L::TB, L::CHUNK, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (leader)
            umma_bf16_ta(tmem + L::TM_DK, sreg + (kk >> 1) * 32 + 16 + (kk & 1) * 8, sdesc_add(gq, kk * 2048), idG,
                         (j > 0 || kk > 0) ? 1u : 0u);
        if (leader) {
          umma_commit(&m.grad_done[j & 1]);
          umma_commit(&m.q_empty[qs]);
        }
        __syncwarp();
      }
    }
    if (leader) {
      umma_commit(&m.final_grad);
      g.drain(&m.final_grad, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int hsel = (warp - 3) >> 2;  // which 32 query columns of every step
    const int r = quarter * 32 + lane;
    const int kvidx = tk * kTile + r;
    const int32_t segk = p.seg ? p.seg[(size_t)b * p.N + kvidx] : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const int4 kt = trow[tk];
    bool ok = true;
    int i = 0;
    for (int hq = h0; ok && hq < h1; ++hq) {
      int4 te = walk.kt, te_next;  // table entries of this and the next visited query tile
      for (int tq = walk.first(), tq_next; tq < walk.end(); tq = tq_next, te = te_next, ++i) {
        tq_next = walk.next(tq, te_next);  // loaded now, used after this tile's work
        const int qs = i % kQStages, ds = i % kDoStages;
        ok = g.wait(&m.q_full[qs], (i / kQStages) & 1, 12) && g.wait(&m.do_full[ds], (i / kDoStages) & 1, 13);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        ok = g.wait(&m.s_full[i & 1], (i >> 1) & 1, 14);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sreg = tmem + lane_base + L::reg_s(i) + hsel * 32;
        const uint32_t dreg = tmem + lane_base + L::reg_dp(i) + hsel * 32;
        const bool masked = !tile_pair_full(tq, te, tk, kt);
        const int c0 = hsel * 32;        // first query column of this thread within the tile
        const int q0 = tq * kTile + c0;  // its token index
        // ---- phase A: P^T = exp2(S^T * scale*log2e - lse*log2e), bf16 over S^T
        {
          uint32_t sv[32];
          tmem_ld32(sreg, sv);
          const float4* l4 = reinterpret_cast<const float4*>(&m.lse[qs][c0]);
          uint32_t pw[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 lv = l4[e4];
            const float lz[4] = {lv.x, lv.y, lv.z, lv.w};
            float sz[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) sz[e] = __uint_as_float(sv[e4 * 4 + e]);
            if (masked) {
              const int4 gv = p.seg ? __ldg(reinterpret_cast<const int4*>(p.seg + (size_t)b * p.N + q0) + e4)
                                    : make_int4(0, 0, 0, 0);
              const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                sz[e] = (q0 + e4 * 4 + e >= kvidx && gz[e] == segk) ? sz[e] : -INFINITY;
            }
            float pz[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) pz[e] = ex2(fmaf(sz[e], sl2, -lz[e]));
            pw[e4 * 2] = pack_bf16x2(pz[0], pz[1]);
            pw[e4 * 2 + 1] = pack_bf16x2(pz[2], pz[3]);
          }
          // packed columns 0..15 of this thread's slice: S^T columns it has already read
          tmem_st16_nowait(sreg, pw);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&m.p_full[i & 1]);
        // ---- phase B: dS^T = P^T * (dP^T - delta), bf16 next to P^T
        ok = g.wait(&m.dp_full[i & 1], (i >> 1) & 1, 15);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        tc_fence_after();
        const float4* d4 = reinterpret_cast<const float4*>(&m.dl[ds][c0]);
        uint32_t dpa[32], pb[16];
        tmem_ld32_ld16(dreg, sreg, dpa, pb);
        tc_fence_before();
        mbar_arrive(&m.dp_free[i & 1]);
        {
          uint32_t dw[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dv = d4[e4];
            const uint32_t w0 = pb[e4 * 2], w1 = pb[e4 * 2 + 1];
            const float pp[4] = {__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u),
                                 __uint_as_float(w1 << 16), __uint_as_float(w1 & 0xFFFF0000u)};
            dw[e4 * 2] = pack_bf16x2(pp[0] * (__uint_as_float(dpa[e4 * 4]) - dv.x),
                                     pp[1] * (__uint_as_float(dpa[e4 * 4 + 1]) - dv.y));
            dw[e4 * 2 + 1] = pack_bf16x2(pp[2] * (__uint_as_float(dpa[e4 * 4 + 2]) - dv.z),
                                         pp[3] * (__uint_as_float(dpa[e4 * 4 + 3]) - dv.w));
          }
          // packed columns 16..31 of this thread's slice (read in phase A)
          tmem_st16_nowait(sreg + 16, dw);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&m.ds_full[i & 1]);
        mbar_arrive(&m.do_empty[ds]);  // this step's delta vector has been read
      }
    }
    if (ok && i > 0) {
      ok = g.wait(&m.final_grad, 0, 16);
      ok = __all_sync(~0u, ok);
    }
    if (ok && i > 0) {
      tc_fence_after();
      // This thread's halves of the dV and dK rows go into the V and K tiles'
      // shared memory (free: every MMA has completed), in the
      // 128-byte-swizzled layout a TMA store reads; one thread then stores
      // both tiles, so the writes to global memory are whole 128-byte rows.
      uint8_t* sv = base + L::OFF_V;
      uint8_t* sk = base + L::OFF_K;
      const float sc = p.scale;
#pragma unroll
      for (int c0 = hsel * 32; c0 < D && c0 < (hsel + 1) * 32; c0 += 32) {
        uint32_t v[32], k[32];
        tmem_ld32x2(tmem + lane_base + L::TM_DV + c0, tmem + lane_base + L::TM_DK + c0, v, k);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col = c0 + 8 * q4;  // first of the 8 columns in this 16-byte unit
          const uint32_t off = (col >> 6) * L::CHUNK + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4);
          st_shared_v4(smem_u32(sv + off), pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]), __uint_as_float(v[q4 * 8 + 1])),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]), __uint_as_float(v[q4 * 8 + 3])),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]), __uint_as_float(v[q4 * 8 + 5])),
                       pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]), __uint_as_float(v[q4 * 8 + 7])));
          st_shared_v4(smem_u32(sk + off),
                       pack_bf16x2(__uint_as_float(k[q4 * 8 + 0]) * sc, __uint_as_float(k[q4 * 8 + 1]) * sc),
                       pack_bf16x2(__uint_as_float(k[q4 * 8 + 2]) * sc, __uint_as_float(k[q4 * 8 + 3]) * sc),
                       pack_bf16x2(__uint_as_float(k[q4 * 8 + 4]) * sc, __uint_as_float(k[q4 * 8 + 5]) * sc),
                       pack_bf16x2(__uint_as_float(k[q4 * 8 + 6]) * sc, __uint_as_float(k[q4 * 8 + 7]) * sc));
        }
      }
      fence_async_smem();  // these writes are read by the TMA stores
      mbar_arrive(&m.o_staged);
      if (warp == 3 && lane == 0 && g.wait(&m.o_staged, 0, 17)) {
        for (int c = 0; c < D / 64; ++c) {
          tma_store_rows(&tmDV, sv + c * L::CHUNK, c * 64, tk * kTile, hk, b, p.Hkv, p.N, T4);
          tma_store_rows(&tmDK, sk + c * L::CHUNK, c * 64, tk * kTile, hk, b, p.Hkv, p.N, T4);
        }
        bulk_commit();
        bulk_wait_all();  // the stores have read shared memory (and completed) before the CTA exits
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
cudaError_t launch_dkv_d(const AttnParams& p, int Dio, const RowStrides& rs, const void* q, const void* k,
                         const void* v, const void* dout, cudaStream_t st) {
  using L = DkvLayout<D>;
  CUtensorMap tq, tdo, tk, tv, tdk, tdv;
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
  if (!qmap(&tq, q) || !qmap(&tdo, dout) || !kmap(&tk, k) || !kmap(&tv, v) || !kmap(&tdk, p.dk) ||
      !kmap(&tdv, p.dv))
    return cudaErrorInvalidValue;
  // the tensor maps' form is fixed at compile time: the contiguous case runs
  // exactly the 2-D code
  const auto kfn = pp.tma4 ? dkv_kernel<D, DM, true> : dkv_kernel<D, DM, false>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * p.Hkv * p.B);
  kfn<<<grid, kDkvThreads, L::SMEM, st>>>(tq, tdo, tk, tv, tdk, tdv, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dkv(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k,
                           const void* v, const void* dout, cudaStream_t st) {
  // head dim 96 runs the 128-wide tile layout: its tensor maps are 96
  // elements wide, so TMA fills columns 96..127 of every loaded tile with
  // zeros and drops them from every store; the MMAs contract over 96 (six
  // K-steps) and produce 96 columns (N = 96), so no work is spent on them.
  if (D == 64) return launch_dkv_d<64>(p, 64, rs, q, k, v, dout, st);
  if (D == 96) return launch_dkv_d<128, 96>(p, 96, rs, q, k, v, dout, st);
  return launch_dkv_d<128>(p, 128, rs, q, k, v, dout, st);
}

}  // namespace pa
