// fwd.cu -- packed (block-diagonal causal) attention forward for sm_103a.
//
// One CTA per (query tile of 128 rows, query head, batch row), launched in the
// order of the prologue's work list (longest key walks first). It visits only
// key tiles whose segment-id range overlaps the query tile's (the changelog's
// PACKED forward: cross-segment blocks are skipped, not masked) and applies
// the element mask (j <= i and seg[i] == seg[j]) only on tile pairs that are
// not entirely visible. The saved state is O and its log-sum-exp
// (mlx-train-perf 0.5.1 README, "Flash-attention training path").
//
// Per visited key tile j: S_j = Q K_j^T (128 x 128, Q and K in shared memory)
// into TMEM S buffer j mod 2, P_j = 2^(S_j log2e scale - m) as bf16 into P
// buffer j mod 2, and O += P_j V_j with P_j fed straight from TMEM into one O
// accumulator. The softmax runs in two warpgroups, one thread per query row
// holding the row's 128 scores: group 0 takes the even visited tiles and
// group 1 the odd ones, so two tiles' exponentials are in flight at once, and
// each group owns the S and P buffer of its tiles. A group releases its S
// buffer as soon as it has loaded the scores, so S_{j+2} runs while P_j is
// being formed; P_{j+2} waits only for PV_j. The only step that passes from
// tile to tile is the row maximum in use, which each group hands to the other
// through shared memory as soon as it has its tile's maximum. One warp issues
// the S products, another the PV products, each waiting only on its own
// dependencies.
//
// Online softmax works in log2 units of the scaled score and rescales O only
// when a row's maximum rises by more than 8 (a factor 256); P is always
// computed against the maximum in use, so O and l stay consistent and O / l
// is exact in real arithmetic. Each group keeps its own partial sums against
// the maximum it last used; the epilogue brings both to the final maximum and
// adds them. O is divided by a sum that takes the bf16-rounded weights the PV
// product used on masked tiles and the exact weights on entirely visible
// ones; lse uses the exact fp32 sum. O leaves through the Q tile's shared
// memory and a TMA store.
//
// Warp roles: warp 0 TMA producer (Q once; K through a 3-stage ring, V
// through a 2-stage ring, the per-key segment ids of key tiles that span
// several segments through a ring of their own), warp 1 S issuer and TMEM
// owner, warp 2 PV issuer, warps 3..6 softmax group 0 and warps 7..10
// softmax group 1 (TMEM lane quarter = warp index mod 4).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"
#include "tmap.h"

namespace pa {

namespace {

template <int D>
struct FwdLayout {
  static constexpr int NSK = 3, NSV = 2;  // K stages, V stages
  static constexpr uint32_t TB = 128 * D * 2;   // one 128-row tile of Q, K or V
  static constexpr uint32_t CHUNK = 128 * 128;  // one 64-column chunk of a 128-row tile
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + TB;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TB;
  static constexpr uint32_t TILE_BYTES = OFF_V + NSV * TB;
  static constexpr uint32_t MISC_BYTES = 8192;
  static constexpr uint32_t SMEM = TILE_BYTES + MISC_BYTES + 1024;
  // TMEM: O (D columns) at 0; S buffers of 128 columns at 128 and 256; P
  // buffers of 64 columns (bf16 pairs) at 384 and 448. Tile j uses S and P
  // buffer j mod 2, the buffers of the softmax group that owns it.
  static constexpr uint32_t TM_O = 0, TM_S = 128, TM_P = 384, TMEM_COLS = 512;
};

struct FwdMisc {
  uint64_t q_full, k_full[3], k_empty[3], v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], mh_full[2][4], sums_full, fin_s, fin_pv;
  uint64_t seg_full[4], seg_empty[4];  // per-key segment ids of the tiles that need them (see seg_stage)
  uint64_t o_staged;                   // O rows written to shared memory by all softmax threads
  uint32_t tmem_base;
  int abort_flag;
  alignas(16) int32_t segkv[4][128];
  float mh[2][128];       // [tile parity][row]: row maximum in use after the tile
  float sums[2][2][128];  // [group][l, lr][row]: each group's sums at the final maximum
};

// Mask 32 scores of keys k0 .. k0+31 for query row qidx (segment segq): a
// score stays only where the key is not after the query (checked when causal
// is set) and lies in the same segment. The keys' segment ids come from sg,
// or are all segk when sg is null.
__device__ __forceinline__ void mask32(uint32_t (&x)[32], const int32_t* sg, int32_t segk, int k0, int qidx,
                                       int32_t segq, bool causal) {
  const int4* g4 = reinterpret_cast<const int4*>(sg);
#pragma unroll
  for (int e4 = 0; e4 < 8; ++e4) {
    const int4 gv = sg ? g4[e4] : make_int4(segk, segk, segk, segk);
    const int32_t gz[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = e4 * 4 + e;
      x[c] = ((!causal || k0 + c <= qidx) && gz[e] == segq) ? x[c] : __float_as_uint(-INFINITY);
    }
  }
}

__device__ __forceinline__ float max32(const uint32_t (&x)[32]) {
  float a = __uint_as_float(x[0]), b = __uint_as_float(x[1]);
#pragma unroll
  for (int e = 2; e < 30; e += 4) {
    a = fmax3(a, __uint_as_float(x[e]), __uint_as_float(x[e + 1]));
    b = fmax3(b, __uint_as_float(x[e + 2]), __uint_as_float(x[e + 3]));
  }
  return fmax3(a, b, fmaxf(__uint_as_float(x[30]), __uint_as_float(x[31])));
}

// Pairs of keys, of each 16, whose 2^t the FMA pipe computes (ex2_fma2)
// instead of the MUFU. The polynomial costs about five issue slots a key
// instead of one, and on GB300 the softmax warps are bound by issue, not by
// the MUFU: with 2, 4 or 6 pairs of 16 the 8k forward took 0.490, 0.588 and
// 0.509 ms against 0.450 ms with none (0.5% relative change in O), so the
// default is none and the option stays for other parts.
#ifndef PA_FWD_FMA_EX2_PAIRS
#define PA_FWD_FMA_EX2_PAIRS 0
#endif
constexpr int kFmaPairs = PA_FWD_FMA_EX2_PAIRS;
static_assert(kFmaPairs >= 0 && kFmaPairs <= 16, "pairs of 16");

// P for 32 keys: 2^(s sl2 - moff) packed to bf16 pairs into 16 TMEM columns
// (not waited); adds the exact weights to ls and, with ROUNDED, the
// bf16-rounded ones to lr. The scaling and the sums run two keys per
// instruction (packed FP32). kFmaPairs of the 16 pairs, spread evenly, take
// their exponentials on the FMA pipe.
template <bool ROUNDED>
__device__ __forceinline__ void exp_store32(const uint32_t (&x)[32], uint64_t sc, uint64_t off, uint32_t taddr,
                                            uint64_t& ls, uint64_t& lr) {
  uint64_t s2[2] = {0ull, 0ull}, r2[2] = {0ull, 0ull};
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const uint64_t t2 = fma2(f2(__uint_as_float(x[e]), __uint_as_float(x[e + 1])), sc, off);
    const int i = e >> 1;
    float e0, e1;
    if ((i * kFmaPairs) / 16 != ((i + 1) * kFmaPairs) / 16) {
      const float2 y2 = f2_split(ex2_fma2(t2));
      e0 = y2.x;
      e1 = y2.y;
    } else {
      const float2 t = f2_split(t2);
      e0 = ex2(t.x);
      e1 = ex2(t.y);
    }
    const uint32_t y = pack_bf16x2(e0, e1);
    s2[(e >> 1) & 1] = add2(s2[(e >> 1) & 1], f2(e0, e1));
    if (ROUNDED)
      r2[(e >> 1) & 1] = add2(r2[(e >> 1) & 1], f2(__uint_as_float(y << 16), __uint_as_float(y & 0xFFFF0000u)));
    pk[e >> 1] = y;
  }
  tmem_st16_nowait(taddr, pk);
  ls = add2(ls, add2(s2[0], s2[1]));
  if (ROUNDED) lr = add2(lr, add2(r2[0], r2[1]));
}

// Per-key segment ids travel only for key tiles that span several segments.
// The n-th such tile of softmax group g (the group owning visited tile j is
// j mod 2) uses stage g + 2 (n mod 2), phase n / 2: each group owns two
// stages and waits every phase of them in order.
__device__ __forceinline__ bool needs_ids(const AttnParams& p, int4 te) { return p.seg && te.x != te.y; }
__device__ __forceinline__ int seg_stage(int g, int n) { return g + 2 * (n & 1); }

template <int D, int DM, bool T4>
__global__ void __launch_bounds__(352, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
               const AttnParams p) {
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
  // the prologue's work list: longest key walks first, all heads of a tile together
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m.s_full[s], 1);
      mbar_init(&m.s_free[s], 128);  // the softmax group that owns the tile
      mbar_init(&m.p_full[s], 128);
      mbar_init(&m.pv_done[s], 1);
    }
    for (int s = 0; s < 2; ++s)
      for (int q = 0; q < 4; ++q) mbar_init(&m.mh_full[s][q], 32);  // one warp: 32 rows
    mbar_init(&m.sums_full, 256);
    mbar_init(&m.o_staged, 256);
    for (int s = 0; s < 4; ++s) {
      mbar_init(&m.seg_full[s], 1);
      mbar_init(&m.seg_empty[s], 128);  // the softmax group that owns the tile
    }
    mbar_init(&m.fin_s, 1);
    mbar_init(&m.fin_pv, 1);
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
    // Lane 0 loads Q, then per key tile its per-key segment ids where the
    // tile needs them (a ring of their own) and K (a 3-stage ring); lane 1
    // the V ring: each ring refills as soon as its own stage is released.
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      mbar_expect_tx(&m.q_full, L::TB);
      for (int c = 0; c < D / 64; ++c) tma_load_rows(base + L::OFF_Q + c * L::CHUNK, &tmQ, &m.q_full, c * 64,
                                                     tq * kTile, h, b, p.Hq, p.N, T4);
      int jk = 0;
      int ns[2] = {0, 0};  // segment-id copies issued for each softmax group's tiles
      int4 te, te_next;  // table entries of this and the next visited key tile
      for (int tk = walk.first(te), tk_next; tk <= tq; tk = tk_next, te = te_next, ++jk) {
        tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
        const int sk = jk % NSK;
        if (needs_ids(p, te)) {  // the tile's per-key segment ids, ahead of its K
          const int grp = jk & 1, n = ns[grp], ss = seg_stage(grp, n);
          if (!g.wait(&m.seg_empty[ss], ((n >> 1) & 1) ^ 1, 15)) break;
          mbar_expect_tx(&m.seg_full[ss], 512);
          bulk_load(m.segkv[ss], p.seg + (size_t)b * p.N + tk * kTile, 512, &m.seg_full[ss]);
          ++ns[grp];
        }
        if (!g.wait(&m.k_empty[sk], ((jk / NSK) & 1) ^ 1, 1)) break;
        mbar_expect_tx(&m.k_full[sk], L::TB);
        for (int c = 0; c < D / 64; ++c)
          tma_load_rows(base + L::OFF_K + sk * L::TB + c * L::CHUNK, &tmK, &m.k_full[sk], c * 64,
                        tk * kTile, hk, b, p.Hkv, p.N, T4);
      }
      // no copy may still be landing when the CTA exits
      g.drain(&m.q_full, 0);
      for (int i = (jk > NSK ? jk - NSK : 0); i < jk; ++i) g.drain(&m.k_full[i % NSK], (i / NSK) & 1);
      for (int grp = 0; grp < 2; ++grp)  // at most one copy per stage can be in flight: its last
        for (int n = (ns[grp] > 2 ? ns[grp] - 2 : 0); n < ns[grp]; ++n) g.drain(&m.seg_full[seg_stage(grp, n)], (n >> 1) & 1);
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
    // ------------------------------------------------------------ S issuer
    // The whole warp runs the issue loop and every wait; lane 0 alone issues
    // the tcgen05 instructions.
    const bool leader = lane == 0;
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint64_t qd = sdesc_sw128(sQ, 16, 1024);
    bool ok = g.wait_warp(&m.q_full, 0, 3);
    int j = 0;
    int4 te, te_next;  // table entries of this and the next visited key tile
    for (int tk = walk.first(te), tk_next; ok && tk <= tq; tk = tk_next, te = te_next, ++j) {
      tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
      const int sb = j & 1, sk = j % NSK;
      // S_j into buffer sb once the softmax has loaded S_{j-2} from it
      if (j >= 2 && !g.wait_warp(&m.s_free[sb], ((j - 2) >> 1) & 1, 4)) { ok = false; break; }
      if (!g.wait_warp(&m.k_full[sk], (j / NSK) & 1, 5)) { ok = false; break; }
      tc_fence_after();
      const uint64_t kd = sdesc_sw128(sK + sk * L::TB, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < DM / 16; ++kk) {
        const uint32_t ko = (kk >> 2) * L::CHUNK + (kk & 3) * 32;
        if (leader) umma_bf16(tmem + L::TM_S + sb * 128, sdesc_add(qd, ko), sdesc_add(kd, ko), idS, kk > 0 ? 1u : 0u);
      }
      if (leader) {
        umma_commit(&m.s_full[sb]);
        umma_commit(&m.k_empty[sk]);
      }
      __syncwarp();
    }
    if (leader) {
      umma_commit(&m.fin_s);
      g.drain(&m.fin_s, 0);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // O += P_j V_j with P_j (bf16, packed in the first 64 columns of its S
    // buffer) as the A operand straight from TMEM and V MN-major.
    const bool leader = lane == 0;
    constexpr uint32_t idO = idesc_bf16_f32(128, DM, false, true);
    bool ok = true;
    int j = 0;
    int4 te, te_next;  // table entries of this and the next visited key tile
    for (int tk = walk.first(te), tk_next; ok && tk <= tq; tk = tk_next, te = te_next, ++j) {
      tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
      const int sb = j & 1, sv = j % NSV;
      if (!g.wait_warp(&m.v_full[sv], (j / NSV) & 1, 6)) { ok = false; break; }
      if (!g.wait_warp(&m.p_full[sb], (j >> 1) & 1, 7)) { ok = false; break; }
      tc_fence_after();
      const uint64_t vd = sdesc_sw128(sV + sv * L::TB, L::CHUNK, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (leader)
          umma_bf16_ta(tmem + L::TM_O, tmem + L::TM_P + sb * 64 + kk * 8, sdesc_add(vd, kk * 2048), idO,
                       (j > 0 || kk > 0) ? 1u : 0u);
      if (leader) {
        umma_commit(&m.pv_done[sb]);
        umma_commit(&m.v_empty[sv]);
      }
      __syncwarp();
    }
    if (leader) {
      umma_commit(&m.fin_pv);
      g.drain(&m.fin_pv, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Group 0 (warps 3..6) takes the even visited tiles, group 1 (warps
    // 7..10) the odd ones; thread r of a group owns query row r (TMEM lane r).
    const int grp = (warp - 3) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qidx = tq * kTile + r;
    // this row's lse in the caller's (B, Hq, Nr) layout (tail rows have none)
    const size_t lse_row = (size_t)(b * p.Hq + h) * p.Nr + qidx;
    const int32_t segq = p.seg ? p.seg[(size_t)b * p.N + qidx] : 0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t tO = tmem + lane_base + L::TM_O;
    const float sl2 = p.scale_log2;
    float m_w = -INFINITY;           // the maximum this group's sums are taken against
    uint64_t l2 = 0ull, lr2 = 0ull;  // exact and bf16-rounded weight sums, two partial sums each
    bool ok = true;
    int jj = 0;     // visited tiles
    int n_ids = 0;  // this group's tiles that needed per-key segment ids
    int4 te, te_next;  // table entries of this and the next visited key tile
    for (int tk = walk.first(te), tk_next; tk <= tq; tk = tk_next, te = te_next, ++jj) {
      tk_next = walk.next(tk, te_next);  // loaded now, used after this tile's work
      if ((jj & 1) != grp) continue;
      const bool masked = !tile_pair_full(tq, walk.qt, tk, te);
      // this group's S buffer, released as soon as the scores are loaded
      ok = g.wait(&m.s_full[grp], (jj >> 1) & 1, 9);
      if (!__all_sync(~0u, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t x0[32], x1[32], x2[32], x3[32];
      tmem_ld128(tmem + lane_base + L::TM_S + grp * 128, x0, x1, x2, x3);
      tc_fence_before();
      mbar_arrive(&m.s_free[grp]);
      const uint32_t tP = tmem + lane_base + L::TM_P + grp * 64;
      const bool ids = needs_ids(p, te);  // then the tile is masked too
      const int ss = seg_stage(grp, n_ids);
      if (ids) {  // per-key segment ids, released once the mask is applied
        ok = g.wait(&m.seg_full[ss], (n_ids >> 1) & 1, 8);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
      }
      if (masked) {
        // per-key segment ids only where the key tile spans several
        // segments; otherwise the tile's one segment decides for all keys
        const bool causal = tk == tq;
        const int32_t* sg = ids ? m.segkv[ss] : nullptr;
        const int k0 = tk * kTile;
        mask32(x0, sg, te.x, k0, qidx, segq, causal);
        mask32(x1, sg ? sg + 32 : sg, te.x, k0 + 32, qidx, segq, causal);
        mask32(x2, sg ? sg + 64 : sg, te.x, k0 + 64, qidx, segq, causal);
        mask32(x3, sg ? sg + 96 : sg, te.x, k0 + 96, qidx, segq, causal);
      }
      if (ids) {
        mbar_arrive(&m.seg_empty[ss]);
        ++n_ids;
      }
      const float ms = fmax3(fmaxf(max32(x0), max32(x1)), max32(x2), max32(x3)) * sl2;
      // the maximum in use after the previous tile, from the other group
      float m_prev = -INFINITY;
      if (jj > 0) {
        ok = g.wait(&m.mh_full[(jj - 1) & 1][quarter], ((jj - 1) >> 1) & 1, 10);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        m_prev = m.mh[(jj - 1) & 1][r];
      }
      // the lanes of a warp take the rescale branch together
      const bool rescale = __any_sync(~0u, ms > m_prev + 8.f);
      const float m_new = rescale ? fmaxf(m_prev, ms) : m_prev;
      m.mh[jj & 1][r] = m_new;
      mbar_arrive(&m.mh_full[jj & 1][quarter]);
      if (m_w != m_new) {  // this group's sums to the new maximum
        const float a = (m_w == -INFINITY) ? 0.f : ex2(m_w - m_new);
        l2 = mul2(l2, f2(a, a));
        lr2 = mul2(lr2, f2(a, a));
        m_w = m_new;
      }
      const float moff = (m_new == -INFINITY) ? 0.f : m_new;
      const uint64_t sc = f2(sl2, sl2), off = f2(-moff, -moff);
      // P for keys 32c .. 32c+31 -> packed columns 16c .. 16c+15 of this
      // group's P buffer, once PV_{jj-2} has read the P that was there
      // The normaliser of O sums the bf16-rounded weights the PV product
      // uses on masked tiles, where a row with few keys has all of them; on
      // entirely visible tiles it takes the exact weights, whose rounding
      // errors average out over the 128 keys of the tile.
      if (jj >= 2) {
        ok = g.wait(&m.pv_done[grp], ((jj - 2) >> 1) & 1, 16);
        if (!__all_sync(~0u, ok)) { ok = false; break; }
        tc_fence_after();
      }
      uint64_t t2 = 0ull, tr2 = 0ull;
      if (masked) {
        exp_store32<true>(x0, sc, off, tP, t2, tr2);
        exp_store32<true>(x1, sc, off, tP + 16, t2, tr2);
        exp_store32<true>(x2, sc, off, tP + 32, t2, tr2);
        exp_store32<true>(x3, sc, off, tP + 48, t2, tr2);
      } else {
        exp_store32<false>(x0, sc, off, tP, t2, tr2);
        exp_store32<false>(x1, sc, off, tP + 16, t2, tr2);
        exp_store32<false>(x2, sc, off, tP + 32, t2, tr2);
        exp_store32<false>(x3, sc, off, tP + 48, t2, tr2);
        tr2 = t2;
      }
      l2 = add2(l2, t2);
      lr2 = add2(lr2, tr2);
      if (rescale && jj > 0) {  // O holds earlier tiles: rescale it once their PV is done
        // (PV_{jj-2} has completed, and with it PV_{jj-3}: this parity wait on
        // the other group's barrier cannot match an older phase)
        const float alpha = (m_prev == -INFINITY) ? 0.f : ex2(m_prev - m_new);
        ok = g.wait(&m.pv_done[grp ^ 1], ((jj - 1) >> 1) & 1, 11);
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
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&m.p_full[grp]);
    }
    // ------------------------------------------------------------ epilogue
    // The final maximum is the one the last tile's group handed on; both
    // groups take their sums to it, add them up and write half of O each.
    float m_fin = -INFINITY;
    if (ok && jj > 0) {
      ok = g.wait(&m.mh_full[(jj - 1) & 1][quarter], ((jj - 1) >> 1) & 1, 12);
      ok = __all_sync(~0u, ok);
      if (ok) m_fin = m.mh[(jj - 1) & 1][r];
    }
    if (ok) {
      const float a = (m_w == m_fin) ? 1.f : (m_w == -INFINITY ? 0.f : ex2(m_w - m_fin));
      const float2 lp = f2_split(l2), lrp = f2_split(lr2);
      m.sums[grp][0][r] = (lp.x + lp.y) * a;
      m.sums[grp][1][r] = (lrp.x + lrp.y) * a;
      mbar_arrive(&m.sums_full);
      ok = g.wait(&m.sums_full, 0, 13);
      ok = __all_sync(~0u, ok);
    }
    if (ok && jj > 0) {  // the last PV has accumulated into O
      ok = g.wait(&m.fin_pv, 0, 14);  // the PV issuer's final commit covers every PV
      ok = __all_sync(~0u, ok);
    }
    if (ok && jj > 0) {
      tc_fence_after();
      // both groups add the two groups' sums in the same order
      const float lt = m.sums[0][0][r] + m.sums[1][0][r];
      const float inv = 1.f / (m.sums[0][1][r] + m.sums[1][1][r]);
      // This group's half of the O row goes into the Q tile's shared memory
      // (free: every S product has completed), in the 128-byte-swizzled layout
      // a TMA store reads; one thread then stores the whole tile, so the
      // writes to global memory are whole 128-byte rows.
      uint8_t* so = base + L::OFF_Q;
#pragma unroll 1
      for (int c0 = grp * (D / 2); c0 < (grp + 1) * (D / 2); c0 += 32) {
        uint32_t a[32];
        tmem_ld32(tO + c0, a);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int col = c0 + 8 * q4;  // first of the 8 columns in this 16-byte unit
          const uint32_t off = (col >> 6) * L::CHUNK + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4);
          st_shared_v4(smem_u32(so + off),
                       pack_bf16x2(__uint_as_float(a[q4 * 8 + 0]) * inv, __uint_as_float(a[q4 * 8 + 1]) * inv),
                       pack_bf16x2(__uint_as_float(a[q4 * 8 + 2]) * inv, __uint_as_float(a[q4 * 8 + 3]) * inv),
                       pack_bf16x2(__uint_as_float(a[q4 * 8 + 4]) * inv, __uint_as_float(a[q4 * 8 + 5]) * inv),
                       pack_bf16x2(__uint_as_float(a[q4 * 8 + 6]) * inv, __uint_as_float(a[q4 * 8 + 7]) * inv));
        }
      }
      fence_async_smem();  // these writes are read by the TMA store
      mbar_arrive(&m.o_staged);
      if (warp == 3 && lane == 0 && g.wait(&m.o_staged, 0, 15)) {
        for (int c = 0; c < D / 64; ++c) tma_store_rows(&tmO, so + c * L::CHUNK, c * 64, tq * kTile,
                                                        h, b, p.Hq, p.N, T4);
        bulk_commit();
        bulk_wait_all();  // the store has read shared memory (and completed) before the CTA exits
      }
      if (grp == 0 && qidx < p.Nr) p.lse[lse_row] = m_fin * 0.6931471805599453f + logf(lt);
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
cudaError_t launch_fwd_d(const AttnParams& p, int Dio, const RowStrides& rs, const void* q, const void* k,
                         const void* v, cudaStream_t st) {
  using L = FwdLayout<D>;
  CUtensorMap tq, tk, tv, to;
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
  if (!qmap(&tq, q) || !kmap(&tk, k) || !kmap(&tv, v) || !qmap(&to, p.out)) return cudaErrorInvalidValue;
  // the tensor maps' form is fixed at compile time: the contiguous case runs
  // exactly the 2-D code
  const auto kfn = pp.tma4 ? fwd_kernel<D, DM, true> : fwd_kernel<D, DM, false>;
  cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.T * p.Hq * p.B);
  kfn<<<grid, 352, L::SMEM, st>>>(tq, tk, tv, to, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k, const void* v,
                       cudaStream_t st) {
  // head dim 96 runs the 128-wide tile layout: its tensor maps are 96
  // elements wide, so TMA fills columns 96..127 of every loaded tile with
  // zeros and drops them from every store; the MMAs contract over 96 (six
  // K-steps) and produce 96 columns (N = 96), so no work is spent on them.
  if (D == 64) return launch_fwd_d<64>(p, 64, rs, q, k, v, st);
  if (D == 96) return launch_fwd_d<128, 96>(p, 96, rs, q, k, v, st);
  return launch_fwd_d<128>(p, 128, rs, q, k, v, st);
}

}  // namespace pa
