// common.cuh -- definitions shared by the packed-attention kernels.
//
// Tiles are 128 tokens. For every (row b, tile t) the prologue kernel writes
// one int4 {smin, smax, kv_lo, q_hi}:
//   smin/smax  smallest / largest segment id inside the tile,
//   kv_lo      first key tile <= t whose id range overlaps tile t's,
//   q_hi       last query tile >= t whose id range overlaps tile t's.
// A (query tile, key tile) pair can hold a visible pair only if the key tile
// is not after the query tile and the two id ranges overlap; every other pair
// is skipped without being computed (the changelog entry for the PACKED
// kernels: cross-segment blocks are skipped; the 0.5.0 note in the README's
// "Sequence packing": dK/dV ends its query walk at the key block's segment
// end). Range overlap is a conservative test, so any id values stay correct;
// contiguous runs (what packing produces) make it exact at tile granularity.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace pa {

constexpr int kTile = 128;
// Status-word site number of the bounded-wait self-test (the kernels use
// smaller ones).
constexpr uint32_t kSelftestWaitSite = 99;

struct AttnParams {
  // N: tokens per row as the kernels see them (whole tiles, T = N / 128);
  // Nr <= N: the caller's tokens per row. Rows n >= Nr are a tail that TMA
  // reads as zeros and never stores, with the row's last segment id.
  int B, Hq, Hkv, N, T, G, Nr;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  const int32_t* seg;   // (B, N) or null (every token in one segment)
  const int4* tiles;    // (B, T) table written by the prologue
  // Work lists written by the prologue: entries b*T + t, longest walks first;
  // work_q orders the query tiles of the forward and dQ kernels, work_k the
  // key tiles of the dK/dV kernel.
  const int32_t* work_q;
  const int32_t* work_k;
  uint32_t* status;     // device status word
  // forward outputs
  __nv_bfloat16* out;
  float* lse;
  // backward
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse_in;
  float* delta;  // (B, Hq, N), written by the delta kernel
  float* lse2;   // (B, Hq, N) lse * log2(e), written by the delta kernel
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  // single-pass backward only: fp32 dQ accumulator (B, Hq, N, dq_ld), zeroed
  // by the delta kernel when non-null
  float* dq_acc;
  int dq_ld;
  // tensor maps of the (B, H, N, D) tensors: 2-D over B*H*N rows (contiguous
  // tensors) or 4-D {D, N, H, B} with the caller's strides
  int tma4;
};

__device__ __forceinline__ bool tiles_overlap(int4 a, int4 b) { return a.x <= b.y && b.x <= a.y; }

// Every element of the (query tile, key tile) pair is visible: strictly below
// the diagonal and both tiles inside one and the same segment.
__device__ __forceinline__ bool tile_pair_full(int tq, int4 q, int tk, int4 k) {
  return tk < tq && q.x == q.y && k.x == k.y && q.x == k.x;
}

// Key tiles a query tile visits, in increasing order.
struct KvWalk {
  const int4* row;  // tiles of this batch row
  int tq;
  int4 qt;
  __device__ __forceinline__ KvWalk(const int4* r, int tq_) : row(r), tq(tq_), qt(r[tq_]) {}
  __device__ __forceinline__ int first() const { return next(qt.z - 1); }
  __device__ __forceinline__ int next(int tk) const {
    for (++tk; tk < tq; ++tk)
      if (tiles_overlap(row[tk], qt)) return tk;
    return tk;  // tq itself: the diagonal tile always holds visible pairs
  }
  __device__ __forceinline__ int count() const {
    int n = 0;
    for (int tk = first(); tk <= tq; tk = next(tk)) ++n;
    return n;
  }
  // The same walk, also returning the table entry of the tile it lands on
  // (loaded once). Callers ask for the next tile at the start of their work
  // on the current one, so the load's latency hides behind that work.
  __device__ __forceinline__ int next(int tk, int4& e) const {
    for (++tk; tk < tq; ++tk) {
      e = row[tk];
      if (tiles_overlap(e, qt)) return tk;
    }
    e = qt;
    return tk;
  }
  __device__ __forceinline__ int first(int4& e) const { return next(qt.z - 1, e); }
};

// Query tiles a key tile is visited by, in increasing order.
struct QWalk {
  const int4* row;
  int tk;
  int4 kt;
  __device__ __forceinline__ QWalk(const int4* r, int tk_) : row(r), tk(tk_), kt(r[tk_]) {}
  __device__ __forceinline__ int first() const { return tk; }
  __device__ __forceinline__ int next(int tq) const {
    for (++tq; tq <= kt.w; ++tq)
      if (tiles_overlap(row[tq], kt)) return tq;
    return kt.w + 1;
  }
  __device__ __forceinline__ int end() const { return kt.w + 1; }
  // The same walk, also returning the table entry of the tile it lands on
  // (see KvWalk::next(int, int4&)).
  __device__ __forceinline__ int next(int tq, int4& e) const {
    for (++tq; tq <= kt.w; ++tq) {
      e = row[tq];
      if (tiles_overlap(e, kt)) return tq;
    }
    e = kt;
    return kt.w + 1;
  }
};

}  // namespace pa
