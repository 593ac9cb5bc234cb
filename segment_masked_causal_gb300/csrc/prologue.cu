// prologue.cu -- the segment-range tile table and the delta preprocess.
//
// Tile table: for each 128-token tile of each batch row, the smallest and
// largest segment id it holds, the first key tile whose id range overlaps it
// (the first key tile a query tile must visit) and the last query tile whose
// range overlaps it (where a key tile's query walk ends: mlx-train-perf 0.5.1
// README, "Sequence packing", the 0.5.0 dK/dV change). With seg == null every
// token is in segment 0.
//
// Delta: D_i = <dO_i, O_i>, the per-row term of the softmax backward
// (dS = P * (dP - D)); one fp32 value per query row, read by both backward
// kernels. Bandwidth-bound: 16-byte loads, rows split over D/8 lanes and
// reduced with shuffles.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "sm103.cuh"

namespace pa {

namespace {

__global__ void __launch_bounds__(256) tile_table_kernel(const int32_t* __restrict__ seg, int N, int T,
                                                         int4* __restrict__ tiles, uint32_t* status) {
  extern __shared__ int2 mm[];  // T entries {min, max}
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (b == 0 && threadIdx.x == 0 && status) *status = 0u;
  for (int t = warp; t < T; t += blockDim.x >> 5) {
    int lo = 0, hi = 0;
    if (seg) {
      const int4 v = reinterpret_cast<const int4*>(seg + (size_t)b * N + (size_t)t * kTile)[lane];
      lo = min(min(v.x, v.y), min(v.z, v.w));
      hi = max(max(v.x, v.y), max(v.z, v.w));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(~0u, lo, o));
        hi = max(hi, __shfl_xor_sync(~0u, hi, o));
      }
    }
    if (lane == 0) mm[t] = make_int2(lo, hi);
  }
  __syncthreads();
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const int2 me = mm[t];
    int lo = t, hi = t;
    for (int u = 0; u < t; ++u)
      if (mm[u].x <= me.y && me.x <= mm[u].y) { lo = u; break; }
    for (int u = T - 1; u > t; --u)
      if (mm[u].x <= me.y && me.x <= mm[u].y) { hi = u; break; }
    tiles[(size_t)b * T + t] = make_int4(me.x, me.y, lo, hi);
  }
}

// Work lists: the (row, tile) entries b*T + t in decreasing order of the
// number of tiles their walk visits at most -- key tiles kv_lo..tq for a
// query tile of the forward and dQ kernels, query tiles tk..q_hi for a key
// tile of the dK/dV kernel -- so the kernels start the longest walks first.
// Ties keep a fixed canonical order (query tiles from the last down, key
// tiles from the first up, batch rows increasing within one tile index), so a
// row in one segment gets exactly the longest-causal-walk-first order and
// the order never depends on timing. A counting sort over the costs 1..T:
// all threads count, one scan turns the counts into starting positions, and
// one warp per list places the entries 32 at a time, ranking equal costs
// within the warp by lane so that the sort is stable.
constexpr int kMaxSortedTiles = 4095;  // T above this: canonical order, unsorted

__device__ __forceinline__ int canon_q(int e, int B, int T) { return (e % B) * T + (T - 1 - e / B); }
__device__ __forceinline__ int canon_k(int e, int B, int T) { return (e % B) * T + e / B; }

// The counting sort itself, for a block of 1024 threads. range(ent) gives
// {kv_lo, q_hi} of table entry ent; cnt0 and cnt1 hold T + 1 ints each.
template <class Range>
__device__ __forceinline__ void build_work_lists(int B, int T, Range range, int* cnt0, int* cnt1,
                                                 int32_t* __restrict__ wq, int32_t* __restrict__ wk) {
  __shared__ int part[2][32];
  int* cnt[2] = {cnt0, cnt1};
  const int n = B * T;
  for (int c = threadIdx.x; c <= T; c += blockDim.x) cnt0[c] = cnt1[c] = 0;
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int eq = canon_q(e, B, T), ek = canon_k(e, B, T);
    atomicAdd(&cnt0[eq % T - range(eq).x + 1], 1);
    atomicAdd(&cnt1[range(ek).y - ek % T + 1], 1);
  }
  __syncthreads();
  // Starting position of cost c = entries of cost > c. Thread i sums a run of
  // costs (highest first), the warps scan those sums, then each thread writes
  // its run's starting positions.
  const int per = (T + blockDim.x) / blockDim.x;  // costs per thread, covering 1..T
  const int hi = T - threadIdx.x * per;           // this thread's run: costs hi, hi-1, .., hi-per+1 (>= 1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int l = 0; l < 2; ++l) {
    int s = 0;
    for (int c = hi; c > hi - per && c >= 1; --c) s += cnt[l][c];
    int x = s;  // inclusive scan over the block, in thread order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(~0u, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) part[l][warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x >> 5) ? part[l][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(~0u, w, o);
        if (lane >= o) w += y;
      }
      part[l][lane] = w;
    }
    __syncthreads();
    int pos = x - s + (warp > 0 ? part[l][warp - 1] : 0);  // exclusive start of this run
    for (int c = hi; c > hi - per && c >= 1; --c) {
      const int k = cnt[l][c];
      cnt[l][c] = pos;
      pos += k;
    }
    __syncthreads();
  }
  if (warp < 2) {
    int32_t* out = warp == 0 ? wq : wk;
    int* next = cnt[warp];
    for (int e0 = 0; e0 < n; e0 += 32) {
      const int e = e0 + lane;
      const bool live = e < n;
      int ent = 0, key = -1 - lane;  // lanes past the end take keys of their own
      if (live) {
        ent = warp == 0 ? canon_q(e, B, T) : canon_k(e, B, T);
        key = warp == 0 ? ent % T - range(ent).x + 1 : range(ent).y - ent % T + 1;
      }
      const unsigned same = __match_any_sync(~0u, key);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const int at = live ? next[key] + rank : 0;
      __syncwarp();
      if (live && rank == 0) next[key] += __popc(same);
      __syncwarp();
      if (live) out[at] = ent;
    }
  }
}

__global__ void __launch_bounds__(1024) work_list_kernel(const int4* __restrict__ tiles, int B, int T,
                                                         int32_t* __restrict__ wq, int32_t* __restrict__ wk) {
  const int n = B * T;
  if (T > kMaxSortedTiles) {
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      wq[e] = canon_q(e, B, T);
      wk[e] = canon_k(e, B, T);
    }
    return;
  }
  __shared__ int cnt[2][kMaxSortedTiles + 1];  // [list][cost]: counts, then next free position
  build_work_lists(B, T, [&](int ent) { const int4 v = tiles[ent]; return make_int2(v.z, v.w); }, cnt[0], cnt[1],
                   wq, wk);
}

// Rows with few tiles in all (B * T <= kSmallPrologue): the table and both
// lists in one CTA, with the per-tile id ranges kept in shared memory. Each
// warp takes four tiles at a time, so four loads of segment ids are in flight.
constexpr int kSmallPrologue = 4096;
constexpr size_t small_prologue_smem(int n, int T) { return (size_t)n * 16 + (size_t)2 * (T + 1) * 4; }

__global__ void __launch_bounds__(1024) prologue_small_kernel(const int32_t* __restrict__ seg, int B, int N, int T,
                                                              int4* __restrict__ tiles, int32_t* __restrict__ wq,
                                                              int32_t* __restrict__ wk, uint32_t* status) {
  extern __shared__ int2 sm2[];
  const int n = B * T;
  int2* mm = sm2;                                  // {min, max} per tile
  int2* range = sm2 + n;                           // {kv_lo, q_hi} per tile
  int* cnt = reinterpret_cast<int*>(sm2 + 2 * n);  // 2 (T + 1)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, warps = blockDim.x >> 5;
  if (threadIdx.x == 0 && status) *status = 0u;
  for (int e0 = 4 * warp; e0 < n; e0 += 4 * warps) {
    int4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + u;
      v[u] = make_int4(0, 0, 0, 0);
      if (seg && e < n) v[u] = reinterpret_cast<const int4*>(seg + (size_t)(e / T) * N + (size_t)(e % T) * kTile)[lane];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      int lo = min(min(v[u].x, v[u].y), min(v[u].z, v[u].w));
      int hi = max(max(v[u].x, v[u].y), max(v[u].z, v[u].w));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(~0u, lo, o));
        hi = max(hi, __shfl_xor_sync(~0u, hi, o));
      }
      if (lane == 0 && e0 + u < n) mm[e0 + u] = make_int2(lo, hi);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int2* row = mm + (e / T) * T;
    const int t = e % T;
    const int2 me = row[t];
    int lo = t, hi = t;
    for (int u = 0; u < t; ++u)
      if (row[u].x <= me.y && me.x <= row[u].y) { lo = u; break; }
    for (int u = T - 1; u > t; --u)
      if (row[u].x <= me.y && me.x <= row[u].y) { hi = u; break; }
    range[e] = make_int2(lo, hi);
    tiles[e] = make_int4(me.x, me.y, lo, hi);
  }
  __syncthreads();
  build_work_lists(B, T, [&](int ent) { return range[ent]; }, cnt, cnt + T + 1, wq, wk);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Lanes that share one row of the delta kernel: a power of two dividing the
// row's D/8 16-byte vectors, so a row's lanes sit in one warp.
constexpr int delta_lanes(int D) { return (D / 8) % 16 == 0 ? 16 : (D / 8) % 8 == 0 ? 8 : 4; }

template <int D>
__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                    const __nv_bfloat16* __restrict__ dout,
                                                    const float* __restrict__ lse, float* __restrict__ delta,
                                                    float* __restrict__ lse2, float* __restrict__ zero_acc,
                                                    size_t rows, bool contiguous, int N, int Nr, int H, int64_t s_n,
                                                    int64_t s_h, int64_t s_b) {
  // each of the row's LPR lanes takes every LPR-th 16-byte vector
  constexpr int VEC = D / 8;
  constexpr int LPR = delta_lanes(D);
  static_assert(VEC % LPR == 0, "head dim must be a multiple of 32");
  const size_t gtid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const int sub = threadIdx.x % LPR;
  for (size_t t = gtid; t < rows * LPR; t += stride) {
    // row = (b * H + h) * N + n of the kernels' rows; the caller's tensors
    // hold n < Nr (rows < 2^31), and contiguous ones with Nr = N skip the
    // divisions
    const size_t row = t / LPR;
    size_t off = row * D, lrow = row;
    bool tail = false;
    if (!contiguous) {
      const uint32_t r32 = (uint32_t)row, bh = r32 / (uint32_t)N, b = bh / (uint32_t)H, n = r32 - bh * (uint32_t)N;
      tail = n >= (uint32_t)Nr;
      off = (size_t)b * s_b + (size_t)(bh - b * (uint32_t)H) * s_h + (size_t)n * s_n;
      lrow = (size_t)bh * Nr + n;
    }
    // a tail query row gets P = 0 (lse = +inf) and delta = 0, so it adds
    // nothing; its lanes still take part in the shuffles below
    float acc = 0.f;
#pragma unroll
    for (int v = sub; v < VEC; v += LPR) {
      if (tail) break;
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + off) + v);
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(dout + off) + v);
      acc = fmaf(bf16lo(a.x), bf16lo(c.x), acc);
      acc = fmaf(bf16hi(a.x), bf16hi(c.x), acc);
      acc = fmaf(bf16lo(a.y), bf16lo(c.y), acc);
      acc = fmaf(bf16hi(a.y), bf16hi(c.y), acc);
      acc = fmaf(bf16lo(a.z), bf16lo(c.z), acc);
      acc = fmaf(bf16hi(a.z), bf16hi(c.z), acc);
      acc = fmaf(bf16lo(a.w), bf16lo(c.w), acc);
      acc = fmaf(bf16hi(a.w), bf16hi(c.w), acc);
      if (zero_acc) {
        float4* z = reinterpret_cast<float4*>(zero_acc + row * D) + 2 * v;
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int of = LPR / 2; of > 0; of >>= 1) acc += __shfl_xor_sync(~0u, acc, of);
    if (sub == 0) {
      delta[row] = acc;
      lse2[row] = tail ? INFINITY : lse[lrow] * 1.4426950408889634f;  // the backward's softmax works in base 2
    }
  }
}

// Self-test of the bounded waits: a warp waits, through the kernels' own
// wait path, on an mbarrier that nothing ever arrives on. Each wait gives up
// after its limit, records PA_DEVERR_TIMEOUT with the site in the status word
// and returns false, and the kernel exits normally: no trap, and the context
// stays usable.
__global__ void __launch_bounds__(32) wait_timeout_kernel(uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const Guard g{&abort_flag, status};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  (void)g.wait(&bar, 0, kSelftestWaitSite);
}

}  // namespace

cudaError_t launch_tile_table(const AttnParams& p, int4* tiles, cudaStream_t st) {
  const int n = p.B * p.T;
  if (n <= kSmallPrologue && p.T <= kMaxSortedTiles) {
    const size_t smem = small_prologue_smem(n, p.T);
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(prologue_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    prologue_small_kernel<<<1, 1024, smem, st>>>(p.seg, p.B, p.N, p.T, tiles, const_cast<int32_t*>(p.work_q),
                                                  const_cast<int32_t*>(p.work_k), p.status);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)p.T * sizeof(int2);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(tile_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  tile_table_kernel<<<p.B, 256, smem, st>>>(p.seg, p.N, p.T, tiles, p.status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  work_list_kernel<<<1, 1024, 0, st>>>(tiles, p.B, p.T, const_cast<int32_t*>(p.work_q),
                                       const_cast<int32_t*>(p.work_k));
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint32_t* status, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

// y[i] = 2^x[i] through the FMA-pipe exponential (ex2_fma2), each
// input in both lanes of the packed pair; lane 1 must agree with lane 0.
__global__ void exp2_fma_selftest_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float2 r = f2_split(ex2_fma2(f2(x[i], x[i])));
    y[i] = (__float_as_uint(r.x) == __float_as_uint(r.y)) ? r.x : __uint_as_float(0x7FC00001u);
  }
}

cudaError_t launch_exp2_fma_selftest(const float* x, float* y, int64_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  exp2_fma_selftest_kernel<<<(unsigned)(blocks < 1024 ? blocks : 1024), 256, 0, st>>>(x, y, n);
  return cudaGetLastError();
}

cudaError_t launch_delta(const AttnParams& p, int D, const RowStrides& rs, cudaStream_t st) {
  const bool contig = p.Nr == p.N && rs.q_n == D && rs.q_h == (int64_t)p.N * D && rs.q_b == (int64_t)p.Hq * p.N * D;
  const size_t rows = (size_t)p.B * p.Hq * p.N;
  const size_t threads = rows * (size_t)delta_lanes(D);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t blocks = (threads + 255) / 256;
  const size_t cap = (size_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (D == 128)
    delta_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(p.o, p.dout, p.lse_in, p.delta, p.lse2, p.dq_acc, rows, contig,
                                                     p.N, p.Nr, p.Hq, rs.q_n, rs.q_h, rs.q_b);
  else if (D == 96)
    delta_kernel<96><<<(unsigned)blocks, 256, 0, st>>>(p.o, p.dout, p.lse_in, p.delta, p.lse2, p.dq_acc, rows, contig,
                                                     p.N, p.Nr, p.Hq, rs.q_n, rs.q_h, rs.q_b);
  else
    delta_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(p.o, p.dout, p.lse_in, p.delta, p.lse2, p.dq_acc, rows, contig,
                                                     p.N, p.Nr, p.Hq, rs.q_n, rs.q_h, rs.q_b);
  return cudaGetLastError();
}

}  // namespace pa
