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

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Lanes that share one row of the delta kernel: a power of two dividing the
// row's D/8 16-byte vectors, so a row's lanes sit in one warp.
constexpr int delta_lanes(int D) { return (D / 8) % 16 == 0 ? 16 : (D / 8) % 8 == 0 ? 8 : 4; }

template <int D>
__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                    const __nv_bfloat16* __restrict__ dout,
                                                    const float* __restrict__ lse, float* __restrict__ delta,
                                                    float* __restrict__ lse2, size_t rows) {
  // each of the row's LPR lanes takes every LPR-th 16-byte vector
  constexpr int VEC = D / 8;
  constexpr int LPR = delta_lanes(D);
  static_assert(VEC % LPR == 0, "head dim must be a multiple of 32");
  const size_t gtid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const int sub = threadIdx.x % LPR;
  for (size_t t = gtid; t < rows * LPR; t += stride) {
    const size_t row = t / LPR;
    float acc = 0.f;
#pragma unroll
    for (int v = sub; v < VEC; v += LPR) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + v);
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + v);
      acc = fmaf(bf16lo(a.x), bf16lo(c.x), acc);
      acc = fmaf(bf16hi(a.x), bf16hi(c.x), acc);
      acc = fmaf(bf16lo(a.y), bf16lo(c.y), acc);
      acc = fmaf(bf16hi(a.y), bf16hi(c.y), acc);
      acc = fmaf(bf16lo(a.z), bf16lo(c.z), acc);
      acc = fmaf(bf16hi(a.z), bf16hi(c.z), acc);
      acc = fmaf(bf16lo(a.w), bf16lo(c.w), acc);
      acc = fmaf(bf16hi(a.w), bf16hi(c.w), acc);
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(~0u, acc, off);
    if (sub == 0) {
      delta[row] = acc;
      lse2[row] = lse[row] * 1.4426950408889634f;  // for the dK/dV softmax, which works in base 2
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
  const size_t smem = (size_t)p.T * sizeof(int2);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(tile_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  tile_table_kernel<<<p.B, 256, smem, st>>>(p.seg, p.N, p.T, tiles, p.status);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint32_t* status, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_delta(const AttnParams& p, int D, cudaStream_t st) {
  const size_t rows = (size_t)p.B * p.Hq * p.N;
  const size_t threads = rows * (size_t)delta_lanes(D);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t blocks = (threads + 255) / 256;
  const size_t cap = (size_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (D == 128)
    delta_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(p.o, p.dout, p.lse_in, p.delta, p.lse2, rows);
  else if (D == 96)
    delta_kernel<96><<<(unsigned)blocks, 256, 0, st>>>(p.o, p.dout, p.lse_in, p.delta, p.lse2, rows);
  else
    delta_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(p.o, p.dout, p.lse_in, p.delta, p.lse2, rows);
  return cudaGetLastError();
}

}  // namespace pa
