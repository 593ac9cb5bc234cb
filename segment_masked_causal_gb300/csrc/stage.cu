// stage.cu -- copies between the caller's tensors and the kernels' layout.
//
// The attention kernels read and write contiguous (B, H, Np, D) tensors whose
// rows are a whole number of 128-token tiles (Np = N rounded up to 128). When
// a caller's N is not a multiple of 128, or its tensors are strided (for
// instance (B, N, H, D) memory viewed as (B, H, N, D)), the public calls copy
// the inputs into that layout inside the workspace, run the kernels there and
// copy the results back. These are plain memory-bound copies: 16-byte vectors,
// grid-stride loops over the destination (inputs) or the source (outputs).
//
// Tail tokens n in [N, Np) are zero rows (q, k, v, o, dO), lse 0, and the
// last real segment id: a tail query then has dO = 0 and delta = 0, so it adds
// nothing to any key's dK or dV, and a tail key lies after every real query,
// so causality hides it from all of them. The tail's own outputs are dropped.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace pa {
namespace {

// dst (R, Np, VEC) uint4 <- src strided rows; zeros for n >= N.
__global__ void __launch_bounds__(256) stage_rows_in_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                            RowsView v) {
  const uint64_t total = (uint64_t)v.B * v.H * v.Np * v.vec;
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += step) {
    const uint64_t row = u / v.vec;
    const int c = (int)(u - row * v.vec);
    const uint64_t r = row / v.Np;
    const int n = (int)(row - r * v.Np);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (n < v.N) {
      const uint64_t b = r / v.H, h = r - b * v.H;
      x = __ldg(src + (b * v.sb + h * v.sh + (uint64_t)n * v.sn) / 8 + c);
    }
    dst[u] = x;
  }
}

// dst strided rows <- src (R, Np, VEC) uint4, real tokens only.
__global__ void __launch_bounds__(256) stage_rows_out_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                             RowsView v) {
  const uint64_t total = (uint64_t)v.B * v.H * v.N * v.vec;
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += step) {
    const uint64_t row = u / v.vec;
    const int c = (int)(u - row * v.vec);
    const uint64_t r = row / v.N;
    const int n = (int)(row - r * v.N);
    const uint64_t b = r / v.H, h = r - b * v.H;
    dst[(b * v.sb + h * v.sh + (uint64_t)n * v.sn) / 8 + c] = __ldg(src + (r * v.Np + n) * v.vec + c);
  }
}

// (R, Np) 32-bit words <- (R, N); the tail is 0 or the row's last word.
__global__ void __launch_bounds__(256) stage_words_in_kernel(uint32_t* __restrict__ dst,
                                                             const uint32_t* __restrict__ src, uint64_t R, int N,
                                                             int Np, int repeat_last) {
  const uint64_t total = R * (uint64_t)Np;
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += step) {
    const uint64_t r = u / Np;
    const int n = (int)(u - r * Np);
    dst[u] = n < N ? __ldg(src + r * N + n) : (repeat_last ? __ldg(src + r * N + (N - 1)) : 0u);
  }
}

// (R, N) 32-bit words <- (R, Np).
__global__ void __launch_bounds__(256) stage_words_out_kernel(uint32_t* __restrict__ dst,
                                                              const uint32_t* __restrict__ src, uint64_t R, int N,
                                                              int Np) {
  const uint64_t total = R * (uint64_t)N;
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += step) {
    const uint64_t r = u / N;
    const int n = (int)(u - r * N);
    dst[u] = __ldg(src + r * Np + n);
  }
}

unsigned grid_for(uint64_t units) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (units + 255) / 256;
  const uint64_t cap = (uint64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  return (unsigned)(blocks ? blocks : 1);
}

}  // namespace

cudaError_t launch_stage_rows_in(void* dst, const void* src, const RowsView& v, cudaStream_t st) {
  const uint64_t units = (uint64_t)v.B * v.H * v.Np * v.vec;
  if (units == 0) return cudaSuccess;
  stage_rows_in_kernel<<<grid_for(units), 256, 0, st>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src), v);
  return cudaGetLastError();
}

cudaError_t launch_stage_rows_out(void* dst, const void* src, const RowsView& v, cudaStream_t st) {
  const uint64_t units = (uint64_t)v.B * v.H * v.N * v.vec;
  if (units == 0) return cudaSuccess;
  stage_rows_out_kernel<<<grid_for(units), 256, 0, st>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                                         v);
  return cudaGetLastError();
}

cudaError_t launch_stage_words_in(void* dst, const void* src, uint64_t R, int N, int Np, bool repeat_last,
                                  cudaStream_t st) {
  stage_words_in_kernel<<<grid_for(R * (uint64_t)Np), 256, 0, st>>>(
      static_cast<uint32_t*>(dst), static_cast<const uint32_t*>(src), R, N, Np, repeat_last ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_stage_words_out(void* dst, const void* src, uint64_t R, int N, int Np, cudaStream_t st) {
  stage_words_out_kernel<<<grid_for(R * (uint64_t)N), 256, 0, st>>>(static_cast<uint32_t*>(dst),
                                                                     static_cast<const uint32_t*>(src), R, N, Np);
  return cudaGetLastError();
}

}  // namespace pa
