// stage.cu -- copies between the caller's tensors and the kernels' layout.
//
// The attention kernels read and write contiguous (B, H, Np, D) tensors whose
// rows are a whole number of 128-token tiles (Np = N rounded up to 128). When
// a caller's N is not a multiple of 128, or its tensors are strided (for
// instance (B, N, H, D) memory viewed as (B, H, N, D)), the public calls copy
// the inputs into that layout inside the workspace, run the kernels there and
// copy the results back. The same copies take fp32 tensors: inputs are rounded
// to bf16 (nearest even) on the way in and bf16 results widened exactly on the
// way out. These are plain memory-bound copies: 16-byte bf16 vectors in
// grid-stride loops over the destination (inputs) or the source (outputs).
//
// Tail tokens n in [N, Np) are zero rows (q, k, v, o, dO), lse 0, and the
// last real segment id: a tail query then has dO = 0 and delta = 0, so it adds
// nothing to any key's dK or dV, and a tail key lies after every real query,
// so causality hides it from all of them. The tail's own outputs are dropped.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"

namespace pa {
namespace {

// One 16-byte vector of 8 bf16 from element offset e (a multiple of 8) of
// a bf16 tensor, or of 8 fp32 values (rounded to nearest even) from a float
// tensor (e a multiple of 4).
__device__ __forceinline__ uint4 load8(const uint16_t* src, uint64_t e) {
  return __ldg(reinterpret_cast<const uint4*>(src + e));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 load8(const float* src, uint64_t e) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(src + e));
  const float4 b = __ldg(reinterpret_cast<const float4*>(src + e) + 1);
  return make_uint4(pack2(a.x, a.y), pack2(a.z, a.w), pack2(b.x, b.y), pack2(b.z, b.w));
}
__device__ __forceinline__ void store8(uint16_t* dst, uint64_t e, uint4 x) {
  *reinterpret_cast<uint4*>(dst + e) = x;
}
__device__ __forceinline__ void store8(float* dst, uint64_t e, uint4 x) {
  // bf16 -> fp32 is exact: the bf16 bits are the float's top half
  float4* d = reinterpret_cast<float4*>(dst + e);
  d[0] = make_float4(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xFFFF0000u), __uint_as_float(x.y << 16),
                     __uint_as_float(x.y & 0xFFFF0000u));
  d[1] = make_float4(__uint_as_float(x.z << 16), __uint_as_float(x.z & 0xFFFF0000u), __uint_as_float(x.w << 16),
                     __uint_as_float(x.w & 0xFFFF0000u));
}

// dst (R, Np, VEC) bf16 vectors <- src strided rows of T; zeros for n >= N.
template <typename T>
__global__ void __launch_bounds__(256) stage_rows_in_kernel(uint4* __restrict__ dst, const T* __restrict__ src,
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
      x = load8(src, b * v.sb + h * v.sh + (uint64_t)n * v.sn + (uint64_t)c * 8);
    }
    dst[u] = x;
  }
}

// dst strided rows of T <- src (R, Np, VEC) bf16 vectors, real tokens only.
template <typename T>
__global__ void __launch_bounds__(256) stage_rows_out_kernel(T* __restrict__ dst, const uint4* __restrict__ src,
                                                             RowsView v) {
  const uint64_t total = (uint64_t)v.B * v.H * v.N * v.vec;
  const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t u = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; u < total; u += step) {
    const uint64_t row = u / v.vec;
    const int c = (int)(u - row * v.vec);
    const uint64_t r = row / v.N;
    const int n = (int)(row - r * v.N);
    const uint64_t b = r / v.H, h = r - b * v.H;
    store8(dst, b * v.sb + h * v.sh + (uint64_t)n * v.sn + (uint64_t)c * 8, __ldg(src + (r * v.Np + n) * v.vec + c));
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

cudaError_t launch_stage_rows_in(void* dst, const void* src, const RowsView& v, bool f32, cudaStream_t st) {
  const uint64_t units = (uint64_t)v.B * v.H * v.Np * v.vec;
  if (units == 0) return cudaSuccess;
  if (f32)
    stage_rows_in_kernel<float><<<grid_for(units), 256, 0, st>>>(static_cast<uint4*>(dst),
                                                                 static_cast<const float*>(src), v);
  else
    stage_rows_in_kernel<uint16_t><<<grid_for(units), 256, 0, st>>>(static_cast<uint4*>(dst),
                                                                    static_cast<const uint16_t*>(src), v);
  return cudaGetLastError();
}

cudaError_t launch_stage_rows_out(void* dst, const void* src, const RowsView& v, bool f32, cudaStream_t st) {
  const uint64_t units = (uint64_t)v.B * v.H * v.N * v.vec;
  if (units == 0) return cudaSuccess;
  if (f32)
    stage_rows_out_kernel<float><<<grid_for(units), 256, 0, st>>>(static_cast<float*>(dst),
                                                                  static_cast<const uint4*>(src), v);
  else
    stage_rows_out_kernel<uint16_t><<<grid_for(units), 256, 0, st>>>(static_cast<uint16_t*>(dst),
                                                                     static_cast<const uint4*>(src), v);
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
