// noalloc.cu -- pa_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) when they run the
// backward pass. Examples are code inside a region that a custom allocator or
// a memory pool forbids from allocating, runtimes that hand out only their
// own tensors, and plugins that must not touch the device heap. pa_bwd needs
// a caller-supplied workspace for its scratch (the segment-range tile table,
// the per-row delta and a status word); this entry point uses a fixed array
// compiled into the library instead, so the caller passes only its inputs and
// outputs.
//
// The array is a file-scope __device__ variable of kScratchBytes (8 MiB).
// Every GPU that loads this library holds it until the process exits. In host
// code its name is only a host-side stand-in, never a device address, so its
// device address is looked up once per device, with that device current, by
// cudaGetSymbolAddress, and that pointer is what the kernels receive.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "kernels.h"

constexpr size_t kScratchBytes = size_t(8) << 20;
static_assert(kScratchBytes == PA_NOALLOC_SCRATCH_BYTES, "header and array size disagree");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set-up on first use).
pa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_ARCH;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_bwd_noalloc(const pa_dims* dims, const void* q, const void* k, const void* v,
                                    const void* out, const void* dout, const float* lse, const int32_t* seg,
                                    void* dq, void* dk, void* dv, uint32_t* device_status, pa_stream_t stream) {
  const size_t need = pa_workspace_bytes(dims);
  if (need == 0)  // invalid dims: let the regular entry point (causal when seg is NULL) name the reason
    return seg ? pa_bwd(dims, q, k, v, out, dout, lse, seg, dq, dk, dv, nullptr, 0, stream)
               : pa_bwd_causal(dims, q, k, v, out, dout, lse, dq, dk, dv, nullptr, 0, stream);
  if (need > kScratchBytes) return PA_ERR_WORKSPACE;
  // The same device check as every other entry point, before the symbol
  // lookup: on a device this library has no code for, that lookup would fail
  // with a generic CUDA error instead of PA_ERR_ARCH.
  pa_status s = pa::device_check();
  if (s != PA_OK) return s;
  void* scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != PA_OK) return s;
  // Nothing needs clearing here: the tile-table kernel zeroes the status word
  // and every later kernel overwrites the table, work lists and delta it reads.
  s = seg ? pa_bwd(dims, q, k, v, out, dout, lse, seg, dq, dk, dv, scratch, kScratchBytes, stream)
          : pa_bwd_causal(dims, q, k, v, out, dout, lse, dq, dk, dv, scratch, kScratchBytes, stream);
  if (s != PA_OK || !device_status) return s;
  // status word is the first 4 bytes of the workspace layout
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemcpy(device_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
