// kernels.h -- host-side launchers of the packed-attention kernels (internal).
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace pa {

// Tile table (B, T) x {smin, smax, kv_lo, q_hi}; also clears the status word.
cudaError_t launch_tile_table(const AttnParams& p, int4* tiles, cudaStream_t st);
// delta[b, h, i] = sum_c dO[b, h, i, c] * O[b, h, i, c] (fp32), and lse2 = lse * log2(e).
cudaError_t launch_delta(const AttnParams& p, int D, cudaStream_t st);
// Self-test of the bounded waits: one warp waits on an mbarrier nothing arrives on.
cudaError_t launch_wait_timeout_selftest(uint32_t* status, cudaStream_t st);
cudaError_t launch_fwd(const AttnParams& p, int D, const void* q, const void* k, const void* v, cudaStream_t st);
cudaError_t launch_bwd_dq(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                          const void* dout, cudaStream_t st);
cudaError_t launch_bwd_dkv(const AttnParams& p, int D, const void* q, const void* k, const void* v,
                           const void* dout, cudaStream_t st);

}  // namespace pa
