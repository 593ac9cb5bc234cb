// kernels.h -- host-side launchers of the packed-attention kernels (internal).
#pragma once
#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "common.cuh"

namespace pa {

// PA_OK when the current device is compute capability 10.3 with enough
// opt-in shared memory for the kernels, else PA_ERR_ARCH (or PA_ERR_CUDA if
// the query itself fails). Cached per device.
pa_status device_check();

// Element strides of the (B, H, N, D) tensors the kernels read and write in
// place (D contiguous): q, out, dout and dq use the q_* strides, k, v, dk and
// dv the k_* strides.
struct RowStrides {
  int64_t q_n, q_h, q_b, k_n, k_h, k_b;
};
inline RowStrides contiguous_rows(int Hq, int Hkv, int N, int D) {
  return RowStrides{D, (int64_t)N * D, (int64_t)Hq * N * D, D, (int64_t)N * D, (int64_t)Hkv * N * D};
}
inline bool is_contiguous(const RowStrides& s, int Hq, int Hkv, int N, int D) {
  const RowStrides c = contiguous_rows(Hq, Hkv, N, D);
  return s.q_n == c.q_n && s.q_h == c.q_h && s.q_b == c.q_b && s.k_n == c.k_n && s.k_h == c.k_h && s.k_b == c.k_b;
}

// Tile table (B, T) x {smin, smax, kv_lo, q_hi} and the two work lists; also
// clears the status word.
cudaError_t launch_tile_table(const AttnParams& p, int4* tiles, cudaStream_t st);
// delta[b, h, i] = sum_c dO[b, h, i, c] * O[b, h, i, c] (fp32), and lse2 = lse * log2(e);
// also zeroes the rows of p.dq_acc when it is non-null.
cudaError_t launch_delta(const AttnParams& p, int D, const RowStrides& rs, cudaStream_t st);
// Self-test of the bounded waits: one warp waits on an mbarrier nothing arrives on.
cudaError_t launch_wait_timeout_selftest(uint32_t* status, cudaStream_t st);
cudaError_t launch_exp2_fma_selftest(const float* x, float* y, int64_t n, cudaStream_t st);
cudaError_t launch_fwd(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k, const void* v,
                       cudaStream_t st);
cudaError_t launch_bwd_dq(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k,
                          const void* v, const void* dout, cudaStream_t st);
cudaError_t launch_bwd_dkv(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k,
                           const void* v, const void* dout, cudaStream_t st);
// Single-pass backward: dK, dV and the fp32 dQ accumulator p.dq_acc (zeroed
// beforehand), then p.dq = the accumulator rounded to bf16.
cudaError_t launch_bwd_fused(const AttnParams& p, int D, const RowStrides& rs, const void* q, const void* k,
                             const void* v, const void* dout, cudaStream_t st);
cudaError_t launch_dq_round(const AttnParams& p, int D, cudaStream_t st);

// A (B, H, N, D) bf16 or fp32 tensor with element strides sb, sh, sn (16-byte
// multiples) and contiguous D, against the kernels' contiguous bf16
// (B, H, Np, D) copy; vec = D / 8 bf16 16-byte vectors per token row.
struct RowsView {
  int B, H, N, Np, vec;
  int64_t sb, sh, sn;
};
// Copies in (tail rows n >= N zero) and out (real rows only); f32: the
// caller's tensor is fp32 (rounded to bf16 in, widened out).
cudaError_t launch_stage_rows_in(void* dst, const void* src, const RowsView& v, bool f32, cudaStream_t st);
cudaError_t launch_stage_rows_out(void* dst, const void* src, const RowsView& v, bool f32, cudaStream_t st);
// (R, N) 32-bit words to (R, Np) with a tail of 0 or of the row's last word, and back.
cudaError_t launch_stage_words_in(void* dst, const void* src, uint64_t R, int N, int Np, bool repeat_last,
                                  cudaStream_t st);
cudaError_t launch_stage_words_out(void* dst, const void* src, uint64_t R, int N, int Np, cudaStream_t st);

// Fused linear cross-entropy forward. The vocabulary's 128-row tiles are cut
// into `splits` runs of `per` tiles, one CTA column each; `part` holds
// 3 * splits * N floats of per-split partial results.
struct LceSplit {
  int splits, per;
};
constexpr int kLceMaxSplits = 64;
LceSplit lce_split(int N, int V, int slots);
// CTAs of the cross-entropy kernel resident at once on the current device.
int lce_slots();
// Fused linear cross-entropy backward: the vocabulary in chunks of vc rows;
// workspace after the 256-byte status region: the fp32 dH accumulator (only
// with more than one chunk), dz (N x vc) and dz^T (vc x ld_dzt), bf16.
struct LceBwdLayout {
  int vc, chunks, ld_dzt;
  size_t acc, dz, dzt, bytes;
};
LceBwdLayout lce_bwd_layout(int N, int V, int D);
cudaError_t launch_lce_bwd(int N, int V, int D, const void* hidden, const void* head, const int32_t* targets,
                           const float* lse, const float* g, void* dhidden, void* dhead, void* ws, uint32_t* status,
                           cudaStream_t st);
cudaError_t launch_lce_fwd(int N, int V, int D, const void* hidden, const void* head, const int32_t* targets,
                           float* nll, float* lse, float* target_logit, float* part, uint32_t* status,
                           cudaStream_t st);

}  // namespace pa
