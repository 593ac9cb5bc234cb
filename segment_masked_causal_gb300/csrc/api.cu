// api.cu -- the extern "C" boundary of libpa (declared in include/pa.h).
//
// Every entry point validates its arguments on the host before touching the
// device, refuses anything unsupported with a typed status (no fallback), and
// otherwise enqueues the kernels on the caller's stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <initializer_list>
#include <mutex>

#include "../../include/pa.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Tokens per row as the kernels see them: N rounded up to whole tiles.
inline int padded_n(const pa_dims* d) { return (d->N + pa::kTile - 1) / pa::kTile * pa::kTile; }
inline bool tiled(const pa_dims* d) { return d->N % pa::kTile == 0; }

// The kernels' part (status word, tile table, delta, lse * log2 e) sized for
// padded_n, then the staging copies used when the caller's tensors are not in
// the kernels' layout (N not a multiple of 128, or strided tensors).
struct WsLayout {
  size_t status, tiles, work_q, work_k, delta, lse2, pseg, base;
  size_t sq, sk, sv, so, sdo, sdq, sdk, sdv, slse, sseg, staged;
};

bool dims_ok(const pa_dims* d, pa_status* why) {
  if (!d) { *why = PA_ERR_NULL; return false; }
  if (d->B <= 0 || d->Hq <= 0 || d->Hkv <= 0 || d->N <= 0) { *why = PA_ERR_SHAPE; return false; }
  if (d->D != 64 && d->D != 96 && d->D != 128) { *why = PA_ERR_HEAD_DIM; return false; }
  if (d->Hq % d->Hkv != 0) { *why = PA_ERR_GQA; return false; }
  // tensor-map row coordinates and tile counts are 32-bit
  const int64_t rows = (int64_t)d->B * d->Hq * padded_n(d);
  if (d->N > (1 << 30) || rows >= (int64_t(1) << 31) || (int64_t)padded_n(d) / pa::kTile > 65535 * 2) {
    *why = PA_ERR_SHAPE;
    return false;
  }
  if (!(std::isfinite(d->scale))) { *why = PA_ERR_SHAPE; return false; }
  return true;
}

WsLayout ws_layout(const pa_dims* d) {
  WsLayout w;
  const size_t Np = (size_t)padded_n(d), T = Np / pa::kTile;
  const size_t qrows = (size_t)d->B * d->Hq * Np, krows = (size_t)d->B * d->Hkv * Np;
  const size_t qb = round_up(qrows * d->D * 2), kb = round_up(krows * d->D * 2);
  w.status = 0;
  w.tiles = kAlign;
  w.work_q = w.tiles + round_up((size_t)d->B * T * sizeof(int4));
  w.work_k = w.work_q + round_up((size_t)d->B * T * sizeof(int32_t));
  w.delta = w.work_k + round_up((size_t)d->B * T * sizeof(int32_t));
  w.lse2 = w.delta + round_up(qrows * sizeof(float));
  w.pseg = w.lse2 + round_up(qrows * sizeof(float));  // segment ids padded to whole tiles (ragged N)
  w.base = w.pseg + round_up((size_t)d->B * Np * sizeof(int32_t));
  w.sq = w.base;
  w.so = w.sq + qb;
  w.sdo = w.so + qb;
  w.sdq = w.sdo + qb;
  w.sk = w.sdq + qb;
  w.sv = w.sk + kb;
  w.sdk = w.sv + kb;
  w.sdv = w.sdk + kb;
  w.slse = w.sdv + kb;
  w.sseg = w.slse + round_up(qrows * sizeof(float));
  w.staged = w.sseg + round_up((size_t)d->B * Np * sizeof(int32_t));
  return w;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status device_ok() { return pa::device_check(); }

}  // namespace

// Per-device: compute capability 10.3 and enough opt-in shared memory.
pa_status pa::device_check() {
  static std::mutex mu;
  static int checked[64] = {0};  // 0 unknown, 1 ok, 2 refused
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PA_ERR_ARCH;
  std::lock_guard<std::mutex> lk(mu);
  if (checked[dev] == 0) {
    int maj = 0, min = 0, smem = 0;
    if (cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    checked[dev] = (maj == 10 && min == 3 && smem >= 232448) ? 1 : 2;
  }
  return checked[dev] == 1 ? PA_OK : PA_ERR_ARCH;
}

namespace {

// d holds the kernels' N (whole tiles); Nr > 0 is the caller's N when it is
// not a whole number of tiles.
pa::AttnParams make_params(const pa_dims* d, const int32_t* seg, void* ws, int Nr = 0) {
  pa::AttnParams p{};
  p.B = d->B; p.Hq = d->Hq; p.Hkv = d->Hkv; p.N = d->N; p.T = d->N / pa::kTile; p.G = d->Hq / d->Hkv;
  p.Nr = Nr > 0 ? Nr : d->N;
  p.scale = d->scale > 0.f ? d->scale : 1.f / std::sqrt((float)d->D);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.seg = seg;
  const WsLayout w = ws_layout(d);
  uint8_t* base = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<uint32_t*>(base + w.status);
  p.tiles = reinterpret_cast<const int4*>(base + w.tiles);
  p.work_q = reinterpret_cast<const int32_t*>(base + w.work_q);
  p.work_k = reinterpret_cast<const int32_t*>(base + w.work_k);
  p.delta = reinterpret_cast<float*>(base + w.delta);
  p.lse2 = reinterpret_cast<float*>(base + w.lse2);
  return p;
}

// The kernels run on the caller's tensors directly only when N is a whole
// number of tiles; the single-step calls require that.
pa_status common_checks(const pa_dims* d, void* ws, size_t ws_bytes) {
  pa_status why = PA_OK;
  if (!dims_ok(d, &why)) return why;
  if (!tiled(d)) return PA_ERR_SHAPE;
  if (!ws) return PA_ERR_NULL;
  if (!aligned16(ws)) return PA_ERR_ALIGN;
  if (ws_bytes < ws_layout(d).base) return PA_ERR_WORKSPACE;
  return PA_OK;
}

// Validation shared by every call: dims, workspace, then the given pointers
// (all required, 16-byte aligned), then the device.
pa_status check_call(const pa_dims* d, void* ws, size_t ws_bytes, std::initializer_list<const void*> required,
                     const int32_t* seg) {
  pa_status s = common_checks(d, ws, ws_bytes);
  if (s != PA_OK) return s;
  for (const void* x : required)
    if (!x) return PA_ERR_NULL;
  for (const void* x : required)
    if (!aligned16(x)) return PA_ERR_ALIGN;
  if (seg && !aligned16(seg)) return PA_ERR_ALIGN;
  return device_ok();
}

inline cudaStream_t cu(pa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// The kernels' view of the caller's (B, H, N, D) tensors: the given strides,
// or contiguous ones.
pa::RowStrides rows_of(const pa_dims* d, const pa_strides* s) {
  if (!s) return pa::contiguous_rows(d->Hq, d->Hkv, d->N, d->D);
  return pa::RowStrides{s->q_n, s->q_h, s->q_b, s->k_n, s->k_h, s->k_b};
}
inline pa::RowStrides rows_or(const pa_dims* d, const pa::RowStrides* rs) {
  return rs ? *rs : pa::contiguous_rows(d->Hq, d->Hkv, d->N, d->D);
}

pa_status step_tile_table(const pa_dims* d, const int32_t* seg, void* ws, size_t ws_bytes, pa_stream_t stream) {
  pa_status s = check_call(d, ws, ws_bytes, {}, seg);
  if (s != PA_OK) return s;
  pa::AttnParams p = make_params(d, seg, ws);
  return pa::launch_tile_table(p, const_cast<int4*>(p.tiles), cu(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status step_fwd(const pa_dims* d, const void* q, const void* k, const void* v, const int32_t* seg, void* out,
                   float* lse, void* ws, size_t ws_bytes, pa_stream_t stream, const pa::RowStrides* rs = nullptr,
                   int Nr = 0) {
  pa_status s = check_call(d, ws, ws_bytes, {q, k, v, out, lse}, seg);
  if (s != PA_OK) return s;
  pa::AttnParams p = make_params(d, seg, ws, Nr);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  return pa::launch_fwd(p, d->D, rows_or(d, rs), q, k, v, cu(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status step_delta(const pa_dims* d, const void* out, const void* dout, const float* lse, void* ws,
                     size_t ws_bytes, pa_stream_t stream, const pa::RowStrides* rs = nullptr, int Nr = 0) {
  pa_status s = check_call(d, ws, ws_bytes, {out, dout, lse}, nullptr);
  if (s != PA_OK) return s;
  pa::AttnParams p = make_params(d, nullptr, ws, Nr);
  p.lse_in = lse;
  p.o = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  return pa::launch_delta(p, d->D, rows_or(d, rs), cu(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status step_dq(const pa_dims* d, const void* q, const void* k, const void* v, const void* dout,
                  const float* lse, const int32_t* seg, void* dq, void* ws, size_t ws_bytes, pa_stream_t stream,
                  const pa::RowStrides* rs = nullptr, int Nr = 0) {
  pa_status s = check_call(d, ws, ws_bytes, {q, k, v, dout, lse, dq}, seg);
  if (s != PA_OK) return s;
  pa::AttnParams p = make_params(d, seg, ws, Nr);
  p.lse_in = lse;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  return pa::launch_bwd_dq(p, d->D, rows_or(d, rs), q, k, v, dout, cu(stream)) == cudaSuccess ? PA_OK
                                                                                             : PA_ERR_CUDA;
}

pa_status step_dkv(const pa_dims* d, const void* q, const void* k, const void* v, const void* dout,
                   const float* lse, const int32_t* seg, void* dk, void* dv, void* ws, size_t ws_bytes,
                   pa_stream_t stream, const pa::RowStrides* rs = nullptr, int Nr = 0) {
  pa_status s = check_call(d, ws, ws_bytes, {q, k, v, dout, lse, dk, dv}, seg);
  if (s != PA_OK) return s;
  pa::AttnParams p = make_params(d, seg, ws, Nr);
  p.lse_in = lse;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  return pa::launch_bwd_dkv(p, d->D, rows_or(d, rs), q, k, v, dout, cu(stream)) == cudaSuccess ? PA_OK
                                                                                              : PA_ERR_CUDA;
}

pa_status fwd_impl(const pa_dims* d, const void* q, const void* k, const void* v, const int32_t* seg, void* out,
                   float* lse, void* ws, size_t ws_bytes, pa_stream_t stream, const pa::RowStrides* rs = nullptr,
                   int Nr = 0) {
  pa_status s = check_call(d, ws, ws_bytes, {q, k, v, out, lse}, seg);
  if (s != PA_OK) return s;
  if ((s = step_tile_table(d, seg, ws, ws_bytes, stream)) != PA_OK) return s;
  return step_fwd(d, q, k, v, seg, out, lse, ws, ws_bytes, stream, rs, Nr);
}

pa_status bwd_impl(const pa_dims* d, const void* q, const void* k, const void* v, const void* out,
                   const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv, void* ws,
                   size_t ws_bytes, pa_stream_t stream, const pa::RowStrides* rs = nullptr, int Nr = 0) {
  pa_status s = check_call(d, ws, ws_bytes, {q, k, v, out, dout, lse, dq, dk, dv}, seg);
  if (s != PA_OK) return s;
  if ((s = step_tile_table(d, seg, ws, ws_bytes, stream)) != PA_OK) return s;
  if ((s = step_delta(d, out, dout, lse, ws, ws_bytes, stream, rs, Nr)) != PA_OK) return s;
  if ((s = step_dq(d, q, k, v, dout, lse, seg, dq, ws, ws_bytes, stream, rs, Nr)) != PA_OK) return s;
  return step_dkv(d, q, k, v, dout, lse, seg, dk, dv, ws, ws_bytes, stream, rs, Nr);
}

// bf16 tensors whose N is not a whole number of tiles: the kernels run on
// N rounded up to 128 (dp), reading the caller's tensors through 4-D maps
// whose N extent is the real N (the tail reads as zeros and is never
// stored), with the segment ids copied into the workspace padded by the
// row's last id.
struct Ragged {
  pa_dims dp;
  pa::RowStrides rs;
  const int32_t* pseg;
};
pa_status ragged_prepare(const pa_dims* d, const pa_strides* s, const int32_t* seg, void* ws, size_t ws_bytes,
                         std::initializer_list<const void*> required, pa_stream_t stream, Ragged* r) {
  r->dp = *d;
  r->dp.N = padded_n(d);
  r->rs = rows_of(d, s);
  pa_status st = check_call(&r->dp, ws, ws_bytes, required, seg);
  if (st != PA_OK) return st;
  r->pseg = nullptr;
  if (seg) {
    int32_t* pseg = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + ws_layout(&r->dp).pseg);
    if (pa::launch_stage_words_in(pseg, seg, (uint64_t)d->B, d->N, r->dp.N, true, cu(stream)) != cudaSuccess)
      return PA_ERR_CUDA;
    r->pseg = pseg;
  }
  return PA_OK;
}

// Single-pass backward: the fp32 dQ accumulator sits after the kernels'
// part of the workspace.
size_t fused_acc_offset(const pa_dims* d) { return round_up(ws_layout(d).base); }
size_t fused_ws_bytes(const pa_dims* d) {
  return fused_acc_offset(d) + round_up((size_t)d->B * d->Hq * d->N * d->D * sizeof(float));
}

pa_status bwd_fused_impl(const pa_dims* d, const void* q, const void* k, const void* v, const void* out,
                         const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv,
                         void* ws, size_t ws_bytes, pa_stream_t stream) {
  pa_status s = check_call(d, ws, ws_bytes, {q, k, v, out, dout, lse, dq, dk, dv}, seg);
  if (s != PA_OK) return s;
  if (ws_bytes < fused_ws_bytes(d)) return PA_ERR_WORKSPACE;
  if ((s = step_tile_table(d, seg, ws, ws_bytes, stream)) != PA_OK) return s;
  pa::AttnParams p = make_params(d, seg, ws);
  p.lse_in = lse;
  p.o = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_acc = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + fused_acc_offset(d));
  p.dq_ld = d->D;
  const cudaStream_t st = cu(stream);
  const pa::RowStrides rs = rows_of(d, nullptr);
  if (pa::launch_delta(p, d->D, rs, st) != cudaSuccess ||
      pa::launch_bwd_fused(p, d->D, rs, q, k, v, dout, st) != cudaSuccess ||
      pa::launch_dq_round(p, d->D, st) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

// ------------------------------------------------------------ staged calls
// Element strides of the q group (q, out, dout, dq) and the k group (k, v,
// dk, dv); D is contiguous.
pa_strides contiguous_strides(const pa_dims* d) {
  pa_strides s;
  s.q_n = s.k_n = d->D;
  s.q_h = s.k_h = (int64_t)d->N * d->D;
  s.q_b = (int64_t)d->Hq * d->N * d->D;
  s.k_b = (int64_t)d->Hkv * d->N * d->D;
  return s;
}

// Strides of at least D elements that keep every row 16-byte aligned.
pa_status strides_ok(const pa_dims* d, const pa_strides* s, bool f32) {
  if (!s) return PA_ERR_NULL;
  for (int64_t x : {s->q_b, s->q_h, s->q_n, s->k_b, s->k_h, s->k_n})
    if (x < d->D) return PA_ERR_SHAPE;
  for (int64_t x : {s->q_b, s->q_h, s->q_n, s->k_b, s->k_h, s->k_n})
    if (x % (f32 ? 4 : 8) != 0) return PA_ERR_ALIGN;
  return PA_OK;
}

// Validation of a staged call: dims (any N), strides, the staged workspace,
// the pointers, the device.
pa_status check_staged(const pa_dims* d, const pa_strides* s, bool f32, void* ws, size_t ws_bytes,
                       std::initializer_list<const void*> required, const int32_t* seg) {
  pa_status why = PA_OK;
  if (!dims_ok(d, &why)) return why;
  if ((why = strides_ok(d, s, f32)) != PA_OK) return why;
  if (!ws) return PA_ERR_NULL;
  if (!aligned16(ws)) return PA_ERR_ALIGN;
  if (ws_bytes < ws_layout(d).staged) return PA_ERR_WORKSPACE;
  for (const void* x : required)
    if (!x) return PA_ERR_NULL;
  for (const void* x : required)
    if (!aligned16(x)) return PA_ERR_ALIGN;
  if (seg && !aligned16(seg)) return PA_ERR_ALIGN;
  return device_ok();
}

struct Staging {
  pa_dims dp;  // the kernels' dims: N padded to whole tiles
  pa::RowsView vq, vk;
  uint8_t* w;
  WsLayout L;
  Staging(const pa_dims* d, const pa_strides* s, void* ws) : dp(*d), w(static_cast<uint8_t*>(ws)), L(ws_layout(d)) {
    dp.N = padded_n(d);
    vq = pa::RowsView{d->B, d->Hq, d->N, dp.N, d->D / 8, s->q_b, s->q_h, s->q_n};
    vk = pa::RowsView{d->B, d->Hkv, d->N, dp.N, d->D / 8, s->k_b, s->k_h, s->k_n};
  }
  void* at(size_t off) const { return w + off; }
};

pa_status fwd_staged(const pa_dims* d, const pa_strides* s, bool f32, const void* q, const void* k, const void* v,
                     const int32_t* seg, void* out, float* lse, void* ws, size_t ws_bytes, pa_stream_t stream) {
  pa_status st = check_staged(d, s, f32, ws, ws_bytes, {q, k, v, out, lse}, seg);
  if (st != PA_OK) return st;
  const Staging g(d, s, ws);
  const cudaStream_t cs = cu(stream);
  const uint64_t qr = (uint64_t)d->B * d->Hq;
  if (pa::launch_stage_rows_in(g.at(g.L.sq), q, g.vq, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_in(g.at(g.L.sk), k, g.vk, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_in(g.at(g.L.sv), v, g.vk, f32, cs) != cudaSuccess ||
      (seg && pa::launch_stage_words_in(g.at(g.L.sseg), seg, (uint64_t)d->B, d->N, g.dp.N, true, cs) != cudaSuccess))
    return PA_ERR_CUDA;
  const int32_t* sseg = seg ? static_cast<const int32_t*>(g.at(g.L.sseg)) : nullptr;
  st = fwd_impl(&g.dp, g.at(g.L.sq), g.at(g.L.sk), g.at(g.L.sv), sseg, g.at(g.L.so),
                static_cast<float*>(g.at(g.L.slse)), ws, ws_bytes, stream);
  if (st != PA_OK) return st;
  if (pa::launch_stage_rows_out(out, g.at(g.L.so), g.vq, f32, cs) != cudaSuccess ||
      pa::launch_stage_words_out(lse, g.at(g.L.slse), qr, d->N, g.dp.N, cs) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status bwd_staged(const pa_dims* d, const pa_strides* s, bool f32, const void* q, const void* k, const void* v,
                     const void* out, const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk,
                     void* dv, void* ws, size_t ws_bytes, pa_stream_t stream) {
  pa_status st = check_staged(d, s, f32, ws, ws_bytes, {q, k, v, out, dout, lse, dq, dk, dv}, seg);
  if (st != PA_OK) return st;
  const Staging g(d, s, ws);
  const cudaStream_t cs = cu(stream);
  const uint64_t qr = (uint64_t)d->B * d->Hq;
  if (pa::launch_stage_rows_in(g.at(g.L.sq), q, g.vq, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_in(g.at(g.L.sk), k, g.vk, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_in(g.at(g.L.sv), v, g.vk, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_in(g.at(g.L.so), out, g.vq, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_in(g.at(g.L.sdo), dout, g.vq, f32, cs) != cudaSuccess ||
      pa::launch_stage_words_in(g.at(g.L.slse), lse, qr, d->N, g.dp.N, false, cs) != cudaSuccess ||
      (seg && pa::launch_stage_words_in(g.at(g.L.sseg), seg, (uint64_t)d->B, d->N, g.dp.N, true, cs) != cudaSuccess))
    return PA_ERR_CUDA;
  const int32_t* sseg = seg ? static_cast<const int32_t*>(g.at(g.L.sseg)) : nullptr;
  st = bwd_impl(&g.dp, g.at(g.L.sq), g.at(g.L.sk), g.at(g.L.sv), g.at(g.L.so), g.at(g.L.sdo),
                static_cast<const float*>(g.at(g.L.slse)), sseg, g.at(g.L.sdq), g.at(g.L.sdk), g.at(g.L.sdv), ws,
                ws_bytes, stream);
  if (st != PA_OK) return st;
  if (pa::launch_stage_rows_out(dq, g.at(g.L.sdq), g.vq, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_out(dk, g.at(g.L.sdk), g.vk, f32, cs) != cudaSuccess ||
      pa::launch_stage_rows_out(dv, g.at(g.L.sdv), g.vk, f32, cs) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

// The public forward and backward: the kernels run on the caller's tensors
// when they are contiguous bf16 and N is whole tiles, else through the
// staging copies.
pa_status io_ok(int32_t io_dtype) {
  return (io_dtype == PA_IO_BF16 || io_dtype == PA_IO_F32) ? PA_OK : PA_ERR_DTYPE;
}

pa_status fwd_any(const pa_dims* d, const pa_strides* s, int32_t io, const void* q, const void* k, const void* v,
                  const int32_t* seg, void* out, float* lse, void* ws, size_t ws_bytes, pa_stream_t stream) {
  pa_status why = PA_OK;
  if (!dims_ok(d, &why)) return why;
  if ((why = io_ok(io)) != PA_OK) return why;
  const bool f32 = io == PA_IO_F32;
  if (s && (why = strides_ok(d, s, f32)) != PA_OK) return why;
  if (!f32 && tiled(d)) {
    const pa::RowStrides rs = rows_of(d, s);
    return fwd_impl(d, q, k, v, seg, out, lse, ws, ws_bytes, stream, &rs);
  }
  if (!f32) {
    Ragged r;
    pa_status st = ragged_prepare(d, s, seg, ws, ws_bytes, {q, k, v, out, lse}, stream, &r);
    if (st != PA_OK) return st;
    return fwd_impl(&r.dp, q, k, v, r.pseg, out, lse, ws, ws_bytes, stream, &r.rs, d->N);
  }
  const pa_strides c = contiguous_strides(d);
  return fwd_staged(d, s ? s : &c, f32, q, k, v, seg, out, lse, ws, ws_bytes, stream);
}

pa_status bwd_any(const pa_dims* d, const pa_strides* s, int32_t io, const void* q, const void* k, const void* v,
                  const void* out, const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk,
                  void* dv, void* ws, size_t ws_bytes, pa_stream_t stream) {
  pa_status why = PA_OK;
  if (!dims_ok(d, &why)) return why;
  if ((why = io_ok(io)) != PA_OK) return why;
  const bool f32 = io == PA_IO_F32;
  if (s && (why = strides_ok(d, s, f32)) != PA_OK) return why;
  if (!f32 && tiled(d)) {
    const pa::RowStrides rs = rows_of(d, s);
    return bwd_impl(d, q, k, v, out, dout, lse, seg, dq, dk, dv, ws, ws_bytes, stream, &rs);
  }
  if (!f32) {
    Ragged r;
    pa_status st = ragged_prepare(d, s, seg, ws, ws_bytes, {q, k, v, out, dout, lse, dq, dk, dv}, stream, &r);
    if (st != PA_OK) return st;
    return bwd_impl(&r.dp, q, k, v, out, dout, lse, r.pseg, dq, dk, dv, ws, ws_bytes, stream, &r.rs, d->N);
  }
  const pa_strides c = contiguous_strides(d);
  return bwd_staged(d, s ? s : &c, f32, q, k, v, out, dout, lse, seg, dq, dk, dv, ws, ws_bytes, stream);
}

}  // namespace

extern "C" {

size_t pa_workspace_bytes(const pa_dims* dims) {
  pa_status why;
  if (!dims_ok(dims, &why)) return 0;
  const WsLayout w = ws_layout(dims);
  return tiled(dims) ? w.base : w.staged;
}

size_t pa_workspace_bytes_strided(const pa_dims* dims) {
  pa_status why;
  if (!dims_ok(dims, &why)) return 0;
  return ws_layout(dims).staged;
}

pa_status pa_fwd_strided(const pa_dims* dims, const pa_strides* strides, int32_t io_dtype, const void* q,
                         const void* k, const void* v, const int32_t* seg, void* out, float* lse, void* ws,
                         size_t ws_bytes, pa_stream_t stream) {
  if (!strides) return PA_ERR_NULL;
  return fwd_any(dims, strides, io_dtype, q, k, v, seg, out, lse, ws, ws_bytes, stream);
}

pa_status pa_bwd_strided(const pa_dims* dims, const pa_strides* strides, int32_t io_dtype, const void* q,
                         const void* k, const void* v, const void* out, const void* dout, const float* lse,
                         const int32_t* seg, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                         pa_stream_t stream) {
  if (!strides) return PA_ERR_NULL;
  return bwd_any(dims, strides, io_dtype, q, k, v, out, dout, lse, seg, dq, dk, dv, ws, ws_bytes, stream);
}

pa_status pa_fwd(const pa_dims* dims, const void* q, const void* k, const void* v, const int32_t* seg, void* out,
                 float* lse, void* ws, size_t ws_bytes, pa_stream_t stream) {
  if (!seg) return PA_ERR_NULL;
  return fwd_any(dims, nullptr, PA_IO_BF16, q, k, v, seg, out, lse, ws, ws_bytes, stream);
}

pa_status pa_fwd_causal(const pa_dims* dims, const void* q, const void* k, const void* v, void* out, float* lse,
                        void* ws, size_t ws_bytes, pa_stream_t stream) {
  return fwd_any(dims, nullptr, PA_IO_BF16, q, k, v, nullptr, out, lse, ws, ws_bytes, stream);
}

pa_status pa_bwd(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                 const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv, void* ws,
                 size_t ws_bytes, pa_stream_t stream) {
  if (!seg) return PA_ERR_NULL;
  return bwd_any(dims, nullptr, PA_IO_BF16, q, k, v, out, dout, lse, seg, dq, dk, dv, ws, ws_bytes, stream);
}

pa_status pa_bwd_causal(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, void* ws,
                        size_t ws_bytes, pa_stream_t stream) {
  return bwd_any(dims, nullptr, PA_IO_BF16, q, k, v, out, dout, lse, nullptr, dq, dk, dv, ws, ws_bytes, stream);
}

size_t pa_bwd_fused_workspace_bytes(const pa_dims* dims) {
  pa_status why;
  if (!dims_ok(dims, &why) || !tiled(dims)) return 0;
  return fused_ws_bytes(dims);
}

pa_status pa_bwd_fused(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv,
                       void* ws, size_t ws_bytes, pa_stream_t stream) {
  return bwd_fused_impl(dims, q, k, v, out, dout, lse, seg, dq, dk, dv, ws, ws_bytes, stream);
}

pa_status pa_build_tile_table(const pa_dims* dims, const int32_t* seg, void* ws, size_t ws_bytes,
                              pa_stream_t stream) {
  return step_tile_table(dims, seg, ws, ws_bytes, stream);
}

pa_status pa_fwd_tiles(const pa_dims* dims, const void* q, const void* k, const void* v, const int32_t* seg,
                       void* out, float* lse, void* ws, size_t ws_bytes, pa_stream_t stream) {
  return step_fwd(dims, q, k, v, seg, out, lse, ws, ws_bytes, stream);
}

pa_status pa_bwd_delta(const pa_dims* dims, const void* out, const void* dout, const float* lse, void* ws,
                       size_t ws_bytes, pa_stream_t stream) {
  return step_delta(dims, out, dout, lse, ws, ws_bytes, stream);
}

pa_status pa_bwd_dq(const pa_dims* dims, const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, const int32_t* seg, void* dq, void* ws, size_t ws_bytes, pa_stream_t stream) {
  return step_dq(dims, q, k, v, dout, lse, seg, dq, ws, ws_bytes, stream);
}

pa_status pa_bwd_dkv(const pa_dims* dims, const void* q, const void* k, const void* v, const void* dout,
                     const float* lse, const int32_t* seg, void* dk, void* dv, void* ws, size_t ws_bytes,
                     pa_stream_t stream) {
  return step_dkv(dims, q, k, v, dout, lse, seg, dk, dv, ws, ws_bytes, stream);
}

// ------------------------------------------------------ linear cross-entropy
static bool lce_dims_ok(int32_t N, int32_t V, int32_t D) {
  return N > 0 && V > 0 && D >= 64 && D <= 16384 && D % 64 == 0;
}

size_t pa_lce_workspace_bytes(int32_t N, int32_t V, int32_t D) {
  if (!lce_dims_ok(N, V, D)) return 0;
  // partial sums for the largest split count lce_split may choose
  const int VT = (V + pa::kTile - 1) / pa::kTile;
  const size_t splits = VT < pa::kLceMaxSplits ? VT : pa::kLceMaxSplits;
  return kAlign + round_up((size_t)3 * splits * N * sizeof(float));
}

pa_status pa_lce_fwd(int32_t N, int32_t V, int32_t D, const void* hidden, const void* head, const int32_t* targets,
                     float* nll, float* lse, float* target_logit, void* ws, size_t ws_bytes, pa_stream_t stream) {
  if (!lce_dims_ok(N, V, D)) return PA_ERR_SHAPE;
  for (const void* x : {hidden, head, (const void*)targets, (const void*)nll, (const void*)lse,
                        (const void*)target_logit, (const void*)ws})
    if (!x) return PA_ERR_NULL;
  for (const void* x : {hidden, head, (const void*)targets, (const void*)nll, (const void*)lse,
                        (const void*)target_logit, (const void*)ws})
    if (!aligned16(x)) return PA_ERR_ALIGN;
  if (ws_bytes < pa_lce_workspace_bytes(N, V, D)) return PA_ERR_WORKSPACE;
  pa_status why = device_ok();
  if (why != PA_OK) return why;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess) return PA_ERR_CUDA;
  return pa::launch_lce_fwd(N, V, D, hidden, head, targets, nll, lse, target_logit,
                            reinterpret_cast<float*>(w + kAlign), reinterpret_cast<uint32_t*>(w), st) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

size_t pa_lce_bwd_workspace_bytes(int32_t N, int32_t V, int32_t D) {
  if (!lce_dims_ok(N, V, D)) return 0;
  return pa::lce_bwd_layout(N, V, D).bytes;
}

pa_status pa_lce_bwd(int32_t N, int32_t V, int32_t D, const void* hidden, const void* head, const int32_t* targets,
                     const float* lse, const float* g, void* dhidden, void* dhead, void* ws, size_t ws_bytes,
                     pa_stream_t stream) {
  if (!lce_dims_ok(N, V, D)) return PA_ERR_SHAPE;
  const void* req[] = {hidden, head, targets, lse, g, dhidden, ws};
  for (const void* x : req)
    if (!x) return PA_ERR_NULL;
  for (const void* x : req)
    if (!aligned16(x)) return PA_ERR_ALIGN;
  if (dhead && !aligned16(dhead)) return PA_ERR_ALIGN;
  if (ws_bytes < pa_lce_bwd_workspace_bytes(N, V, D)) return PA_ERR_WORKSPACE;
  pa_status why = device_ok();
  if (why != PA_OK) return why;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess) return PA_ERR_CUDA;
  return pa::launch_lce_bwd(N, V, D, hidden, head, targets, lse, g, dhidden, dhead, ws,
                            static_cast<uint32_t*>(ws), st) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_selftest_wait_timeout(void* ws, size_t ws_bytes, pa_stream_t stream) {
  if (!ws) return PA_ERR_NULL;
  if (!aligned16(ws)) return PA_ERR_ALIGN;
  if (ws_bytes < sizeof(uint32_t)) return PA_ERR_WORKSPACE;
  pa_status why = device_ok();
  if (why != PA_OK) return why;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess ||
      pa::launch_wait_timeout_selftest(static_cast<uint32_t*>(ws), st) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status pa_selftest_exp2_fma(const float* x, float* y, int64_t n, pa_stream_t stream) {
  if (n < 0) return PA_ERR_SHAPE;
  if (n == 0) return PA_OK;
  if (!x || !y) return PA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 3u) return PA_ERR_ALIGN;
  pa_status why = device_ok();
  if (why != PA_OK) return why;
  return pa::launch_exp2_fma_selftest(x, y, n, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                                     : PA_ERR_CUDA;
}

uint32_t pa_device_status(const void* ws, pa_stream_t stream) {
  if (!ws) return 0xFFFFFFFFu;
  uint32_t h = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return 0xFFFFFFFFu;
  if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return 0xFFFFFFFFu;
  const uint32_t zero = 0;
  if (cudaMemcpy(const_cast<void*>(ws), &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return 0xFFFFFFFFu;
  return h;
}

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_HEAD_DIM: return "head dim must be 64, 96 or 128";
    case PA_ERR_GQA: return "Hq must be a multiple of Hkv";
    case PA_ERR_SHAPE:
      return "bad shape (B, H, N > 0; B*Hq*N < 2^31; finite scale; N % 128 == 0 for the single-step calls; "
             "strides >= D)";
    case PA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case PA_ERR_WORKSPACE: return "workspace too small (see pa_workspace_bytes)";
    case PA_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case PA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case PA_ERR_DTYPE: return "io dtype must be PA_IO_BF16 or PA_IO_F32";
    case PA_ERR_HOST_MEMORY: return "host memory for the call's scratch could not be allocated";
  }
  return "unknown status";
}

}  // extern "C"
