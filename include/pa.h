/*
 * pa.h -- C ABI of libpa: packed (block-diagonal causal) attention on GB300.
 *
 * The operation (mlx-train-perf changelog, entry adding
 * `flash_attention(segments=...)` and the PACKED forward, dQ and dK/dV
 * kernels; mlx-train-perf 0.5.1 README, "Sequence packing" and
 * "Flash-attention training path"): several sequences are packed into one
 * row; a per-token int32 segment id says which sequence each token belongs
 * to, and token i attends token j iff j <= i and seg[i] == seg[j]. No (N, N)
 * mask exists anywhere. The forward saves only the output and its
 * log-sum-exp; the backward recomputes attention tile by tile.
 *
 *   S_ij  = scale * <q_i, k_j>           over visible (i, j) only
 *   lse_i = ln sum_j exp(S_ij)
 *   o_i   = sum_j exp(S_ij - lse_i) v_j
 *   and the gradients of o with respect to q, k and v.
 *
 * Layouts (all contiguous, row-major; same README, "If you maintain a
 * trainer": q/k/v are (B, H, N, D), grouped-query heads mapped contiguously):
 *   q, out, dout, dq : (B, Hq,  N, D) bf16
 *   k, v, dk, dv     : (B, Hkv, N, D) bf16;  query head h reads kv head h / (Hq/Hkv)
 *   lse              : (B, Hq,  N)    fp32, natural log
 *   seg              : (B, N)         int32, shared by all heads. Ids are
 *                      compared for equality only: any values are valid.
 *                      Tile skipping is fastest when each id forms one
 *                      contiguous run, which is what packing produces.
 * Head dim 96 (README, "If you maintain a trainer": head_dim in {64, 96,
 * 128}) runs the 128-wide kernels; the tensors stay 96 wide, the tile loads
 * fill columns 96..127 with zeros and the stores leave them out, so a D = 96
 * call takes about as long as a D = 128 one.
 *
 * Ownership: every pointer is device memory owned by the caller. The library
 * allocates no device memory and keeps no pointer after a call returns. The
 * workspace `ws` (pa_workspace_bytes) holds, in this order and each region
 * starting on a 256-byte boundary: the device status word (uint32 at byte
 * 0); the per-tile segment-range table, (B, N/128) int4 {smallest id,
 * largest id, first key tile whose id range overlaps, last query tile whose
 * id range overlaps} at byte 256; two work lists of B*N/128 int32 entries
 * b*(N/128) + t each, the query tiles and then the key tiles ordered by
 * decreasing walk length; then the backward's per-row delta = rowsum(dO * O)
 * and lse * log2(e). For N % 128 != 0 the table and lists describe the
 * padded row (N rounded up to 128).
 *
 * Execution: every call validates its arguments synchronously and returns an
 * error before launching anything; otherwise it enqueues its kernels on
 * `stream` and returns PA_OK without synchronising. Outputs are overwritten,
 * never accumulated into. There is no fallback path: an unsupported shape or
 * device is refused with a typed status (same README, "When it refuses":
 * typed refusals, never silent fallbacks).
 *
 * Device-side waits are bounded; a pipeline that stalls for ~2 s ends its
 * kernel and sets bits in the workspace status word (pa_device_status).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef struct {
  int32_t B;    /* rows (independent packed rows)                    */
  int32_t Hq;   /* query heads                                       */
  int32_t Hkv;  /* key/value heads; Hq % Hkv == 0                    */
  int32_t N;    /* tokens per row (single-step calls: multiple of 128) */
  int32_t D;    /* head dim: 64, 96 or 128                           */
  float scale;  /* softmax scale; <= 0 selects 1/sqrt(D)             */
} pa_dims;

typedef enum {
  PA_OK = 0,
  PA_ERR_NULL = 1,      /* a required pointer is NULL                          */
  PA_ERR_HEAD_DIM = 2,  /* D not in {64, 96, 128}                              */
  PA_ERR_GQA = 3,       /* Hq % Hkv != 0                                       */
  PA_ERR_SHAPE = 4,     /* B, H, N <= 0, sizes overflow int32, a stride < D,
                           or N % 128 != 0 in a single-step call             */
  PA_ERR_ALIGN = 5,     /* a pointer is not 16-byte aligned                    */
  PA_ERR_WORKSPACE = 6, /* ws_bytes < pa_workspace_bytes(dims)                 */
  PA_ERR_ARCH = 7,      /* current device is not compute capability 10.3       */
  PA_ERR_CUDA = 8,      /* a CUDA runtime / driver call or launch failed       */
  PA_ERR_DTYPE = 9,     /* io_dtype is not a pa_io_dtype                       */
  PA_ERR_HOST_MEMORY = 10 /* a host-side call could not allocate its scratch    */
} pa_status;

/* Device status bits (pa_device_status). */
#define PA_DEVERR_TIMEOUT 0x1u /* a bounded wait expired; bits 8.. name the site */
#define PA_DEVERR_DRAIN 0x2u   /* teardown after a timeout could not drain       */
#define PA_DEVERR_SMEM 0x4u    /* a kernel's shared memory was not 1 KiB aligned;
                                  the kernel did no work                          */

/*
 * Workspace size in bytes for `dims` (0 if dims are invalid), for the calls
 * on contiguous tensors. When N is not a multiple of 128 it also includes
 * room for the staging copies described at pa_fwd_strided; the bf16 calls
 * need only the size for N rounded up to 128, which this never undercuts.
 */
size_t pa_workspace_bytes(const pa_dims* dims);

/*
 * Forward. Writes out (B,Hq,N,D) bf16 and lse (B,Hq,N) fp32.
 * seg (B,N) int32 must not be NULL (use pa_fwd_causal for plain causal).
 */
pa_status pa_fwd(const pa_dims* dims, const void* q, const void* k, const void* v, const int32_t* seg,
                 void* out, float* lse, void* ws, size_t ws_bytes, pa_stream_t stream);

/*
 * Backward. Inputs: q, k, v, the forward's out and lse, dout = dL/d(out) and
 * seg. Writes dq (B,Hq,N,D), dk and dv (B,Hkv,N,D), bf16. The gradients of all
 * query heads of a group are summed into their kv head's dk/dv.
 */
pa_status pa_bwd(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                 const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv,
                 void* ws, size_t ws_bytes, pa_stream_t stream);

/*
 * Plain causal variants (mlx-train-perf 0.5.1 README, "If you maintain a
 * trainer": flash_attention(q, k, v, scale=..., causal=True)). They run the
 * same kernels with every token in one segment, so their results are
 * bit-identical to pa_fwd / pa_bwd on an all-equal seg (the changelog states
 * single-segment packed output is bit-identical to the causal kernels).
 */
pa_status pa_fwd_causal(const pa_dims* dims, const void* q, const void* k, const void* v, void* out,
                        float* lse, void* ws, size_t ws_bytes, pa_stream_t stream);
pa_status pa_bwd_causal(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv, void* ws,
                        size_t ws_bytes, pa_stream_t stream);

/*
 * Strided tensors and any N (README, "If you maintain a trainer": q/k/v are
 * (B, H, N, D); a model that holds them as (B, N, H, D) passes that memory
 * with its strides instead of transposing it).
 *
 * Same operation and results as pa_fwd / pa_bwd (seg may be NULL for plain
 * causal), for tensors whose element (b, h, n, c) sits at element offset
 * b*x_b + h*x_h + n*x_n + c: q, out, dout and dq use the q_* strides; k, v,
 * dk and dv the k_* strides. lse stays contiguous (B, Hq, N) fp32 and seg
 * (B, N) int32. Every stride must be >= D and a multiple of 16 bytes (8 bf16
 * or 4 fp32 elements); distinct (b, h, n) rows of an output must not overlap.
 *
 * io_dtype is the element type of q, k, v, out, dout, dq, dk and dv
 * (README, "If you maintain a trainer": the kernels take bf16 or fp32).
 * PA_IO_F32 tensors are rounded to bf16 (nearest even) on the way in and the
 * bf16 results widened exactly on the way out, so an fp32 call returns what
 * the bf16 call returns on the rounded inputs: fp32 is an I/O format here,
 * not a compute precision.
 *
 * How: with bf16 tensors the kernels read and write the caller's tensors in
 * place, whatever their strides and N: they work on Np = N rounded up to
 * 128 tokens through 4-D TMA tensor maps {D, N, H, B} with the given strides,
 * which read the tokens past N as zeros and never store them, and the
 * segment ids are copied into the workspace with the row's last id repeated
 * up to Np (workspace: pa_workspace_bytes for dims with N rounded up to
 * 128). With fp32 tensors the call copies its inputs into bf16 (B, H, Np, D)
 * buffers inside the workspace, runs the kernels there and copies the
 * results out (workspace: pa_workspace_bytes_strided). Either way the extra
 * tokens lie after every real query, so causality hides them; they get zero
 * dO and delta and an infinite lse, so they add nothing to dK and dV, and
 * their outputs are dropped. pa_fwd / pa_bwd and the causal variants take
 * the same in-place path when N % 128 != 0.
 * Errors: as pa_fwd / pa_bwd, plus PA_ERR_NULL (strides), PA_ERR_SHAPE (a
 * stride < D), PA_ERR_ALIGN (a stride not a 16-byte multiple), PA_ERR_DTYPE.
 */
typedef enum { PA_IO_BF16 = 0, PA_IO_F32 = 1 } pa_io_dtype;
typedef struct {
  int64_t q_b, q_h, q_n; /* element strides of q, out, dout, dq */
  int64_t k_b, k_h, k_n; /* element strides of k, v, dk, dv     */
} pa_strides;

size_t pa_workspace_bytes_strided(const pa_dims* dims);
pa_status pa_fwd_strided(const pa_dims* dims, const pa_strides* strides, int32_t io_dtype, const void* q,
                         const void* k, const void* v, const int32_t* seg, void* out, float* lse, void* ws,
                         size_t ws_bytes, pa_stream_t stream);
pa_status pa_bwd_strided(const pa_dims* dims, const pa_strides* strides, int32_t io_dtype, const void* q,
                         const void* k, const void* v, const void* out, const void* dout, const float* lse,
                         const int32_t* seg, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                         pa_stream_t stream);

/*
 * The steps of the path, one kernel each, for callers that schedule or time
 * them individually. pa_fwd is pa_build_tile_table + pa_fwd_tiles; pa_bwd is
 * pa_build_tile_table + pa_bwd_delta + pa_bwd_dq + pa_bwd_dkv, all on one
 * stream, in that order. The later steps read the tile table (and the bwd
 * steps the per-row values of pa_bwd_delta) from `ws`, so they must follow
 * the steps that write it with the same dims and the same seg (NULL seg =
 * plain causal throughout). pa_build_tile_table writes the tile table and
 * the two work lists (the forward, dQ and dK/dV calls take their tiles in
 * that order) and clears the workspace status word. pa_bwd_delta takes the forward's out and lse and stores, per
 * query row, delta = rowsum(dO * O) and lse * log2(e) (the dK/dV step reads
 * that copy; pa_bwd_dkv still validates its lse argument). These calls take
 * contiguous tensors with N % 128 == 0 only (else PA_ERR_SHAPE).
 */
pa_status pa_build_tile_table(const pa_dims* dims, const int32_t* seg, void* ws, size_t ws_bytes,
                              pa_stream_t stream);
pa_status pa_fwd_tiles(const pa_dims* dims, const void* q, const void* k, const void* v, const int32_t* seg,
                       void* out, float* lse, void* ws, size_t ws_bytes, pa_stream_t stream);
pa_status pa_bwd_delta(const pa_dims* dims, const void* out, const void* dout, const float* lse, void* ws,
                       size_t ws_bytes, pa_stream_t stream);
pa_status pa_bwd_dq(const pa_dims* dims, const void* q, const void* k, const void* v, const void* dout,
                    const float* lse, const int32_t* seg, void* dq, void* ws, size_t ws_bytes, pa_stream_t stream);
pa_status pa_bwd_dkv(const pa_dims* dims, const void* q, const void* k, const void* v, const void* dout,
                     const float* lse, const int32_t* seg, void* dk, void* dv, void* ws, size_t ws_bytes,
                     pa_stream_t stream);

/*
 * Single-pass backward (no counterpart on the pages; built to compare with
 * the split dQ / dK-dV design of pa_bwd). One kernel walks the key tiles as
 * pa_bwd_dkv does and also forms each key tile's share of dQ (dS K), which
 * it adds into an fp32 accumulator in the workspace with vector reductions;
 * a last kernel rounds the accumulator to bf16 into dq. Same arguments and
 * operation as pa_bwd; seg may be NULL (plain causal).
 *   - Results: dk and dv are bitwise those of pa_bwd / pa_bwd_causal. dq
 *     matches them within rounding but is not bitwise reproducible from run
 *     to run: the shares of one query row are added in whatever order the
 *     key tiles finish.
 *   - Workspace: pa_bwd_fused_workspace_bytes(dims) = pa_workspace_bytes(dims)
 *     plus B*Hq*N*D*4 bytes for the accumulator (0 if dims are invalid or
 *     N % 128 != 0).
 *   - Errors: as pa_bwd, and PA_ERR_SHAPE when N % 128 != 0 (no staging
 *     copies on this path).
 */
size_t pa_bwd_fused_workspace_bytes(const pa_dims* dims);
pa_status pa_bwd_fused(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv,
                       void* ws, size_t ws_bytes, pa_stream_t stream);

/*
 * Backward without a caller workspace, for callers that cannot allocate device
 * memory when they run it: code inside a region where its allocator or memory
 * pool forbids new allocations, or a host runtime that only hands out its own
 * tensors. The pages have no counterpart; this is a deployment convenience.
 *
 * Same arguments and results as pa_bwd (seg may be NULL for plain causal, as
 * in pa_bwd_causal), minus the workspace: the scratch lives in one static
 * device array of PA_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library, held by
 * every GPU that loads the library until the process exits. The call makes no
 * allocation of any kind.
 *   - Limit: the call runs when pa_workspace_bytes(dims) <=
 *     PA_NOALLOC_SCRATCH_BYTES and is refused with PA_ERR_WORKSPACE
 *     otherwise; compare the two before calling. With N % 128 == 0 that is
 *     about 1 million query rows (B*Hq*N: 8 bytes of scratch per row). With
 *     N % 128 != 0 the workspace also holds the staging copies (about
 *     8*D*(1 + Hkv/Hq) + 12 bytes per query row), which caps it far lower:
 *     roughly 4,000 to 6,500 query rows at D = 128.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents (the call itself resets what must start at zero). Calls whose
 *     kernels overlap on the GPU -- on different streams, or from different
 *     threads -- race on it and corrupt each other's results: serialise them.
 *   - device_status: if not NULL, the call waits for its kernels and stores
 *     the device status word there (0 = healthy, else PA_DEVERR_* bits);
 *     if NULL, the call returns without synchronising.
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
pa_status pa_bwd_noalloc(const pa_dims* dims, const void* q, const void* k, const void* v, const void* out,
                         const void* dout, const float* lse, const int32_t* seg, void* dq, void* dk, void* dv,
                         uint32_t* device_status, pa_stream_t stream);

/*
 * Synchronises `stream`, then returns the workspace's device status word
 * (0 = healthy; PA_DEVERR_* bits otherwise) and clears it. Returns
 * 0xFFFFFFFF if the read itself fails.
 */
uint32_t pa_device_status(const void* ws, pa_stream_t stream);

/*
 * Self-test of the kernels' bounded waits (failure detection without a GPU
 * fault): clears the workspace status word, then launches on `stream` one
 * warp that waits, through the same wait path the kernels use, on an
 * mbarrier that nothing arrives on. After the wait limit (2 s) it gives up,
 * sets PA_DEVERR_TIMEOUT with site 99 in bits 8.. of the status word (the
 * first 4 bytes of `ws`) and exits; the context stays usable. Read the result
 * with pa_device_status.
 * Errors: PA_ERR_NULL (ws), PA_ERR_ALIGN, PA_ERR_WORKSPACE (ws_bytes < 4),
 * PA_ERR_ARCH, PA_ERR_CUDA (launch failed).
 */
pa_status pa_selftest_wait_timeout(void* ws, size_t ws_bytes, pa_stream_t stream);

/*
 * Self-test of the forward's FMA-pipe exponential (the softmax's
 * exp(s - m) taken as 2^t with t = (s - m) log2 e; mlx-train-perf 0.5.1
 * README, "Packed attention"): y[i] = 2^x[i] for n fp32 values, computed on
 * `stream` by the device routine the forward kernel can use for part of
 * its keys (Cody-Waite range reduction and a fitted cubic, no MUFU; the
 * build option PA_FWD_FMA_EX2_PAIRS sets how many, none by default).
 * x and y are device pointers to n floats each (4-byte aligned; the caller
 * owns both). Relative error about 1e-4 for results >= 2^-126; inputs <= -127
 * (and -inf) give +0.0; inputs must be below 128. A lane mismatch inside
 * the routine is reported as a NaN in y.
 * Errors: PA_ERR_SHAPE (n < 0), PA_ERR_NULL, PA_ERR_ALIGN, PA_ERR_ARCH,
 * PA_ERR_CUDA. n == 0 returns PA_OK without a device call.
 */
pa_status pa_selftest_exp2_fma(const float* x, float* y, int64_t n, pa_stream_t stream);

/*
 * Host packer (mlx-train-perf changelog, "Added": the packed batch iterator
 * fills fixed rows with (tokens, offset) sequences after a seeded per-epoch
 * shuffle, by first-fit, and emits per-token segment buffers; the packed loss
 * masks segment by segment, so the supervised tokens are those of an
 * unpacked run, per the 0.5.1 README, "Sequence packing"). Host memory only;
 * no CUDA call is made and no GPU is needed.
 *
 * Inputs (host, caller-owned, read only):
 *   lengths[count]  tokens per sequence, each >= 1. count >= 0.
 *   offsets[count]  prompt length per sequence, each >= 0 (>= length means
 *                   nothing of it is supervised); NULL = all 0.
 *   tokens          the sequences' tokens concatenated in input order
 *                   (sum(lengths) values); needed when row_tokens or
 *                   row_targets is set.
 *   rows, N         the output holds `rows` rows of N tokens (rows, N >= 1).
 *   seed, epoch     the shuffle. Draw n of (seed, epoch) is
 *                   m(k + (n + 1) * 0x9E3779B97F4A7C15), k = m(seed * 1000003
 *                   + epoch), m the splitmix64 output function, all mod 2^64;
 *                   for i = count-1 down to 1, position i swaps with position
 *                   draw(i) mod (i + 1).
 * Placement: in shuffled order, each sequence goes whole into the lowest-
 *   numbered row with room for it, behind that row's earlier sequences; one
 *   that fits no row is left out (placement -1). So the rows in use are a
 *   prefix; to pack a whole epoch, pass rows >= count and cut the result into
 *   batches of B rows.
 * Outputs (host, caller-owned, fully overwritten; all but seg may be NULL):
 *   seg[rows*N]         int32, row-major (rows, N): the sequences of a row are
 *                       segments 0, 1, ... in placement order; the unfilled
 *                       tail of a row (an unused row: all of it) is one more
 *                       segment. This is the attention calls' seg.
 *   loss_mask[rows*N]   1 where the token at that position is trained to
 *                       predict the next token of its own sequence and that
 *                       token is past the prompt: position p (0-based within
 *                       its sequence) with offset <= p + 1 <= length - 1.
 *                       0 elsewhere, padding included.
 *   row_tokens[rows*N]  the packed tokens; pad_token in the padding.
 *   row_targets[rows*N] where loss_mask is 1, the token that position is
 *                       trained to predict (the next token of its own
 *                       sequence); -1 elsewhere, which pa_lce_fwd ignores.
 *   placement[count]    int64 flat index row*N + start of each input
 *                       sequence (input order), or -1 when it was left out.
 *   rows_used           1 + the highest row holding a sequence (0 if none).
 *   placed_tokens       tokens placed in all rows.
 * Errors: PA_ERR_NULL (seg; lengths when count > 0; tokens when row_tokens
 * or row_targets is set and count > 0), PA_ERR_SHAPE (count < 0, rows or N < 1, a length
 * < 1 or an offset < 0), PA_ERR_HOST_MEMORY (its O(count + rows) scratch
 * could not be allocated). Nothing is written on error.
 */
pa_status pa_pack_first_fit(const int32_t* lengths, const int32_t* offsets, int32_t count, const int32_t* tokens,
                            int32_t pad_token, int32_t rows, int32_t N, uint64_t seed, uint64_t epoch,
                            int32_t* seg, uint8_t* loss_mask, int32_t* row_tokens, int32_t* row_targets,
                            int64_t* placement, int32_t* rows_used, int64_t* placed_tokens);

/*
 * Fused linear cross-entropy, forward (mlx-train-perf 0.5.1 README, "The
 * fused cross-entropy loss" and "If you maintain a trainer":
 * linear_cross_entropy(hidden, head, targets)). With logits z = H W^T it
 * writes, per token i,
 *   lse[i]          = log sum_v exp(z[i, v])
 *   target_logit[i] = z[i, targets[i]]
 *   nll[i]          = lse[i] - target_logit[i]
 * without storing z: the tensor cores form 128 x 128 logit tiles in TMEM
 * and the epilogue folds each into a running maximum and sum.
 *   hidden       : (N, D) bf16, row-major      head : (V, D) bf16, row-major
 *   targets      : (N) int32; a target outside [0, V) is ignored: its nll
 *                  and target_logit are 0 (lse is still written)
 *   nll, lse, target_logit : (N) fp32
 * N, V >= 1; D a multiple of 64 in [64, 16384]. Device pointers, caller-owned,
 * 16-byte aligned; ws >= pa_lce_workspace_bytes(N, V, D) bytes (its first 4
 * bytes are the device status word read by pa_device_status). Asynchronous
 * on `stream`, like the attention calls.
 * Errors: PA_ERR_SHAPE, PA_ERR_NULL, PA_ERR_ALIGN, PA_ERR_WORKSPACE,
 * PA_ERR_ARCH, PA_ERR_CUDA.
 */
size_t pa_lce_workspace_bytes(int32_t N, int32_t V, int32_t D);
pa_status pa_lce_fwd(int32_t N, int32_t V, int32_t D, const void* hidden, const void* head, const int32_t* targets,
                     float* nll, float* lse, float* target_logit, void* ws, size_t ws_bytes, pa_stream_t stream);

/*
 * Fused linear cross-entropy, backward (same README section: the backward
 * recomputes the logit tiles it needs instead of reading a stored matrix).
 * For L = sum_i g[i] * nll[i] it writes
 *   dz[i, v]     = g[i] * (exp(z[i, v] - lse[i]) - [v == targets[i]])
 *   dhidden[i]   = sum_v dz[i, v] head[v]          (N, D) bf16, overwritten
 *   dhead[v]     = sum_i dz[i, v] hidden[i]        (V, D) bf16, overwritten;
 *                  pass NULL when the head does not train (then only
 *                  dhidden is computed)
 * lse (N) fp32 is the forward's; g (N) fp32 is dL/dnll per token (for a
 * masked mean, mask[i] / count). A target outside [0, V) contributes
 * nothing (its row of dz is 0, whatever g[i] is).
 * How: the vocabulary is taken in chunks of Vc rows (8192 for N <= 16384,
 * fewer for longer inputs, so that the two dz buffers of a chunk stay within
 * 512 MiB); per chunk one kernel recomputes the chunk's logits on the tensor
 * cores and writes dz in bf16 (tokens x Vc and Vc x tokens), and two tcgen05
 * GEMMs form dhead's rows of the chunk and add the chunk's share of dhidden
 * to an fp32 accumulator in the workspace. The chunks run in a fixed order,
 * so results do not depend on timing. Nothing of size N x V is stored.
 * Arguments as pa_lce_fwd (16-byte aligned device pointers, caller-owned);
 * ws >= pa_lce_bwd_workspace_bytes(N, V, D), its first 4 bytes the status
 * word. Asynchronous on `stream`.
 * Errors: PA_ERR_SHAPE, PA_ERR_NULL, PA_ERR_ALIGN, PA_ERR_WORKSPACE,
 * PA_ERR_ARCH, PA_ERR_CUDA.
 */
size_t pa_lce_bwd_workspace_bytes(int32_t N, int32_t V, int32_t D);
pa_status pa_lce_bwd(int32_t N, int32_t V, int32_t D, const void* hidden, const void* head, const int32_t* targets,
                     const float* lse, const float* g, void* dhidden, void* dhead, void* ws, size_t ws_bytes,
                     pa_stream_t stream);

/* Static, human-readable name of a status code. */
const char* pa_status_string(pa_status s);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
