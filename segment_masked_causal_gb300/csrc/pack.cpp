// pack.cpp -- host packer: variable-length (tokens, offset) sequences into
// fixed rows, with the per-token segment ids the attention kernels read and a
// per-token supervision mask for the loss.
//
// mlx-train-perf changelog, "Added": the packed batch iterator places
// (tokens, offset) sequences into fixed rows after a seeded per-epoch shuffle,
// by first-fit, and hands out per-token segment buffers with each batch; the
// packed loss masks segment by segment so that the supervised tokens are those
// of an unpacked run (0.5.1 README, "Sequence packing").
//
// Host code only; no CUDA call is made.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "pa.h"

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

// The splitmix64 output function (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014).
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Draw n (n >= 0) of the counter-based stream for (seed, epoch).
struct EpochStream {
  uint64_t key;
  EpochStream(uint64_t seed, uint64_t epoch) : key(mix64(seed * 1000003ull + epoch)) {}
  uint64_t draw(uint64_t n) const { return mix64(key + (n + 1) * kGamma); }
};

// First-fit in O(log R) per item: a max-tree over the rows' free space; the
// leftmost row with room is found by walking down from the root.
class FreeTree {
 public:
  FreeTree(int32_t rows, int64_t cap) {
    leaves_ = 1;
    while (leaves_ < rows) leaves_ <<= 1;
    t_.assign(2 * (size_t)leaves_, -1);
    for (int32_t r = 0; r < rows; ++r) t_[leaves_ + r] = cap;
    for (int64_t i = leaves_ - 1; i >= 1; --i) t_[i] = t_[2 * i] > t_[2 * i + 1] ? t_[2 * i] : t_[2 * i + 1];
  }
  // leftmost row whose free space is >= need, or -1
  int32_t first_fit(int64_t need) const {
    if (t_[1] < need) return -1;
    int64_t i = 1;
    while (i < leaves_) i = (t_[2 * i] >= need) ? 2 * i : 2 * i + 1;
    return (int32_t)(i - leaves_);
  }
  void take(int32_t row, int64_t amount) {
    int64_t i = leaves_ + row;
    t_[i] -= amount;
    for (i >>= 1; i >= 1; i >>= 1) t_[i] = t_[2 * i] > t_[2 * i + 1] ? t_[2 * i] : t_[2 * i + 1];
  }

 private:
  int64_t leaves_;
  std::vector<int64_t> t_;
};

// Everything that allocates runs before the first write to an output, so an
// allocation failure leaves the outputs untouched.
pa_status pack(const int32_t* lengths, const int32_t* offsets, int32_t count, const int32_t* tokens,
               int32_t pad_token, int32_t rows, int32_t N, uint64_t seed, uint64_t epoch, int32_t* seg,
               uint8_t* loss_mask, int32_t* row_tokens, int32_t* row_targets, int64_t* placement,
               int32_t* rows_used, int64_t* placed_tokens) {
  // where each sequence's tokens start in the concatenated `tokens`
  std::vector<int64_t> src(count);
  int64_t total = 0;
  for (int32_t i = 0; i < count; ++i) {
    src[i] = total;
    total += lengths[i];
  }

  // the epoch's order: Fisher-Yates, step i swapping with draw(i) mod (i+1)
  std::vector<int32_t> order(count);
  for (int32_t i = 0; i < count; ++i) order[i] = i;
  const EpochStream rng(seed, epoch);
  for (int32_t i = count - 1; i > 0; --i) {
    const int32_t j = (int32_t)(rng.draw((uint64_t)i) % (uint64_t)(i + 1));
    const int32_t t = order[i];
    order[i] = order[j];
    order[j] = t;
  }

  FreeTree tree(rows, N);
  std::vector<int64_t> used(rows, 0);
  std::vector<int32_t> nseg(rows, 0);

  const int64_t cells = (int64_t)rows * N;
  if (loss_mask) std::memset(loss_mask, 0, (size_t)cells);
  if (row_tokens)
    for (int64_t k = 0; k < cells; ++k) row_tokens[k] = pad_token;
  if (row_targets)
    for (int64_t k = 0; k < cells; ++k) row_targets[k] = -1;
  if (placement)
    for (int32_t i = 0; i < count; ++i) placement[i] = -1;
  int64_t placed = 0;
  int32_t last_row = -1;
  for (const int32_t s : order) {
    const int32_t L = lengths[s];
    const int32_t r = tree.first_fit(L);
    if (r < 0) continue;  // fits no row: left out of this epoch
    tree.take(r, L);
    const int64_t base = (int64_t)r * N + used[r];
    const int32_t id = nseg[r]++;
    for (int32_t p = 0; p < L; ++p) seg[base + p] = id;
    // Position p predicts token p + 1 of the same sequence; it is supervised
    // when that token is past the prompt: offset <= p + 1 <= L - 1.
    const int32_t off = offsets ? offsets[s] : 0;
    for (int32_t p = (off > 1 ? off - 1 : 0); p + 1 < L; ++p) {
      if (loss_mask) loss_mask[base + p] = 1;
      if (row_targets) row_targets[base + p] = tokens[src[s] + p + 1];
    }
    if (row_tokens) std::memcpy(row_tokens + base, tokens + src[s], sizeof(int32_t) * (size_t)L);
    if (placement) placement[s] = base;
    used[r] += L;
    placed += L;
    if (r > last_row) last_row = r;
  }
  // each row's unfilled tail is one further segment: padding, never supervised
  for (int32_t r = 0; r < rows; ++r)
    for (int64_t t = used[r]; t < N; ++t) seg[(int64_t)r * N + t] = nseg[r];
  if (rows_used) *rows_used = last_row + 1;
  if (placed_tokens) *placed_tokens = placed;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_pack_first_fit(const int32_t* lengths, const int32_t* offsets, int32_t count,
                                       const int32_t* tokens, int32_t pad_token, int32_t rows, int32_t N,
                                       uint64_t seed, uint64_t epoch, int32_t* seg, uint8_t* loss_mask,
                                       int32_t* row_tokens, int32_t* row_targets, int64_t* placement,
                                       int32_t* rows_used, int64_t* placed_tokens) {
  if (!seg || (count > 0 && !lengths) || ((row_tokens || row_targets) && count > 0 && !tokens)) return PA_ERR_NULL;
  if (count < 0 || rows <= 0 || N <= 0) return PA_ERR_SHAPE;
  for (int32_t i = 0; i < count; ++i)
    if (lengths[i] <= 0 || (offsets && offsets[i] < 0)) return PA_ERR_SHAPE;
  // no C++ exception may cross the C boundary: the scratch vectors' allocation
  // is the only thing here that can throw
  try {
    return pack(lengths, offsets, count, tokens, pad_token, rows, N, seed, epoch, seg, loss_mask, row_tokens,
                row_targets, placement, rows_used, placed_tokens);
  } catch (const std::bad_alloc&) {
    return PA_ERR_HOST_MEMORY;
  }
}
