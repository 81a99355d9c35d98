// Window-aligned sequence parallelism: the host-side plan (no device work).
//
// [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section "Breaking
// the memory wall: window attention across GPUs", "Window-aligned SP": the smallest unit given to
// a GPU is a whole window, with all heads, so attention inside a window never needs another GPU;
// regular and half-shifted window layers alternate, and since the shift moves every window
// boundary, an all-to-all re-homes the tokens to the owners of the new windows at each switch;
// edge windows are cropped to unequal sizes, so dealing out windows by count skews the load.
//
// This file computes, for any number of ranks: which rank owns each window of a layer (greedy
// longest-first on token counts: windows by size descending, ties by id, each to the rank with the
// fewest tokens so far, ties to the lower rank); each rank's local row order (its windows
// ascending, tokens in row-major order inside -- the packed order of the single-GPU path
// restricted to the rank); and the all-to-all of a layer switch as per-rank send lists and receive
// positions.  Everything is O(tokens x ranks) integer work.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "h3attn.h"

namespace {

struct Layer {
  int L[3], w[3], s[3], n[3];
  bool ok = false;
  Layer(const int32_t grid[3], const int32_t win[3], const int32_t shift[3]) {
    if (grid == nullptr || win == nullptr || shift == nullptr) return;
    int64_t total = 1, wins = 1;
    for (int a = 0; a < 3; ++a) {
      if (grid[a] <= 0 || win[a] <= 0 || shift[a] < 0 || shift[a] >= win[a]) return;
      L[a] = grid[a];
      w[a] = win[a];
      s[a] = shift[a];
      n[a] = (grid[a] + shift[a] + win[a] - 1) / win[a];
      total *= grid[a];
      wins *= n[a];
    }
    ok = total <= INT32_MAX && wins <= INT32_MAX;
  }
  int64_t tokens() const { return static_cast<int64_t>(L[0]) * L[1] * L[2]; }
  int32_t windows() const { return n[0] * n[1] * n[2]; }
  // window of token (t, h, w): axis window floor((x + s) / w), lexicographic id
  int32_t window_of(int t, int h, int x) const {
    return ((t + s[0]) / w[0] * n[1] + (h + s[1]) / w[1]) * n[2] + (x + s[2]) / w[2];
  }
  // tokens of window id (product of the cropped axis extents)
  int64_t size_of(int32_t id) const {
    const int i[3] = {id / (n[1] * n[2]), (id / n[2]) % n[1], id % n[2]};
    int64_t sz = 1;
    for (int a = 0; a < 3; ++a) {
      const int lo = std::max(0, i[a] * w[a] - s[a]);
      const int hi = std::min(L[a], (i[a] + 1) * w[a] - s[a]);
      sz *= hi - lo;
    }
    return sz;
  }
  // window id of every token in row-major order
  std::vector<int32_t> token_windows() const {
    std::vector<int32_t> id(static_cast<size_t>(tokens()));
    size_t k = 0;
    for (int t = 0; t < L[0]; ++t)
      for (int h = 0; h < L[1]; ++h)
        for (int x = 0; x < L[2]; ++x) id[k++] = window_of(t, h, x);
    return id;
  }
};

bool ranks_valid(const int32_t* window_rank, int32_t nwin, int32_t world) {
  for (int32_t i = 0; i < nwin; ++i)
    if (window_rank[i] < 0 || window_rank[i] >= world) return false;
  return true;
}

// Local row of every token in its owner's layout: the owner's windows ascending, tokens in
// row-major order inside a window.
std::vector<int32_t> local_positions(const Layer& g, const std::vector<int32_t>& win_of,
                                     const int32_t* window_rank, int32_t world) {
  const int32_t nwin = g.windows();
  std::vector<int64_t> next(static_cast<size_t>(world), 0), start(static_cast<size_t>(nwin));
  for (int32_t i = 0; i < nwin; ++i) {
    start[i] = next[window_rank[i]];
    next[window_rank[i]] += g.size_of(i);
  }
  std::vector<int32_t> pos(win_of.size());
  for (size_t t = 0; t < win_of.size(); ++t) pos[t] = static_cast<int32_t>(start[win_of[t]]++);
  return pos;
}

// Tokens in the global order of a layer's windows (windows ascending, row-major inside).
std::vector<int32_t> window_major_order(const Layer& g, const std::vector<int32_t>& win_of) {
  const int32_t nwin = g.windows();
  std::vector<int64_t> start(static_cast<size_t>(nwin) + 1, 0);
  for (int32_t i = 0; i < nwin; ++i) start[i + 1] = start[i] + g.size_of(i);
  std::vector<int32_t> order(win_of.size());
  for (size_t t = 0; t < win_of.size(); ++t) order[start[win_of[t]]++] = static_cast<int32_t>(t);
  return order;
}

}  // namespace

h3_status h3_sp_assign_windows(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                               int32_t world, int32_t* window_rank, int64_t* rank_tokens) {
  if (grid == nullptr || win == nullptr || shift == nullptr || window_rank == nullptr)
    return H3_ERR_NULL;
  const Layer g(grid, win, shift);
  if (!g.ok || world <= 0) return H3_ERR_INVALID_ARG;
  const int32_t nwin = g.windows();
  std::vector<int32_t> ids(static_cast<size_t>(nwin));
  std::iota(ids.begin(), ids.end(), 0);
  std::vector<int64_t> size(static_cast<size_t>(nwin));
  for (int32_t i = 0; i < nwin; ++i) size[i] = g.size_of(i);
  std::stable_sort(ids.begin(), ids.end(), [&](int32_t a, int32_t b) { return size[a] > size[b]; });
  std::vector<int64_t> load(static_cast<size_t>(world), 0);
  for (int32_t id : ids) {
    int32_t best = 0;
    for (int32_t r = 1; r < world; ++r)
      if (load[r] < load[best]) best = r;
    window_rank[id] = best;
    load[best] += size[id];
  }
  if (rank_tokens != nullptr)
    for (int32_t r = 0; r < world; ++r) rank_tokens[r] = load[r];
  return H3_OK;
}

h3_status h3_sp_rank_tokens(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                            const int32_t* window_rank, int32_t world, int64_t* rank_tokens) {
  if (grid == nullptr || win == nullptr || shift == nullptr || window_rank == nullptr ||
      rank_tokens == nullptr)
    return H3_ERR_NULL;
  const Layer g(grid, win, shift);
  if (!g.ok || world <= 0) return H3_ERR_INVALID_ARG;
  if (!ranks_valid(window_rank, g.windows(), world)) return H3_ERR_INVALID_ARG;
  std::fill(rank_tokens, rank_tokens + world, 0);
  for (int32_t i = 0; i < g.windows(); ++i) rank_tokens[window_rank[i]] += g.size_of(i);
  return H3_OK;
}

h3_status h3_sp_layer_order(const int32_t grid[3], const int32_t win[3], const int32_t shift[3],
                            const int32_t* window_rank, int32_t world, int32_t rank,
                            int32_t* order, int64_t order_capacity) {
  if (grid == nullptr || win == nullptr || shift == nullptr || window_rank == nullptr)
    return H3_ERR_NULL;
  const Layer g(grid, win, shift);
  if (!g.ok || world <= 0 || rank < 0 || rank >= world) return H3_ERR_INVALID_ARG;
  if (!ranks_valid(window_rank, g.windows(), world)) return H3_ERR_INVALID_ARG;
  const std::vector<int32_t> win_of = g.token_windows();
  int64_t n = 0;
  for (int32_t t : window_major_order(g, win_of)) {
    if (window_rank[win_of[t]] != rank) continue;
    if (order == nullptr || n >= order_capacity) return H3_ERR_INVALID_ARG;
    order[n++] = t;
  }
  return H3_OK;
}

h3_status h3_sp_exchange_plan(const int32_t grid[3], const int32_t win[3],
                              const int32_t shift_from[3], const int32_t* rank_from,
                              const int32_t shift_to[3], const int32_t* rank_to, int32_t world,
                              int32_t rank, int64_t* send_counts, int32_t* send_index,
                              int64_t* recv_counts, int32_t* recv_position) {
  if (grid == nullptr || win == nullptr || shift_from == nullptr || shift_to == nullptr ||
      rank_from == nullptr || rank_to == nullptr || send_counts == nullptr ||
      recv_counts == nullptr)
    return H3_ERR_NULL;
  const Layer a(grid, win, shift_from), b(grid, win, shift_to);
  if (!a.ok || !b.ok || world <= 0 || rank < 0 || rank >= world) return H3_ERR_INVALID_ARG;
  if (!ranks_valid(rank_from, a.windows(), world) || !ranks_valid(rank_to, b.windows(), world))
    return H3_ERR_INVALID_ARG;
  const std::vector<int32_t> wa = a.token_windows(), wb = b.token_windows();
  const std::vector<int32_t> pos_a = local_positions(a, wa, rank_from, world);
  const std::vector<int32_t> pos_b = local_positions(b, wb, rank_to, world);
  const std::vector<int32_t> order_b = window_major_order(b, wb);
  // send: this rank's tokens grouped by their new owner, each group in the new owner's order
  std::fill(send_counts, send_counts + world, 0);
  for (int32_t t : order_b)
    if (rank_from[wa[t]] == rank) ++send_counts[rank_to[wb[t]]];
  std::vector<int64_t> cursor(static_cast<size_t>(world), 0);
  for (int32_t d = 1; d < world; ++d) cursor[d] = cursor[d - 1] + send_counts[d - 1];
  const int64_t n_send = cursor[world - 1] + send_counts[world - 1];
  if (n_send > 0 && send_index == nullptr) return H3_ERR_NULL;
  for (int32_t t : order_b)
    if (rank_from[wa[t]] == rank) send_index[cursor[rank_to[wb[t]]]++] = pos_a[t];
  // receive: rows arrive grouped by source rank, each group in this rank's new order
  std::fill(recv_counts, recv_counts + world, 0);
  for (int32_t t : order_b)
    if (rank_to[wb[t]] == rank) ++recv_counts[rank_from[wa[t]]];
  for (int32_t s = 0; s < world; ++s) cursor[s] = s == 0 ? 0 : cursor[s - 1] + recv_counts[s - 1];
  const int64_t n_recv = cursor[world - 1] + recv_counts[world - 1];
  if (n_recv > 0 && recv_position == nullptr) return H3_ERR_NULL;
  for (int32_t t : order_b)
    if (rank_to[wb[t]] == rank) recv_position[cursor[rank_from[wa[t]]]++] = pos_b[t];
  return H3_OK;
}
