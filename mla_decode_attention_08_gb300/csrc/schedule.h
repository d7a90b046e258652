// Integer formulas of the token-balanced split-KV schedule, shared by the host
// planner and the kernels so both compute the same ranges.
//
// Rows are cut into tiles of kTileTokens tokens; all rows' tiles, row after
// row (each row with tiles preceded by row_start_units units for its start),
// form one sequence of T units; worker c of a grid of G takes the units
// [floor(c*T/G), floor((c+1)*T/G)).  This is the persistent form of the
// flash-decoding split (kernelbot-amd-mixed-mla submission 722089,
// `_mla_multihead_stage1` splits each row into contiguous ranges; submissions
// 663509 and 738050 hand a persistent kernel precomputed work maps).
#pragma once
#include <cstdint>

#ifdef __CUDACC__
#define MLA_HD __host__ __device__ __forceinline__
#else
#define MLA_HD inline
#endif

namespace mla {

constexpr int kNumHeads = 16;
constexpr int kQkDim = 576;
constexpr int kVDim = 512;
constexpr int kTileTokens = 128;

MLA_HD int32_t tiles_of_length(int64_t len) {
  return len > 0 ? static_cast<int32_t>((len + kTileTokens - 1) / kTileTokens) : 0;
}

// Workers for a batch: the fewest that still give no worker more than
// k = ceil(U / min(num_sms, U)) tiles, U = B * ceil(max_kv_len / 128), i.e.
// ceil(U / k).  Fewer workers than SMs when that does not lengthen the longest
// range: the ranges then hold k tiles each and, for rows of a multiple of k
// tiles, start at row starts (bs 32 x 1024: 128 workers of two tiles instead
// of 152 of one or two, some of which straddle two rows).
MLA_HD int32_t plan_grid(int32_t batch, int32_t max_kv_len, int32_t num_sms) {
  const int64_t upper = static_cast<int64_t>(batch) * tiles_of_length(max_kv_len);
  const int64_t g0 = upper < num_sms ? upper : num_sms;
  if (g0 < 1) return 1;
  const int64_t k = (upper + g0 - 1) / g0;
  return static_cast<int32_t>((upper + k - 1) / k);
}

// Clusters of s CTAs (one 227 KB CTA per SM) that a GPU of num_sms SMs runs at
// once, estimated from the GB300 GPC layout (measured: 15 clusters of 8, 36 of
// 4 and 76 of 2 on 152 SMs): num_sms / 10, 7 num_sms / 32 and num_sms / 2.
MLA_HD int32_t cluster_capacity(int32_t s, int32_t num_sms) {
  return s == 8 ? num_sms / 10 : (s == 4 ? num_sms * 7 / 32 : num_sms / 2);
}

// Cluster split for small batches of one query token per row: every row gets
// a cluster of s CTAs that share its tiles (rank r takes the row's tiles
// [r k, min((r + 1) k, nt)), k = ceil(nt / s)) and combine their partial
// results after one cluster barrier, with no second kernel.  s is the
// largest of 8, 4, 2 with s <= ceil(max_kv_len / 128) whose clusters for the
// whole batch fit the GPU at once; it is used (else 0: the persistent split)
// when its longest share, ceil(nt / s) tiles, is at most two tiles longer than
// the persistent schedule's longest range.
MLA_HD int32_t plan_cluster(int32_t batch, int32_t qo_len, int32_t max_kv_len, int32_t num_sms) {
  const int32_t nt = tiles_of_length(max_kv_len);
  if (qo_len != 1 || batch < 1 || num_sms < 1 || nt < 2) return 0;
  int32_t s = 8;
  while (s >= 2 && (s > nt || batch > cluster_capacity(s, num_sms))) s >>= 1;
  if (s < 2) return 0;
  const int64_t upper = static_cast<int64_t>(batch) * nt;
  const int64_t g0 = upper < num_sms ? upper : num_sms;
  const int64_t longest = (upper + g0 - 1) / g0;
  return (nt + s - 1) / s <= longest + 2 ? s : 0;
}

// Row starts.  A worker whose range takes on a new row pays for that row's
// start (its query's preparation and the previous segment's epilogue, about
// three tiles' streaming time) on top of its tiles, and such workers finished
// last.  So when the ranges are long, every row with tiles is preceded in the
// global sequence by kRowStartUnits units that stand for its start: a range
// that takes on a row start gets that many fewer tiles.  With short ranges
// (fewer than kRowStartMinRange tiles each) the units would cost more than
// they balance (ranges of 2 tiles become 2 or 3), and rows start with their
// tiles.  The rule depends only on the batch's tile count T and the grid:
// units per row start = kRowStartUnits when ceil(T / grid) >= kRowStartMinRange,
// else 0 (e4m3 and MXFP4 caches; a bf16 cache's rows start with their tiles).
constexpr int32_t kRowStartUnits = 3;
constexpr int32_t kRowStartMinRange = 8;
MLA_HD int32_t row_start_units(int32_t total_tiles, int32_t grid) {
  if (grid < 1 || total_tiles < 1) return 0;
  const int64_t k = (static_cast<int64_t>(total_tiles) + grid - 1) / grid;
  return k >= kRowStartMinRange ? kRowStartUnits : 0;
}

// floor(c * total / grid) for 0 <= c <= grid and total >= 0, without a 64-bit
// division (a slow call on the GPU): with total = q * grid + r it is
// c * q + floor(c * r / grid), and c * r < grid^2 fits 32 bits whenever
// grid < 65536.
MLA_HD int32_t worker_begin(int32_t c, int32_t total, int32_t grid) {
  const uint32_t g = static_cast<uint32_t>(grid);
  const uint32_t q = static_cast<uint32_t>(total) / g, r = static_cast<uint32_t>(total) % g;
  const uint64_t cr = static_cast<uint64_t>(c) * r;
  const uint32_t extra = cr <= 0xFFFFFFFFull ? static_cast<uint32_t>(cr) / g
                                             : static_cast<uint32_t>(cr / g);
  return static_cast<int32_t>(static_cast<uint32_t>(c) * q + extra);
}

// Worker holding global tile t (0 <= t < total): the largest c with
// worker_begin(c) <= t, i.e. floor(((t + 1) * grid - 1) / total).  A float
// estimate is stepped to the exact answer with worker_begin.
MLA_HD int32_t worker_of_tile(int32_t t, int32_t total, int32_t grid) {
  int32_t c = static_cast<int32_t>(static_cast<float>(t) * static_cast<float>(grid) /
                                   static_cast<float>(total));
  c = c < 0 ? 0 : (c > grid - 1 ? grid - 1 : c);
  while (c > 0 && worker_begin(c, total, grid) > t) --c;
  while (c + 1 < grid && worker_begin(c + 1, total, grid) <= t) ++c;
  return c;
}

// Workspace slot of worker c's partial for a split row whose tiles start at
// prefix_b: slot 2c when c's range begins inside that row, else 2c + 1.
MLA_HD int32_t partial_slot(int32_t c, int32_t worker_t0, int32_t prefix_b) {
  return worker_t0 >= prefix_b ? 2 * c : 2 * c + 1;
}

}  // namespace mla
