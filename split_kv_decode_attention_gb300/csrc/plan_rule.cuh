// plan_rule.cuh -- the split planner's rule: how many KV chunks each
// (request, kv head) is cut into, and how long they are, from the batch's
// lengths against the number of CTAs the split launch keeps resident.
//
// One rule, two callers: the host planner (decode_attn_plan /
// decode_attn_plan_slots, api.cu) and the device planner kernel
// (plan_kernel.cu) that a graph-capturable decode_attn call with device-only
// lengths runs first.  Both evaluate this same code; they differ only in how
// chunks_of(c) -- the number of (request, kv head, chunk) work items at chunk
// length c -- is summed over the requests (a host loop, or a block-wide
// reduction).  The reason for splitting at all is "Capstone FlashAttention",
// §2.3 FlashDecoding: with few (request, head) pairs the SMs starve unless the
// KV sequence itself is cut into chunks that run on different SMs.
#pragma once

#include <stdint.h>

namespace dattn {

// A chunk is never shorter than this many tokens (partials and the combine
// cost ~1.5 KB per row per chunk; a 16 KB+ chunk read keeps that small).
constexpr int kMinChunkTokens = 256;
// Ragged batches: chunks are sized for this many waves of resident CTAs over
// the batch's total work, and hold at least kTokensPerRow tokens per query row
// (fit on GB300 sweeps of chunk length: ~1-2K tokens for 4-16 rows).
constexpr int kRaggedWaves = 8;
constexpr int kTokensPerRow = 64;
// The tcgen05 kernel (17..128 rows) pays ~3 us per work item (epilogue,
// the two softmax groups' merge) and writes 512 B of partial output per row
// of a split item, so its chunks hold four times as many tokens per row.
// (GB300, 64 rows: one chunk per request 198 us against two 205 us; 128
// rows keep two chunks, where the floor gives way to filling the SMs.)
constexpr int kWideTokensPerRow = 256;
// Largest thread-block cluster the split kernel uses (non-portable size).
constexpr int kMaxClusterSplits = 16;
// Tokens per TMA box / MMA tile: chunk lengths are multiples of it.
constexpr int kPlanTile = 16;
// Rows per kv head above which the tcgen05 kernel runs.
constexpr int kPlanMaxNarrowRows = 16;

struct PlanShape {
  int64_t slots;     // CTAs of the split launch resident at once
  int batch;         // requests (>= 0)
  int num_kv_heads;  // Hkv
  int rows;          // query rows per kv head: (Hq / Hkv) * q_len
  int max_seq_len;   // upper bound of every length (>= 0)
};

// a / b for a >= 0, b > 0, in 32 bits when both fit: on the GPU a 64-bit
// division is a long dependent sequence, and the device planner's path is a
// chain of them
__host__ __device__ inline int64_t plan_div(int64_t a, int64_t b) {
  if (((a | b) >> 32) == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

__host__ __device__ inline int64_t plan_ceil_div(int64_t a, int64_t b) { return plan_div(a + b - 1, b); }

// a * b, saturated at 2^62 (both >= 0)
__host__ __device__ inline int64_t plan_sat_mul(int64_t a, int64_t b) {
  const int64_t lim = int64_t{1} << 62;
  if (a == 0 || b == 0) return 0;
  if (((a | b) >> 31) == 0) return a * b;  // (both below 2^31)
  return a > lim / b ? lim : a * b;
}

// Chunk length for a split count: the smallest multiple of 16 that covers
// max_seq_len in `splits` chunks; *eff = the chunks that then exist.  False
// when splits < 1 or the chunk would exceed 2^30 tokens.
__host__ __device__ inline bool plan_chunk_for_splits(int max_seq_len, int64_t splits,
                                                      int32_t* chunk, int32_t* eff) {
  if (splits < 1) return false;
  const int64_t L = max_seq_len;
  int64_t c = plan_ceil_div(L > 1 ? L : 1, splits);
  c = plan_ceil_div(c, kPlanTile) * kPlanTile;
  if (c > (int64_t{1} << 30)) return false;
  *chunk = static_cast<int32_t>(c);
  const int64_t e = plan_ceil_div(L, c);
  *eff = static_cast<int32_t>(e > 1 ? e : 1);
  return true;
}

// The largest c in (lo, hi] with chunks_of(c) >= need, or lo when there is
// none (lo <= hi; lo itself is never tested).  chunks_of is non-increasing in
// c, so the lengths that pass are those up to one boundary and every search
// for it gives the same c.  This one tests hi first (the usual answer), then
// bisects.
template <class ChunksOf>
__host__ __device__ int64_t plan_search_bisect(int64_t lo, int64_t hi, int64_t need,
                                               ChunksOf&& chunks_of) {
  if (hi <= lo || chunks_of(hi) >= need) return hi;
  while (hi - lo > 1) {  // (chunks_of(hi) < need from here on)
    const int64_t mid = (lo + hi) / 2;
    if (chunks_of(mid) >= need) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Chunks per (request, kv head) for the batch (before plan_chunk_for_splits).
//   uniform      all lengths equal, or none known (then max_seq_len is taken)
//   work_tokens  sum of the clamped lengths (ragged batches only)
//   chunks_of(c) sum over requests of max(1, ceil(L_b / c)), times Hkv
// Equal lengths: one full wave of equal chunks -- as many per (request, kv
// head) as there are resident slots for them, at most kMaxClusterSplits so the
// chunks of a head can merge as a cluster.  Ragged lengths: about
// kRaggedWaves waves of chunks over the actual work (long requests are cut
// into pieces that keep the tail short), at least max(256, kTokensPerRow x
// rows) tokens each (kWideTokensPerRow above 16 rows); a small batch keeps at
// least one chunk per slot: while that floor leaves fewer chunks than slots,
// the chunk shrinks to the largest length that fills them (not below 256).
// search(lo, hi, need) finds that length as plan_search_bisect defines it
// (the device planner tests several lengths at once; the answer is the same).
template <class ChunksOf, class Search>
__host__ __device__ int64_t plan_splits(const PlanShape& s, bool uniform, int64_t work_tokens,
                                        ChunksOf&& chunks_of, Search&& search) {
  const int64_t msl = s.max_seq_len;
  const int64_t max_tiles = plan_ceil_div(msl > 1 ? msl : 1, kPlanTile);
  const int64_t pairs = static_cast<int64_t>(s.batch > 1 ? s.batch : 1) * s.num_kv_heads;
  int64_t splits = 1;
  if (uniform) {
    if (pairs < s.slots) {
      const int64_t f = plan_div(s.slots, pairs);
      splits = f < kMaxClusterSplits ? f : kMaxClusterSplits;
    }
  } else {
    const int64_t per_cta =
        plan_ceil_div(plan_sat_mul(work_tokens, s.num_kv_heads), plan_sat_mul(kRaggedWaves, s.slots));
    const int64_t per_row = s.rows > kPlanMaxNarrowRows ? kWideTokensPerRow : kTokensPerRow;
    const int64_t floor_rows = per_row * s.rows;
    const int64_t min_chunk = floor_rows > kMinChunkTokens ? floor_rows : kMinChunkTokens;
    const int64_t target = search(int64_t{kMinChunkTokens},
                                  per_cta > min_chunk ? per_cta : min_chunk, s.slots);
    splits = plan_ceil_div(msl > 1 ? msl : 1, target);
  }
  const int64_t by_min = msl / kMinChunkTokens > 1 ? msl / kMinChunkTokens : 1;
  if (splits > by_min) splits = by_min;
  if (splits > max_tiles) splits = max_tiles;
  return splits > 1 ? splits : 1;
}

template <class ChunksOf>
__host__ __device__ int64_t plan_splits(const PlanShape& s, bool uniform, int64_t work_tokens,
                                        ChunksOf&& chunks_of) {
  return plan_splits(s, uniform, work_tokens, chunks_of, [&](int64_t lo, int64_t hi, int64_t need) {
    return plan_search_bisect(lo, hi, need, chunks_of);
  });
}

}  // namespace dattn
