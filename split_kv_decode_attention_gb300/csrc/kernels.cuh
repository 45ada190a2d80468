// kernels.cuh -- internal interface between the C ABI (api.cu) and the
// decode-attention kernels.  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "decode_attn.h"

namespace dattn {

constexpr int kHeadDim = 128;
constexpr int kTileTokens = 16;        // tokens per TMA box / per MMA tile
constexpr int kMaxRows = 128;          // GQA group x q_len rows per CTA
constexpr int kMaxNarrowRows = 16;     // above this: the tcgen05 kernel
constexpr int kWideMaxPlannedBatch = 1024;  // tcgen05 kernel: device-planned calls up to this batch

// Arguments of the split kernel (one CTA per (chunk, kv head, request)).
struct SplitArgs {
  const uint16_t* q;                   // bf16 [B, q_len, Hq, D]
  int64_t q_sb, q_st, q_sh;
  uint16_t* out;                       // bf16 [B, q_len, Hq, D]
  int64_t o_sb, o_st, o_sh;
  float* lse;                          // fp32 [B, q_len, Hq]
  float* part_o;                       // fp32 [B, q_len, Hq, S, D] (S > 1)
  float* part_lse;                     // fp32 [B, q_len, Hq, S]
  const int32_t* block_table;          // paged only
  int64_t bt_stride;
  const int32_t* seq_lens;
  int32_t* status;                     // optional
  int batch, q_len, num_q_heads, num_kv_heads, group, rows;
  int page_size, num_pages, paged;
  int max_seq_len, chunk_len, num_splits;
  int causal;
  float scale_log2;                    // softmax scale * log2(e)
  int persistent;                      // wide kernel: CTAs walk an item list (set by its launcher)
  int kv_fp8;                          // caches hold FP8 E4M3
  float v_scale;                       // FP8: values = v_scale * V (k_scale is in scale_log2)
  int test_withhold;                   // DA_FLAG_TEST_WITHHOLD_COPY (narrow kernel, two-pass)
  int big_box;                         // contiguous caches: the maps' boxes span a whole stage
  // Device-planned calls (items != nullptr): the planner kernel wrote the
  // chunk length and item count to plan[0..1], per-request prefixes of chunk
  // counts to pre[], and the work items (b, kv head, chunk, clamped length) to
  // items[]; the split grid is `item_slots` CTAs (one per possible item) and
  // partial (item i, row r) sits at part_o[(i * rows + r) * D] / part_lse[i *
  // rows + r].  chunk_len / num_splits above are unused then.
  const int4* items;
  const int32_t* plan;
  const int32_t* pre;
  int item_slots;
};

// Arguments of the device planner kernel (plan_kernel.cu; up to 32 CTAs, each
// running the whole plan and writing its share of the item list).
struct PlanArgs {
  const int32_t* seq_lens;
  int32_t* status;                     // optional
  int32_t* plan;                       // [4]: chunk_len, n_items, max chunks, capacity
  int32_t* pre;                        // [B + 1]
  int4* items;                         // [cap]
  int64_t slots;                       // resident CTAs of the split launch
  int64_t cap;                         // item slots of the split launch
  int batch, num_kv_heads, rows, max_seq_len, q_len, causal;
};

struct CombineArgs {
  const float* part_o;
  const float* part_lse;
  const int32_t* seq_lens;
  uint16_t* out;
  int64_t o_sb, o_st, o_sh;
  float* lse;
  int batch, q_len, num_q_heads;
  int max_seq_len, chunk_len, num_splits;
  // device-planned calls (plan != nullptr): chunk length from plan[0],
  // partials indexed by item (see SplitArgs)
  const int32_t* plan;
  const int32_t* pre;
  int num_kv_heads;
};

// Physical page ids of a chunk's 16-token tiles, for the TMA producer warp.
// Lane i holds the id of tile base + i of the current 32-tile window and of
// the next window, loaded a full window (32 tiles) before it is needed, so
// the block-table latency never sits in front of a TMA issue.  Out-of-range
// entries read as page 0 and set DA_STATUS_BAD_PAGE.  All lanes of the warp
// must call get() together with the same tile.
struct PageWindow {
  const int32_t* bt_row;  // this request's block-table row (nullptr: contiguous)
  int t_begin, n_tiles, page_size, num_pages, lane;
  int32_t* status;
  int cur, nxt, base;

  __device__ __forceinline__ int load(int tile) const {
    if (bt_row == nullptr || tile >= n_tiles) return 0;
    int pg = __ldg(bt_row + (t_begin + tile * 16) / page_size);
    if (pg < 0 || pg >= num_pages) {
      if (status != nullptr) atomicOr(status, static_cast<int32_t>(DA_STATUS_BAD_PAGE));
      pg = 0;
    }
    return pg;
  }
  __device__ __forceinline__ void init() {
    base = 0;
    cur = load(lane);
    nxt = load(32 + lane);
  }
  __device__ __forceinline__ int get(int tile) {
    while (tile >= base + 32) {
      cur = nxt;
      base += 32;
      nxt = load(base + 32 + lane);
    }
    return __shfl_sync(0xffffffffu, cur, tile - base);
  }
};

// Launch the split kernel over grid (num_splits, Hkv, B).  With
// cluster_merge the num_splits CTAs of each (kv head, request) run as one
// thread-block cluster and write the final output (no partials, no combine).
cudaError_t launch_split(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                         bool cluster_merge, cudaStream_t stream);

// True when clusters of num_splits CTAs (2..16) are supported and the device
// can hold num_clusters of them at once (one wave).
bool split_cluster_merge_fits(int rows, bool fp8, int num_splits, int64_t num_clusters);

// Token rows of the TMA boxes the split launch expects: a whole stage (16 x
// tiles per stage) for contiguous caches on the warp-MMA kernel, else 16.
// `ctas` is the launch's grid size (it picks the pipeline shape).
int split_box_tokens(int rows, bool fp8, bool paged, int64_t ctas);

// Resident split CTAs per SM for the kernel variant serving `rows` rows.
int split_ctas_per_sm(int rows, bool fp8);

// Launch the tcgen05 kernel for 17..128 rows per kv head (same grid, same
// outputs and partials as launch_split without cluster merge).
cudaError_t launch_wide(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                        cudaStream_t stream);
int wide_ctas_per_sm();

// Launch the combine kernel (one warp per output row).
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

// Launch the device planner ahead of a device-planned split launch.
cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);

}  // namespace dattn
