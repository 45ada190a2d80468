// combine_kernel.cu -- the cross-chunk reduce of split-KV decode attention.
//
// For each output row (request b, token t, query head h) whose request spans
// n >= 2 chunks, merge the normalised fp32 partials O_s and their natural-log
// LSEs lse_s exactly ("Capstone FlashAttention", §1.2 merge of running max and
// running sum, applied to all chunks at once; §2.3 FlashDecoding's small
// cross-SM reduce kernel):
//     M = max_s lse_s,  w_s = exp(lse_s - M),
//     out = sum_s w_s O_s / sum_s w_s,   lse = M + ln(sum_s w_s).
// One warp per row: lane i owns d = 4i..4i+3, so each partial row is one
// coalesced 512-byte read.  Empty chunks (lse -inf) weigh nothing; a row with
// no finite lse gives out = 0, lse = -inf.

#include "decode_attn.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace dattn {
namespace {

// The merge of one row of a device-planned call, by one warp (lane i owns d =
// 4i..4i+3): partial s of the row has its LSE at pl[s * ls] and its output
// slice at po[s * os] (po already offset by 4 * lane).  The grid-planned path
// below follows the same order of operations, so both give the same bits.  Returns the merged, normalised slice of this
// lane and (every lane) the merged LSE; a row with no finite LSE gives 0 and
// -inf.  Loads go through L2 only (other CTAs of the same kernel may have
// written the partials) with `policy` (each partial is read once).
__device__ __forceinline__ void merge_row_warp(const float* pl, int ls, const float* po, int os,
                                               int n, uint64_t policy, float4* res, float* lse) {
  constexpr uint32_t kFull = 0xffffffffu;
  constexpr int kBatch = 4;
  constexpr float kLog2eM = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  // one round trip for the first 32 LSEs and the first kBatch partial rows
  const float lse0 =
      lane < n ? ld_global_cg_hint1(pl + static_cast<int64_t>(lane) * ls, policy) : -INFINITY;
  float4 v[kBatch];
#pragma unroll
  for (int j = 0; j < kBatch; ++j)
    v[j] = j < n ? ld_global_cg_hint(po + static_cast<int64_t>(j) * os, policy)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = lse0;
  for (int s = lane + 32; s < n; s += 32)
    M = fmaxf(M, ld_global_cg_hint1(pl + static_cast<int64_t>(s) * ls, policy));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 16));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 8));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 4));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 2));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 1));
  if (M == -INFINITY) {
    *res = make_float4(0.f, 0.f, 0.f, 0.f);
    *lse = -INFINITY;
    return;
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  for (int s0 = 0; s0 < n; s0 += 32) {
    const int cnt = min(32, n - s0);
    const float lse_mine =
        s0 == 0 ? lse0
                : (lane < cnt ? ld_global_cg_hint1(pl + static_cast<int64_t>(s0 + lane) * ls, policy)
                              : -INFINITY);
    const float w_mine = lane < cnt ? ex2((lse_mine - M) * kLog2eM) : 0.f;
    for (int j0 = 0; j0 < cnt; j0 += kBatch) {
      if (s0 + j0 > 0) {  // batch 0 of group 0 is already in flight
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          v[j] = j0 + j < cnt ? ld_global_cg_hint(po + static_cast<int64_t>(s0 + j0 + j) * os, policy)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (j0 + j < cnt) {  // (not a multiply by zero: stale values may be NaN)
          const float w = __shfl_sync(kFull, w_mine, (j0 + j) & 31);
          W += w;
          acc.x += w * v[j].x;
          acc.y += w * v[j].y;
          acc.z += w * v[j].z;
          acc.w += w * v[j].w;
        }
      }
    }
  }
  const float inv = 1.f / W;
  *res = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  *lse = M + logf(W);
}


constexpr int kWarpsPerBlock = 8;
constexpr int kBlocksPerSm = 6;  // registers capped so that 48 warps fit per SM
constexpr float kLog2e = 1.4426950408889634f;

// LISTED: a device-planned call (partials indexed by item, chunk length from
// the planner's output); otherwise partials are [row][split].
// (the device-planned form holds more addressing state: 5 blocks per SM, no
// spills, instead of 6)
template <bool LISTED>
__global__ void __launch_bounds__(32 * kWarpsPerBlock, LISTED ? kBlocksPerSm - 1 : kBlocksPerSm)
    combine_kernel(const CombineArgs a) {
  constexpr uint32_t kFull = 0xffffffffu;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.num_q_heads;
  const bool live = row < nrows;
  const int h = live ? static_cast<int>(row % a.num_q_heads) : 0;
  const int t = live ? static_cast<int>((row / a.num_q_heads) % a.q_len) : 0;
  const int b = live ? static_cast<int>(row / (static_cast<int64_t>(a.num_q_heads) * a.q_len)) : 0;
  // the split kernel that wrote the partials may still be running (this
  // kernel may launch during its tail): wait before reading anything
  grid_dependency_wait();
  if (!live) return;

  // Partial s of this row is at pl[s * ls] / po[s * os].  Grid-planned call:
  // [row][split] (ls = 1, os = D).  Device-planned call: by item, item(b,
  // kvh, s) = pre[b] * Hkv + kvh * n + s, row r of the item's rows (ls =
  // rows, os = rows * D); its base needs the request's prefix and the
  // chunk length first (one more round trip).
  constexpr int kBatch = 4;
  const uint64_t dead = l2_evict_first_policy();  // each partial is read once
  // (set by the grid-planned path; the listed one returns before their use)
  const float* pl = nullptr;
  const float* po = nullptr;
  int ls = 0, os = 0;  // per-split strides (<= 128 rows x 128 d)
  int S = 0, L = 0, n = 0;
  if constexpr (LISTED) {
    L = a.seq_lens[b];
    const int pb = a.pre[b];
    const int chunk = a.plan[0];
    L = L < 0 ? 0 : (L > a.max_seq_len ? a.max_seq_len : L);
    n = L > 0 ? (L + chunk - 1) / chunk : 1;
    if (n < 2) return;  // the split kernel wrote this row directly
    const int G = a.num_q_heads / a.num_kv_heads;
    const int rows = G * a.q_len;
    const int kvh = h / G;
    const int64_t base = static_cast<int64_t>(pb) * a.num_kv_heads + static_cast<int64_t>(kvh) * n;
    const int64_t r0 = base * rows + t * G + (h - kvh * G);
    // the merge the split kernel runs in-kernel for these calls (same routine,
    // same bits): here for calls that keep the partials (DA_FLAG_TWO_PASS)
    float4 res;
    float lse_row;
    merge_row_warp(a.part_lse + r0, rows, a.part_o + r0 * kHeadDim + lane * 4, rows * kHeadDim, n,
                   dead, &res, &lse_row);
    uint16_t* orow = a.out + static_cast<int64_t>(b) * a.o_sb + static_cast<int64_t>(t) * a.o_st +
                     static_cast<int64_t>(h) * a.o_sh + lane * 4;
    *reinterpret_cast<uint2*>(orow) =
        make_uint2(pack_bf16x2(res.x, res.y), pack_bf16x2(res.z, res.w));
    if (lane == 0) a.lse[row] = lse_row;
    return;
  } else {
    S = a.num_splits;
    pl = a.part_lse + row * S;
    po = a.part_o + row * S * kHeadDim + lane * 4;
    ls = 1;
    os = kHeadDim;
    L = a.seq_lens[b];
    n = 0;  // known after the first round trip
  }
  // one round trip for the first 32 LSEs and the first kBatch partial rows
  // (grid-planned: with the request length): none of these loads depends on
  // another. Splits past the request's chunk count hold stale values,
  // dropped by the selects below.
  const float lse0 = lane < S ? ld_global_hint1(pl + static_cast<int64_t>(lane) * ls, dead) : -INFINITY;
  float4 v[kBatch];
#pragma unroll
  for (int j = 0; j < kBatch; ++j)
    v[j] = j < S ? ld_global_hint(po + static_cast<int64_t>(j) * os, dead) : make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (!LISTED) {
    L = L < 0 ? 0 : (L > a.max_seq_len ? a.max_seq_len : L);
    n = L > 0 ? (L + a.chunk_len - 1) / a.chunk_len : 1;
    if (n < 2) return;  // the split kernel wrote this row directly
  }

  uint16_t* orow = a.out + static_cast<int64_t>(b) * a.o_sb + static_cast<int64_t>(t) * a.o_st +
                   static_cast<int64_t>(h) * a.o_sh + lane * 4;
  // splits in groups of 32: lane j holds lse of split s0 + j
  float M = lane < n ? lse0 : -INFINITY;
  for (int s = lane + 32; s < n; s += 32) M = fmaxf(M, ld_global_hint1(pl + static_cast<int64_t>(s) * ls, dead));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 16));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 8));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 4));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 2));
  M = fmaxf(M, __shfl_xor_sync(kFull, M, 1));
  if (M == -INFINITY) {
    *reinterpret_cast<uint2*>(orow) = make_uint2(0u, 0u);
    if (lane == 0) a.lse[row] = -INFINITY;
    return;
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  for (int s0 = 0; s0 < n; s0 += 32) {
    const int cnt = min(32, n - s0);
    const float lse_mine =
        s0 == 0 ? lse0 : (lane < cnt ? ld_global_hint1(pl + static_cast<int64_t>(s0 + lane) * ls, dead) : -INFINITY);
    const float w_mine = lane < cnt ? ex2((lse_mine - M) * kLog2e) : 0.f;
    for (int j0 = 0; j0 < cnt; j0 += kBatch) {
      if (s0 + j0 > 0) {  // batch 0 of group 0 is already in flight
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
          v[j] = j0 + j < cnt ? ld_global_hint(po + static_cast<int64_t>(s0 + j0 + j) * os, dead)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (j0 + j < cnt) {  // (not a multiply by zero: stale values may be NaN)
          const float w = __shfl_sync(kFull, w_mine, (j0 + j) & 31);
          W += w;
          acc.x += w * v[j].x;
          acc.y += w * v[j].y;
          acc.z += w * v[j].z;
          acc.w += w * v[j].w;
        }
      }
    }
  }
  const float inv = 1.f / W;
  *reinterpret_cast<uint2*>(orow) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (lane == 0) a.lse[row] = M + logf(W);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int64_t nrows = static_cast<int64_t>(a.batch) * a.q_len * a.num_q_heads;
  if (nrows == 0) return cudaSuccess;
  const int64_t blocks = (nrows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(32 * kWarpsPerBlock);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.plan != nullptr ? cudaLaunchKernelEx(&cfg, combine_kernel<true>, a)
                           : cudaLaunchKernelEx(&cfg, combine_kernel<false>, a);
}

}  // namespace dattn
