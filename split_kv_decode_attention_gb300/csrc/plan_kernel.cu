// plan_kernel.cu -- the split planner on the device, for decode_attn calls
// whose lengths live only in device memory (a serving loop's seq_lens, a
// captured CUDA graph replayed with new lengths).
//
// One CTA reads seq_lens, applies the planner's rule (plan_rule.cuh: the same
// code the host planner runs with host lengths) and writes, into the caller's
// workspace:
//   plan[0] chunk_len, plan[1] n_items, plan[2] chunks of the longest request,
//   plan[3] the item capacity the launch was sized for;
//   pre[b]  exclusive prefix over requests of their chunk counts (pre[B] =
//           n_items / Hkv);
//   items[i] = (b, kv head, chunk, clamped length) for every work item, in
//           (request, kv head, chunk) order: item(b, kvh, s) =
//           pre[b] * Hkv + kvh * n_b + s, with n_b = max(1, ceil(L_b / chunk)).
// The split kernel then runs one CTA per item slot of a host-sized grid (the
// capacity), and partials are indexed by item, so neither the grid nor the
// workspace depends on the lengths.  If the rule's chunk would make more
// items than the capacity, the chunk grows (in multiples of 16) until they
// fit; at chunk >= max_seq_len every request is one item, so a capacity of at
// least B * Hkv always fits.  Data errors (a length outside [0, max_seq_len],
// a causal request shorter than q_len) are reported here, once per call.

#include "decode_attn.h"
#include "kernels.cuh"
#include "plan_rule.cuh"
#include "ptx.cuh"

namespace dattn {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kPlanLenCache = 4096;  // clamped lengths kept in shared memory

struct PlanSmem {
  long long red[2][kPlanWarps];  // block sums, two buffers used alternately
  long long scan[kPlanWarps];    // warp totals of the prefix
  int lens[kPlanLenCache];
};

// Sum of v over the block (every thread gets it).  All threads call it; the
// two buffers alternate, so one barrier per call suffices (a buffer is written
// again only after every thread passed the barrier of the call in between).
__device__ long long block_sum(long long v, PlanSmem& sm, int& parity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sm.red[parity][warp] = v;
  __syncthreads();
  long long t = 0;
#pragma unroll
  for (int w = 0; w < kPlanWarps; ++w) t += sm.red[parity][w];
  parity ^= 1;
  return t;
}

// ceil(L / c) for 0 < L < 2^31, 0 < c <= 2^30 (32-bit unsigned arithmetic)
__device__ __forceinline__ int ceil_div_u(int L, long long c) {
  const unsigned cu = static_cast<unsigned>(c);
  return static_cast<int>((static_cast<unsigned>(L) + cu - 1u) / cu);
}

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(const PlanArgs a) {
  __shared__ PlanSmem sm;
  int parity = 0;
  // launched early behind the previous kernel, which may write seq_lens
  grid_dependency_wait();
  // the split kernel may start launching: it waits for this grid's writes
  if (threadIdx.x == 0) allow_dependent_launch();
  const int tid = threadIdx.x;
  const int B = a.batch;
  const int msl = a.max_seq_len;
  auto clamp_len = [&](int raw) { return raw < 0 ? 0 : (raw > msl ? msl : raw); };
  auto len_of = [&](int b) { return b < kPlanLenCache ? sm.lens[b] : clamp_len(a.seq_lens[b]); };

  // ---- lengths: clamp, report, sum, and whether they are all equal
  const int raw0 = a.seq_lens[0];
  long long work = 0;
  bool diff = false;
  uint32_t bad = 0;
  for (int b = tid; b < B; b += kPlanThreads) {
    const int raw = a.seq_lens[b];
    const int L = clamp_len(raw);
    if (raw != L) bad |= DA_STATUS_SEQ_LEN;
    if (a.causal && L > 0 && L < a.q_len) bad |= DA_STATUS_SHORT_CAUSAL;
    diff = diff || raw != raw0;
    if (b < kPlanLenCache) sm.lens[b] = L;
    work += L;
  }
  work = block_sum(work, sm, parity);  // (its barrier also publishes sm.lens)
  const bool uniform = __syncthreads_or(diff) == 0;
  uint32_t bits = 0;
  if (__syncthreads_or((bad & DA_STATUS_SEQ_LEN) != 0)) bits |= DA_STATUS_SEQ_LEN;
  if (__syncthreads_or((bad & DA_STATUS_SHORT_CAUSAL) != 0)) bits |= DA_STATUS_SHORT_CAUSAL;
  if (tid == 0 && bits != 0 && a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(bits));

  // work items at chunk length c (a block-wide sum; all threads call it)
  auto chunks_of = [&](long long c) -> long long {
    // (every length is <= max_seq_len <= 2^30 here, so a longer chunk
    // counts one per request, the same as 2^30)
    const long long cc = c < (1LL << 30) ? c : (1LL << 30);
    long long n = 0;
    for (int b = tid; b < B; b += kPlanThreads) {
      const int L = len_of(b);
      n += L > 0 ? ceil_div_u(L, cc) : 1;
    }
    return block_sum(n, sm, parity) * a.num_kv_heads;
  };

  PlanShape shape;
  shape.slots = a.slots;
  shape.batch = B;
  shape.num_kv_heads = a.num_kv_heads;
  shape.rows = a.rows;
  shape.max_seq_len = msl;
  const long long splits = plan_splits(shape, uniform, work, chunks_of);
  int32_t chunk = 0, eff = 0;
  // (the host runs this path only when max_seq_len <= 2^30, so every split
  // count gives a valid chunk)
  plan_chunk_for_splits(msl, splits, &chunk, &eff);
  long long n_items = chunks_of(chunk);
  if (n_items > a.cap) {
    // more items than grid slots: the smallest longer chunk (multiple of 16)
    // that fits; hi = the whole sequence in one chunk always does
    long long lo = chunk, hi = plan_ceil_div(msl > 1 ? msl : 1, kPlanTile) * kPlanTile;
    while (hi - lo > kPlanTile) {
      const long long mid = (lo + hi) / 2 / kPlanTile * kPlanTile;
      if (chunks_of(mid) <= a.cap) hi = mid;
      else lo = mid;
    }
    chunk = static_cast<int32_t>(hi);
    eff = static_cast<int32_t>(plan_ceil_div(msl, hi) > 1 ? plan_ceil_div(msl, hi) : 1);
    n_items = chunks_of(chunk);
  }

  // ---- exclusive prefix of chunks per request
  const int lane = tid & 31, warp = tid >> 5;
  long long run = 0;
  for (int b0 = 0; b0 < B; b0 += kPlanThreads) {
    const int b = b0 + tid;
    const int L = b < B ? len_of(b) : 0;
    const long long n = b < B ? (L > 0 ? ceil_div_u(L, chunk) : 1) : 0;
    long long x = n;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) sm.scan[warp] = x;
    __syncthreads();
    long long before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kPlanWarps; ++w) {
      before += w < warp ? sm.scan[w] : 0;
      tot += sm.scan[w];
    }
    if (b < B) a.pre[b] = static_cast<int32_t>(run + before + x - n);
    run += tot;
    __syncthreads();  // sm.scan is rewritten by the next round
  }
  if (tid == 0) a.pre[B] = static_cast<int32_t>(run);
  __syncthreads();  // pre[] visible to the whole block

  // ---- the item list: one warp per request, lanes over (kv head, chunk)
  for (int b = warp; b < B; b += kPlanWarps) {
    const int base = a.pre[b];
    const int n = a.pre[b + 1] - base;
    const int L = len_of(b);
    const int64_t first = static_cast<int64_t>(base) * a.num_kv_heads;
    for (int i = lane; i < n * a.num_kv_heads; i += 32) {
      const int kvh = i / n;
      a.items[first + i] = make_int4(b, kvh, i - kvh * n, L);
    }
  }
  if (tid == 0) {
    a.plan[0] = chunk;
    a.plan[1] = static_cast<int32_t>(n_items);
    a.plan[2] = eff;
    a.plan[3] = static_cast<int32_t>(a.cap);
  }
}

}  // namespace

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, a);
}

}  // namespace dattn
