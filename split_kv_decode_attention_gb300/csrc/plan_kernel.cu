// plan_kernel.cu -- the split planner on the device, for decode_attn calls
// whose lengths live only in device memory (a serving loop's seq_lens, a
// captured CUDA graph replayed with new lengths).
//
// Every CTA reads seq_lens and applies the planner's rule (plan_rule.cuh: the
// same code the host planner runs with host lengths); CTA 0 writes, into the
// caller's workspace:
//   plan[0] chunk_len, plan[1] n_items, plan[2] chunks of the longest request,
//   plan[3] the item capacity the launch was sized for;
//   pre[b]  exclusive prefix over requests of their chunk counts (pre[B] =
//           n_items / Hkv);
//   items[i] = (b, kv head, chunk, clamped length) for every work item, in
//           (request, kv head, chunk) order: item(b, kvh, s) =
//           pre[b] * Hkv + kvh * n_b + s, with n_b = max(1, ceil(L_b / chunk)).
// The item list is shared out: each CTA writes the items of its own
// (request, kv head) pairs.  (The CTAs all reach the same plan, so running
// it in each costs no time; a single CTA's stores of a few thousand 16-byte
// items took ~3 us on GB300.)
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

constexpr int kPlanThreadsLog2 = 8;
constexpr int kPlanThreads = 1 << kPlanThreadsLog2;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kPlanLenCache = 4096;  // clamped lengths (and the prefix) kept in shared memory
// Up to this many requests every warp evaluates a chunk count by itself
// (lanes over the requests, one warp-wide sum, no block barrier): a
// block-wide sum costs a barrier and shared-memory round trips each time.
constexpr int kPlanWarpSumBatch = 256;
// In the split search a candidate length is tested by the fewest threads
// (a power of two, up to a warp) that take at most this many requests each.
constexpr int kPlanSearchLens = 8;
static_assert(kPlanSearchLens * 32 >= kPlanWarpSumBatch, "a warp per candidate covers the batch");
// Rounds of the split search never exceed ~11 (at least 8 candidates per
// round over at most 2^31 lengths); the cap only bounds the loop.
constexpr int kPlanMaxRounds = 64;
// The item list: threads per (request, kv head) pair (its chunks are written
// strided over them), hence pairs per CTA, and the most CTAs launched.
constexpr int kPlanItemLanes = 4;
constexpr int kPlanPairsPerCta = kPlanThreads / kPlanItemLanes;
constexpr int kPlanMaxCtas = 32;

struct PlanSmem {
  long long red[2][kPlanWarps];  // block sums, two buffers used alternately
  long long scan[kPlanWarps];    // warp totals of the prefix
  int lens[kPlanLenCache];
  int pre[kPlanLenCache + 1];    // the prefix, read back while writing the item list
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

// Division by a length c shared by many dividends, by a multiply-high
// (Granlund and Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994): with m = floor((2^32 - 1) / c) + 1, which is
// ceil(2^32 / c) for 2 <= c < 2^31, q = floor(x * m / 2^32) is floor(x / c)
// or one more for every x < 2^32 (x * m / 2^32 exceeds x / c by less than
// x / 2^32 < 1), and q * c > x exactly when it is one more.  The planner's
// chain of candidate tests runs on this instead of a division per request.
__device__ __forceinline__ unsigned len_magic(unsigned c) { return 0xFFFFFFFFu / c + 1u; }

// Chunks of a request of clamped length L at chunk length c (magic mg =
// len_magic(c)): ceil(L / c) = floor((L - 1) / c) + 1, one for an empty
// request (0 <= L <= 2^30, 16 <= c <= 2^30, so q * c <= x + c < 2^32).
__device__ __forceinline__ unsigned chunks_of_len(int L, unsigned c, unsigned mg) {
  if (L <= 0) return 1u;
  const unsigned x = static_cast<unsigned>(L) - 1u;
  unsigned q = __umulhi(x, mg);
  q -= q * c > x ? 1u : 0u;
  return q + 1u;
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
  const bool lead = blockIdx.x == 0;  // (the CTA that writes plan, pre and status)
  if (lead && tid == 0 && bits != 0 && a.status != nullptr)
    atomicOr(a.status, static_cast<int32_t>(bits));

  // work items at chunk length c (all threads call it and get the same sum:
  // per warp up to kPlanWarpSumBatch requests, else a block-wide sum).
  // (Every length is <= max_seq_len <= 2^30 here, so a longer chunk counts
  // one per request, the same as 2^30; a warp's 32-bit sum stays below
  // 256 requests x 2^22 chunks of >= 256 tokens.)
  const int lane = tid & 31, warp = tid >> 5;
  auto clamp_chunk = [](long long c) { return c < (1LL << 30) ? c : (1LL << 30); };
  auto chunks_of = [&](long long c) -> long long {
    const unsigned cc = static_cast<unsigned>(clamp_chunk(c));
    const unsigned mg = len_magic(cc);
    if (B <= kPlanWarpSumBatch) {
      unsigned n32 = 0;
#pragma unroll
      for (int i = 0; i < kPlanWarpSumBatch / 32; ++i) {
        const int b = lane + 32 * i;
        if (b < B) n32 += chunks_of_len(sm.lens[b], cc, mg);
      }
      return static_cast<long long>(__reduce_add_sync(0xffffffffu, n32)) * a.num_kv_heads;
    }
    long long n = 0;
    for (int b = tid; b < B; b += kPlanThreads) n += chunks_of_len(len_of(b), cc, mg);
    return block_sum(n, sm, parity) * a.num_kv_heads;
  };

  PlanShape shape;
  shape.slots = a.slots;
  shape.batch = B;
  shape.num_kv_heads = a.num_kv_heads;
  shape.rows = a.rows;
  shape.max_seq_len = msl;
  // The split search of the rule: the largest length in (lo, hi] whose
  // chunks reach `need`.  Up to kPlanWarpSumBatch requests each group of g
  // threads (at most kPlanSearchLens requests a thread) tests its own
  // candidate, G = 256 / g lengths spread over (lo, hi] with hi the last.
  // The counts fall as the length grows, so the candidates that pass are a
  // prefix and one block-wide count finds the boundary: a round cuts the
  // interval ~G-fold where the bisection halves it, the answer is the
  // bisection's, and a round whose candidates all pass (hi fills the slots:
  // most batches) ends the search.  (GB300: 16 requests, the bisection's 14
  // one-length tests took 7 us; this, 2 rounds.)
  auto search = [&](long long lo, long long hi, long long need) -> long long {
    if (B > kPlanWarpSumBatch) return plan_search_bisect(lo, hi, need, chunks_of);
    int lg = 0;  // log2 g
    while (lg < 5 && (kPlanSearchLens << lg) < B) ++lg;
    const int lgG = kPlanThreadsLog2 - lg;
    const int G = 1 << lgG, g = 1 << lg, sub = tid & (g - 1);
    const long long H = a.num_kv_heads;
    for (int round = 0; hi > lo && round < kPlanMaxRounds; ++round) {
      // candidate j: lo <= cand(j) <= hi, non-decreasing in j, cand(G - 1) = hi
      auto cand = [&](int j) { return lo + (((hi - lo) * (j + 1)) >> lgG); };
      const long long m = cand(tid >> lg);
      const unsigned c = static_cast<unsigned>(clamp_chunk(m));
      const unsigned mg = len_magic(c);
      unsigned n = 0;
#pragma unroll
      for (int i = 0; i < kPlanSearchLens; ++i) {
        const int b = sub + (i << lg);
        if (b < B) n += chunks_of_len(sm.lens[b], c, mg);
      }
      for (int o = g >> 1; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
      // (a candidate at lo counts as passing: lo is the answer unless a
      // longer length passes)
      const bool pass = static_cast<long long>(n) * H >= need || m <= lo;
      const int k = __syncthreads_count(sub == 0 && pass);
      if (k == G) return hi;
      const long long nlo = k > 0 ? cand(k - 1) : lo;
      hi = cand(k) - 1;  // (cand(k) fails, so it is > lo and > cand(k - 1))
      lo = nlo;
    }
    return lo;
  };
  const long long splits = plan_splits(shape, uniform, work, chunks_of, search);
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
  long long run = 0;
  for (int b0 = 0; b0 < B; b0 += kPlanThreads) {
    const int b = b0 + tid;
    const int L = b < B ? len_of(b) : 0;
    const long long n = b < B ? chunks_of_len(L, static_cast<unsigned>(chunk), len_magic(chunk)) : 0;
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
    if (b < B) {
      const int32_t pb = static_cast<int32_t>(run + before + x - n);
      if (lead) a.pre[b] = pb;
      if (b <= kPlanLenCache) sm.pre[b] = pb;  // (kPlanLenCache + 1 entries)
    }
    run += tot;
    __syncthreads();  // sm.scan is rewritten by the next round
  }
  if (tid == 0) {
    if (lead) a.pre[B] = static_cast<int32_t>(run);
    if (B <= kPlanLenCache) sm.pre[B] = static_cast<int32_t>(run);
  }
  __syncthreads();  // pre[] visible to the whole block

  // ---- the item list: kPlanItemLanes threads per (request, kv head) pair
  // write its chunks, CTA c taking the pairs [c * 64, c * 64 + 64) of every
  // grid-sized block of them.  (One warp per request, walking its requests
  // one after another, took 8.3 us for 256 requests; one CTA with a pair per
  // thread ~3 us.)  A launch of more than one CTA has B <= kPlanLenCache, so
  // every CTA reads its own prefix copy.
  const int H = a.num_kv_heads;
  const int n_pairs = B * H;  // (<= the item capacity < 2^31)
  const int sub = tid & (kPlanItemLanes - 1);
  for (int64_t pr = static_cast<int64_t>(blockIdx.x) * kPlanPairsPerCta + tid / kPlanItemLanes;
       pr < n_pairs; pr += static_cast<int64_t>(gridDim.x) * kPlanPairsPerCta) {
    const int b = static_cast<int>(pr) / H;
    const int kvh = static_cast<int>(pr) - b * H;
    const int base = b < kPlanLenCache ? sm.pre[b] : a.pre[b];
    const int n = (b + 1 <= kPlanLenCache ? sm.pre[b + 1] : a.pre[b + 1]) - base;
    const int L = len_of(b);
    int4* dst = a.items + (static_cast<int64_t>(base) * H + static_cast<int64_t>(kvh) * n);
    for (int c = sub; c < n; c += kPlanItemLanes) dst[c] = make_int4(b, kvh, c, L);
  }
  if (lead && tid == 0) {
    a.plan[0] = chunk;
    a.plan[1] = static_cast<int32_t>(n_items);
    a.plan[2] = eff;
    a.plan[3] = static_cast<int32_t>(a.cap);
  }
}

}  // namespace

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  // a CTA per kPlanPairsPerCta pairs, one CTA when the lengths do not fit in
  // shared memory (the other CTAs would need the prefix CTA 0 writes)
  const int64_t pairs = static_cast<int64_t>(a.batch) * a.num_kv_heads;
  int64_t ctas = plan_ceil_div(pairs > 1 ? pairs : 1, kPlanPairsPerCta);
  if (ctas > kPlanMaxCtas) ctas = kPlanMaxCtas;
  if (a.batch > kPlanLenCache) ctas = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
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
