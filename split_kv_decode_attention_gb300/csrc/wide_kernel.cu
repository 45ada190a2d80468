// wide_kernel.cu -- split-KV decode attention for wide query groups (GQA group
// x speculative tokens = 17..128 query rows per KV head) on the 5th-generation
// tensor cores (tcgen05, operands and accumulators in tensor memory).
//
// With many query rows per KV head the per-chunk work is a dense attention
// tile ("Capstone FlashAttention", §2.3 speculative verify of several draft
// tokens at once, §4.5; the CUTLASS split-KV post, §6: 4-token speculation):
// arithmetic intensity reaches G*q_len FLOP per KV byte, far beyond what the
// legacy warp-level MMA sustains at HBM rate.  A work item is one (chunk, kv
// head, request) -- the unit of the narrow kernel's grid -- and the kernel is
// persistent: one CTA per SM walks a list of items ordered longest first
// (full chunks, then the last partial chunk of each request by decreasing
// length), taking positions in snake order (c, 2G-1-c, 2G+c, ...), so the
// last items to start are the shortest and the SMs finish together.  The
// list is rebuilt by every CTA from seq_lens in shared memory; batches too
// large for those tables fall back to one item per CTA (grid = chunks x kv
// heads x requests).  Per CTA:
//   * producer warps stream K/V with TMA through one ring of 64-token stages
//     (four 16-token page tiles, [2 d-halves][64 tokens][64 d], 128-byte
//     swizzle, mbarrier byte counts) without stopping between items, and
//     stage each item's query rows in shared memory with cp.async;
//   * one warp issues the MMAs (one elected lane, warp-uniform operands):
//     S = Q.K^T (M = 128 rows padded, N = 64 keys, K = 128 d; A = Q from
//     TMEM, B = K from shared memory) into one of two TMEM score buffers, and
//     O += P.V (N = 128 d, K = 64 keys; A = P from TMEM, B = V read MN-major
//     straight from the TMA tile) into a TMEM accumulator;
//   * warps 0-7 form two softmax groups that take alternate 64-key tiles,
//     one query row per thread (TMEM lane = row): they read the score row,
//     apply the masks, keep the running max / sum of the online softmax
//     ("Capstone FlashAttention", §1.2), write P in bf16 to TMEM, and rescale
//     their O rows only when the running max has grown by more than 2^8 since
//     the last rescale (P stays <= 256, exact in the deferred normalisation,
//     §2.1); at the end of an item the two groups merge and write the item's
//     output, then load the next item's Q into TMEM.
//     Up to 64 query rows the kernel splits the keys instead of padding the
//     rows: TMEM lane l holds row 16 (l / 32) + (l % 16) and takes keys
//     [0, 32) of every tile when l % 32 < 16, else [32, 64), each lane with
//     its own running max / sum and O row (its P row is zero over the other
//     half, so P.V sums only its keys; TMEM loads and stores take one column
//     address per warp, so every lane still moves the whole score and P row).  All 128 lanes then do useful work --
//     padded rows would leave half the softmax warps computing masked scores
//     -- and the two halves of a row sit in one warp, 16 lanes apart, where
//     the end of the item merges them by shuffles.
// Outputs are the final bf16 rows (single chunk) or fp32 partials + LSE for
// the combine kernel, exactly like split_kernel.cu.  Every wait is bounded;
// TMEM is always released before the CTA exits.

#include <mutex>

#include "decode_attn.h"
#include "kernels.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace dattn {
namespace {

constexpr float kLn2w = 0.6931471805599453f;
constexpr int kWRows = 128;                  // MMA M: query rows per CTA (padded)
constexpr int kWTok = 64;                    // keys per stage (MMA N of S)
constexpr int kWTiles = kWTok / kTileTokens; // 16-token page tiles per stage
// Pipeline shapes (build-time overridable for sweeps; the defaults are the
// GB300 sweep winners): TMA ring stages and producer warps for bf16 caches;
// for FP8 caches also the converter warps, whether the producers stage each
// item's Q rows in shared memory (else the softmax warps load them), and the
// K and V operand slots.
#ifndef DATTN_WIDE_STAGES
#define DATTN_WIDE_STAGES 5
#endif
#ifndef DATTN_WIDE_PRODUCERS
#define DATTN_WIDE_PRODUCERS 5
#endif
#ifndef DATTN_WIDE_F8_STAGES
#define DATTN_WIDE_F8_STAGES 4
#endif
#ifndef DATTN_WIDE_F8_QSTAGE
#define DATTN_WIDE_F8_QSTAGE 0
#endif
#ifndef DATTN_WIDE_F8_PRODUCERS
#define DATTN_WIDE_F8_PRODUCERS 3
#endif
#ifndef DATTN_WIDE_F8_CONVERTERS
#define DATTN_WIDE_F8_CONVERTERS 4
#endif
// FP8: widened K and V live in separate rings (a K slot is free once S =
// Q.K^T is done, a V slot only after P.V), 16 KB per slot
#ifndef DATTN_WIDE_F8_OPK
#define DATTN_WIDE_F8_OPK 2
#endif
#ifndef DATTN_WIDE_F8_OPV
#define DATTN_WIDE_F8_OPV 4
#endif
constexpr int kWHalf = kWTok * 128;          // [64 tokens][64 d] 16-bit = 8 KB
constexpr int kWStageBytes = 4 * kWHalf;     // operand stage: K halves, then V halves
constexpr int kWF8Tile = kTileTokens * 128;  // one FP8 tile (K or V): 16 rows of 128 bytes
// Requests whose schedule tables fit in shared memory (else one item per
// CTA), and up to which the partial chunks are sorted by length.
constexpr int kWMaxSchedBatch = kWideMaxPlannedBatch;
constexpr int kWSortBatch = 256;
// m, l (fp32 probabilities: the LSE) and lq (the same probabilities rounded
// to the 16-bit P operand: normalises O) per group and row; ok per softmax warp
constexpr int kWStatFloats = 6 * kWRows + 8;
constexpr int kWStatBytes = 3200;
constexpr int kWSchedInts = 4 * kWMaxSchedBatch + 4;
static_assert(kWStatFloats * 4 <= kWStatBytes, "statistics buffer");

// Warp roles and shared-memory layout of the two variants.
//   bf16 caches: warps 0-7 softmax, 8..12 TMA producers, 13 MMA; the TMA ring
//     holds the MMA operands directly (5 stages of 32 KB).
//   FP8 caches: warps 0-7 softmax, 8..10 TMA producers, 11..14 converters,
//     15 MMA; the TMA ring holds FP8 stages (4 x 16 KB: 8 boxes of 2 KB per 64
//     keys), the converters widen each stage's K into a ring of 2 f16 K slots
//     and its V into a ring of 4 f16 V slots (16 KB each; the B operands of
//     kind::f16 must be 16-bit).  A K slot is released as soon as its S =
//     Q.K^T completes, a V slot only after its P.V, so the two rings hold
//     each half only as long as it is needed.
// Shared memory: TMA ring, K and V operand rings (FP8 only), Q staging (bf16
// only: [128 rows][16 chunks of 16 B], chunk c of row r at c ^ (r & 15)), the
// groups' merge statistics (two buffers), schedule tables, barriers.
// TMA copies issued by one warp are serialised (~130-240 cycles per box), and
// the time to issue a stage counts against its ring slot, so all producer
// warps share each stage's boxes.
template <bool F8>
struct WCfg {
  static constexpr int kProducers = F8 ? DATTN_WIDE_F8_PRODUCERS : DATTN_WIDE_PRODUCERS;
  static constexpr int kConverters = F8 ? DATTN_WIDE_F8_CONVERTERS : 0;
  static constexpr int kProducerWarp = 8;
  static constexpr int kConverterWarp = kProducerWarp + kProducers;
  static constexpr int kMmaWarp = kConverterWarp + kConverters;
  static constexpr int kThreads = 32 * (kMmaWarp + 1);
  static constexpr int kStages = F8 ? DATTN_WIDE_F8_STAGES : DATTN_WIDE_STAGES;  // TMA ring
  static constexpr int kLoadBytes = F8 ? 2 * kWTiles * kWF8Tile : kWStageBytes;
  static constexpr int kBoxes = F8 ? 2 * kWTiles : 4 * kWTiles;  // 2 KB boxes per stage
  // where the MMAs read K and V: the TMA ring itself (bf16: the two halves of
  // each 32 KB stage), or the FP8 variant's widened K and V rings
  static constexpr int kOpK = F8 ? DATTN_WIDE_F8_OPK : kStages;
  static constexpr int kOpV = F8 ? DATTN_WIDE_F8_OPV : kStages;
  static constexpr int kKSlotBytes = F8 ? 2 * kWHalf : kWStageBytes;  // K slot stride
  static constexpr int kVSlotBytes = F8 ? 2 * kWHalf : kWStageBytes;  // V slot stride
  static constexpr int kOffLoad = 0;
  static constexpr int kOffOpK = F8 ? kOffLoad + kStages * kLoadBytes : kOffLoad;
  static constexpr int kOffOpV = F8 ? kOffOpK + kOpK * kKSlotBytes : kOffLoad + 2 * kWHalf;
  static constexpr int kOffQ = F8 ? kOffOpV + kOpV * kVSlotBytes : kOffLoad + kStages * kLoadBytes;
  // bf16: each item's query rows are staged in shared memory by the producers
  // while the previous item runs; FP8: the softmax warps load them from global
  // memory at the item's start (GB300, fw64: 205 us against 211 us staged --
  // the FP8 producers then issue only TMA boxes)
  static constexpr bool kQStaged = !F8 || DATTN_WIDE_F8_QSTAGE;
  static constexpr int kOffStat = kOffQ + (kQStaged ? kWRows * 256 : 0);
  static constexpr int kOffSched = kOffStat + 2 * kWStatBytes;
  static constexpr int kOffBar = kOffSched + ((kWSchedInts * 4 + 15) & ~15);
  // full[], empty[] of the TMA ring, then (FP8) full[] and empty[] of the K
  // ring and of the V ring, then s_full, s_free, p_full, pv_done per group,
  // q_full, q_empty, item_go, grp_sync, tmem_done
  static constexpr int kNumBars = 2 * kStages + (F8 ? 2 * (kOpK + kOpV) : 0) + 8 + 5;
  static constexpr int kSmemBytes = 1024 + kOffBar + kNumBars * 8 + 16;
  static_assert(kProducers >= 1 && kBoxes <= 32 * kProducers, "one box per producer lane");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};
// Tensor memory (512 columns x 128 lanes, lane = query row): fp32 scores
// S[g] at 64 g, fp32 outputs O[g] at 128 + 128 g, bf16 probabilities P[g]
// (64 keys packed in 32 columns) at 384 + 32 g, and the bf16 query rows Q
// (128 d packed in 64 columns) at 448 -- the A operands of both MMAs.
constexpr uint32_t kWTmemCols = 512;
constexpr uint32_t kWColO = 128;
constexpr uint32_t kWColP = 384;
constexpr uint32_t kWColQ = 448;
constexpr float kRescaleLog2 = 8.f;          // lazy rescale threshold (log2 units)

// One work item: chunk `split` of request b for kv head kvh.
struct Item {
  int b, kvh, split, L, nsplit, t_begin, t_end, n_tiles, n_iters;
};

__device__ __forceinline__ Item make_item(int chunk, int b, int kvh, int split, int L) {
  Item it;
  it.b = b;
  it.kvh = kvh;
  it.split = split;
  it.L = L;
  it.nsplit = L > 0 ? (L + chunk - 1) / chunk : 1;
  it.t_begin = split * chunk;
  it.t_end = min(L, it.t_begin + chunk);
  it.n_tiles = it.t_end > it.t_begin ? (it.t_end - it.t_begin + kTileTokens - 1) / kTileTokens : 0;
  it.n_iters = (it.n_tiles + kWTiles - 1) / kWTiles;
  return it;
}

// Schedule tables in shared memory (ints): clamped lengths [B], exclusive
// prefix of full chunks per request [B + 1], partial-chunk order, totals,
// and the length of each request's last chunk (chunk_len when it is full).
constexpr int kWSchLen = 0;
constexpr int kWSchFpre = kWMaxSchedBatch;
constexpr int kWSchPord = 2 * kWMaxSchedBatch + 1;
constexpr int kWSchTot = 3 * kWMaxSchedBatch + 1;  // full pairs, partial pairs
constexpr int kWSchRem = 3 * kWMaxSchedBatch + 4;
// one item per CTA: its request's clamped length, in the space of the
// unused length table (the item itself is the block index)
constexpr int kWSchOwnLen = kWSchLen;
// the call's chunk length (from the params, or the device planner's output)
constexpr int kWSchChunk = 3 * kWMaxSchedBatch + 3;

// Item k of this CTA. Persistent launch: position k * G + (c or G-1-c,
// alternating: snake order) in the list where pair p < F is the p-th full
// chunk in (request, chunk) order and pair F + i the last chunk of request
// pord[i] (partial or empty); kv heads are innermost, so position = pair *
// Hkv + kvh. Otherwise the block's own item (k = 0 only).
__device__ __forceinline__ bool schedule_item(const int* sch, const SplitArgs& a, int k, Item* it) {
  const int chunk = sch[kWSchChunk];
  if (!a.persistent) {
    if (k > 0) return false;
    *it = make_item(chunk, blockIdx.z, blockIdx.y, blockIdx.x, sch[kWSchOwnLen]);
    return true;
  }
  const int G = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  const int pos = k * G + ((k & 1) ? G - 1 - c : c);
  const int F = sch[kWSchTot];
  if (pos >= (F + sch[kWSchTot + 1]) * a.num_kv_heads) return false;
  const int pair = pos / a.num_kv_heads;
  const int kvh = pos - pair * a.num_kv_heads;
  int b, split;
  if (pair < F) {
    int lo = 0, hi = a.batch - 1;  // last request whose prefix is <= pair
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sch[kWSchFpre + mid] <= pair) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    split = pair - sch[kWSchFpre + b];
  } else {
    b = sch[kWSchPord + pair - F];
    const int L = sch[kWSchLen + b];
    split = L > 0 ? (L - 1) / chunk : 0;
  }
  *it = make_item(chunk, b, kvh, split, sch[kWSchLen + b]);
  return true;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Tile j of an item goes to softmax group g = j & 1 (warps 4g..4g+3): its
// scores land in TMEM buffer S[g], its probabilities in TMEM buffer P[g], and
// P.V accumulates into O[g]; the two groups alternate, so one group's softmax
// overlaps the other's, and their (m, l, O) merge exactly at the end.  Phases
// of the ring and of each group's barriers run on across items.
// KS: key split for items of at most 64 query rows (see the file comment).
template <bool F8, bool KS>
__global__ void __launch_bounds__(WCfg<F8>::kThreads, 1)
    wide_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                const SplitArgs a) {
  using C = WCfg<F8>;
  constexpr uint32_t kFull = 0xffffffffu;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool persistent = a.persistent != 0;

  grid_dependency_wait();
  // device-planned call (always persistent): the chunk length from the
  // planner's output; persistent: the first request length of this thread --
  // both loaded before the barrier and TMEM set-up so their latency overlaps
  // them
  const bool listed = a.items != nullptr;
  const int chunk = listed ? a.plan[0] : a.chunk_len;
  const int L_first = persistent && tid < a.batch ? a.seq_lens[tid] : 0;

  int L0 = 0;  // one item per CTA: its request's clamped length
  if (!persistent) {
    int L = a.seq_lens[blockIdx.z];
    uint32_t bad = 0;
    if (L < 0 || L > a.max_seq_len) {
      bad |= DA_STATUS_SEQ_LEN;
      L = L < 0 ? 0 : a.max_seq_len;
    }
    if (a.causal && L > 0 && L < a.q_len) bad |= DA_STATUS_SHORT_CAUSAL;
    if (bad && a.status != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
      atomicOr(a.status, static_cast<int32_t>(bad));
    const int nsplit = L > 0 ? (L + chunk - 1) / chunk : 1;
    if (static_cast<int>(blockIdx.x) >= nsplit) return;  // before any TMEM is allocated
    L0 = L;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full_bar = bars;                   // [kStages] TMA bytes landed
  uint64_t* empty_bar = bars + C::kStages;     // [kStages] TMA slot free again
  uint64_t* convk_full = empty_bar + C::kStages;                    // FP8: K slot widened
  uint64_t* convk_empty = convk_full + (F8 ? C::kOpK : 0);          // FP8: K slot read by S
  uint64_t* convv_full = convk_empty + (F8 ? C::kOpK : 0);          // FP8: V slot widened
  uint64_t* convv_empty = convv_full + (F8 ? C::kOpV : 0);          // FP8: V slot read by P.V
  uint64_t* s_full = convv_empty + (F8 ? C::kOpV : 0);              // [2] scores in TMEM buffer
  uint64_t* s_free = s_full + 2;               // [2] score buffer read by softmax
  uint64_t* p_full = s_free + 2;               // [2] P buffer (and O rescale) ready for PV
  uint64_t* pv_done = p_full + 2;              // [2] PV of that P buffer finished
  uint64_t* q_full = pv_done + 2;              // Q rows of the next item staged
  uint64_t* q_empty = q_full + 1;              // staging copied into TMEM
  uint64_t* item_go = q_empty + 1;             // Q in TMEM, previous outputs read (items with keys)
  uint64_t* grp_sync = item_go + 1;            // both softmax groups' statistics written (per item)
  uint64_t* tmem_done = grp_sync + 1;          // softmax warps are done with TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int* sched = reinterpret_cast<int*>(smem + C::kOffSched);
  int* s_len = sched + kWSchLen;
  int* s_fpre = sched + kWSchFpre;
  int* s_pord = sched + kWSchPord;
  int* s_tot = sched + kWSchTot;
  int* s_rem = sched + kWSchRem;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], C::kProducers);
      mbar_init(&empty_bar[s], F8 ? C::kConverters : 1);
    }
    if (F8) {
      for (int o = 0; o < C::kOpK; ++o) {
        mbar_init(&convk_full[o], C::kConverters);
        mbar_init(&convk_empty[o], 1);
      }
      for (int o = 0; o < C::kOpV; ++o) {
        mbar_init(&convv_full[o], C::kConverters);
        mbar_init(&convv_empty[o], 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_full, 32 * C::kProducers);
    mbar_init(q_empty, 4);
    mbar_init(item_go, 8);
    mbar_init(grp_sync, 8);
    mbar_init(tmem_done, 8);
    fence_mbar_init();
    if (!persistent) sched[kWSchOwnLen] = L0;
    sched[kWSchChunk] = chunk;
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, kWTmemCols);
    tmem_relinquish();
  }

  // ---- schedule tables (persistent launch): clamped lengths, full chunks
  // per request (scanned by warp 0), partial chunks ordered longest first
  if (persistent) {
    for (int b = tid; b < a.batch; b += C::kThreads) {
      int L = b == tid ? L_first : a.seq_lens[b];
      uint32_t bad = 0;
      if (L < 0 || L > a.max_seq_len) {
        bad |= DA_STATUS_SEQ_LEN;
        L = L < 0 ? 0 : a.max_seq_len;
      }
      if (a.causal && L > 0 && L < a.q_len) bad |= DA_STATUS_SHORT_CAUSAL;
      if (bad && a.status != nullptr && blockIdx.x == 0 && !listed)  // (listed: the planner)
        atomicOr(a.status, static_cast<int32_t>(bad));
      s_len[b] = L;
      const int n = L > 0 ? (L + chunk - 1) / chunk : 1;
      s_rem[b] = L - (n - 1) * chunk;  // 0 for an empty request
      s_fpre[b] = n;                   // chunk count, replaced by the prefix below
    }
    __syncthreads();
    if (warp == 0) {
      int full_run = 0, part_run = 0;
      for (int b0 = 0; b0 < a.batch; b0 += 32) {
        const int b = b0 + lane;
        int f = 0, part = 0;
        if (b < a.batch) {
          const int n = s_fpre[b];
          const int rem = s_rem[b];
          f = rem == chunk ? n : n - 1;
          part = rem == chunk ? 0 : 1;
        }
        int fi = f, pi = part;  // inclusive warp scans
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int fu = __shfl_up_sync(kFull, fi, o);
          const int pu = __shfl_up_sync(kFull, pi, o);
          if (lane >= o) {
            fi += fu;
            pi += pu;
          }
        }
        if (b < a.batch) {
          s_fpre[b] = full_run + fi - f;
          // index order of the partial chunks (re-sorted below for small batches)
          if (part && a.batch > kWSortBatch) s_pord[part_run + pi - 1] = b;
        }
        full_run += __shfl_sync(kFull, fi, 31);
        part_run += __shfl_sync(kFull, pi, 31);
      }
      if (lane == 0) {
        s_fpre[a.batch] = full_run;
        s_tot[0] = full_run;
        s_tot[1] = part_run;
      }
    }
    if (a.batch <= kWSortBatch) {
      // rank of each partial chunk among all partial chunks: longer first,
      // ties by request index
      for (int b = tid; b < a.batch; b += C::kThreads) {
        const int rem = s_rem[b];
        if (rem == chunk) continue;
        int rank = 0;
        for (int o = 0; o < a.batch; ++o) {
          const int ro = s_rem[o];
          rank += (ro != chunk && (ro > rem || (ro == rem && o < b))) ? 1 : 0;
        }
        s_pord[rank] = b;
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  // ============================================================ TMA producer
  if (warp >= C::kProducerWarp && warp < C::kConverterWarp) {
    const int pw_idx = warp - C::kProducerWarp;
    if (lane == 0 && pw_idx == 0 && a.max_seq_len > 0) {
      prefetch_tensor_map(&k_map);
      prefetch_tensor_map(&v_map);
    }
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t q_stage = smem_base + C::kOffQ;
    // this lane's box of every stage
    constexpr int kPerTile = F8 ? 2 : 4;
    const int bx = lane * C::kProducers + pw_idx;
    const int ti = bx / kPerTile;
    const int half = F8 ? 0 : (bx & 1);
    const bool is_v = F8 ? (bx & 1) != 0 : (bx & 2) != 0;
    const int box_off = F8 ? C::kOffLoad + (is_v ? kWTiles * kWF8Tile : 0) + ti * kWF8Tile
                           : C::kOffLoad + (is_v ? 2 * kWHalf : 0) + half * kWHalf + ti * 2048;
    int gs = 0;       // stages of all previous items
    int last_g = -1;  // the last stage this warp issued
    bool ok = true;
    // test hook (DA_FLAG_TEST_WITHHOLD_COPY): CTA 0 never fills the first
    // stage of its first item, so the waits on it run out and report
    // DA_STATUS_TIMEOUT
    const bool withhold =
        a.test_withhold != 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    // token -> (page, slot): shifts when the page size is a power of two (the
    // bf16 producers issue 16 boxes a stage and their instruction count sets
    // the stage pace: w64 226 -> 215 us; the FP8 variant keeps the division)
    const int ps = a.paged ? a.page_size : 1;
    const bool ps_pow2 = !F8 && (ps & (ps - 1)) == 0;
    const int ps_shift = __popc(ps - 1);
    Item it;
    for (int k = 0; ok && schedule_item(sched, a, k, &it); ++k) {
      // ---- this item's query rows into the staging buffer, one row per lane
      // (bf16; the FP8 variant's softmax warps load them themselves)
      if constexpr (C::kQStaged) {
        if (k > 0) {
          int good = 1;
          if (lane == 0) good = mbar_wait(q_empty, (k - 1) & 1) ? 1 : 0;
          if (!__shfl_sync(kFull, good, 0)) {
            ok = false;
            break;
          }
        }
        for (int r = pw_idx * 32 + lane; r < a.rows; r += 32 * C::kProducers) {
          const int t = r / a.group;
          const uint16_t* qrow = a.q + static_cast<int64_t>(it.b) * a.q_sb +
                                 static_cast<int64_t>(t) * a.q_st +
                                 static_cast<int64_t>(it.kvh * a.group + (r - t * a.group)) * a.q_sh;
#pragma unroll
          for (int c = 0; c < 16; ++c)
            cp_async16(q_stage + r * 256 + ((c ^ (r & 15)) << 4), qrow + c * 8);
        }
        cp_async_arrive(q_full);
      }

      // ---- K/V stages of the item: each producer warp issues its share of
      // every stage's 2 KB boxes (box bx = lane * kProducers + pw_idx) -- bf16:
      // tile bx / 4, K or V and the d-half from bx % 4; FP8: tile bx / 2, K or
      // V from bx % 2 (one box holds all 128 d). Each lane loads the page id
      // of its next box a stage ahead and checks it when it is used.
      // (per-item constants hoisted: the producers' instruction count per
      // stage sets the stage pace)
      const int32_t* bt_row =
          a.paged && bx < C::kBoxes ? a.block_table + static_cast<int64_t>(it.b) * a.bt_stride
                                    : nullptr;
      const int tok_lane = it.t_begin + ti * kTileTokens;  // this lane's tile start, stage 0
      const int tile_lane_end = it.n_tiles - ti;          // stage i has data if i * kWTiles < this
      auto page_of = [&](int i) -> int {  // raw block-table entry of this lane's tile in stage i
        if (bt_row == nullptr || i * kWTiles >= tile_lane_end) return 0;
        const int tok = tok_lane + i * kWTok;
        return __ldg(bt_row + (ps_pow2 ? tok >> ps_shift : tok / ps));
      };
      // boxes of this warp in a full stage, and in the item's last one
      const int last_boxes = (it.n_tiles - (it.n_iters - 1) * kWTiles) * kPerTile;
      const uint32_t full_bytes =
          static_cast<uint32_t>((C::kBoxes - pw_idx + C::kProducers - 1) / C::kProducers) * 2048u;
      const uint32_t last_bytes =
          static_cast<uint32_t>(last_boxes > pw_idx
                                    ? (last_boxes - pw_idx + C::kProducers - 1) / C::kProducers
                                    : 0) * 2048u;
      int s = gs % C::kStages;         // ring slot and its use count, advanced per stage
      int use = gs / C::kStages;
      int pg_next = page_of(0);
      for (int i = 0; i < it.n_iters; ++i) {
        int good = 1;
        if (lane == 0 && use > 0) good = mbar_wait_spin(&empty_bar[s], (use - 1) & 1) ? 1 : 0;
        good = __shfl_sync(kFull, good, 0);
        if (!good) {
          ok = false;
          break;
        }
        int pg = pg_next;
        pg_next = page_of(i + 1);
        const bool last = i == it.n_iters - 1;
        const int boxes = last ? last_boxes : C::kBoxes;  // boxes with data
        const bool skip = withhold && gs + i == 0;
        if (lane == 0 && !skip) mbar_arrive_expect_tx(&full_bar[s], last ? last_bytes : full_bytes);
        __syncwarp();
        if (bx < boxes && !skip) {
          if (a.paged && static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
            if (a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(DA_STATUS_BAD_PAGE));
            pg = 0;
          }
          const int tok = tok_lane + i * kWTok;
          const int grp = a.paged ? pg : it.b;
          const int tin = a.paged ? (ps_pow2 ? tok & (ps - 1) : tok % ps) : tok;
          tma_load_4d(smem + box_off + s * C::kLoadBytes, is_v ? &v_map : &k_map, &full_bar[s],
                      half * 64, it.kvh, tin, grp, policy);
        }
        __syncwarp();
        last_g = gs + i;
        if (++s == C::kStages) {
          s = 0;
          ++use;
        }
      }
      if (!ok) break;
      gs += it.n_iters;
    }
    cp_async_wait_all();
    if (lane == 0) {
      if (!ok && a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
      // no copy of this warp may still be landing when the CTA exits
      for (int g = max(0, last_g - C::kStages + 1); g <= last_g; ++g)
        if (!(withhold && g == 0)) mbar_wait(&full_bar[g % C::kStages], (g / C::kStages) & 1);
    }
    return;
  }

  // ======================================================= FP8 converters
  // Widen each landed FP8 stage: its K tiles into the next K slot and its V
  // tiles into the next V slot, each an f16 operand ([2 d-halves][64 tokens]
  // [64 d], 128-byte swizzle): 16-byte chunk c of FP8 row t (d = 16c ..
  // 16c+15) becomes 8-d chunks 2c and 2c+1 of d-half c / 4.  Each 8-lane
  // phase takes one chunk index of 8 consecutive rows, so loads (slot c ^ j)
  // and stores ((2c & 7) ^ j, and ^ 1) hit 8 distinct bank groups.  V rows
  // of keys past the item's chunk are written as zeros (their bytes may
  // hold anything, and NaN * 0 is NaN in P.V).
  if (F8 && warp >= C::kConverterWarp && warp < C::kMmaWarp) {
    const int ct = tid - 32 * C::kConverterWarp;
    int gs = 0;
    bool ok = true;
    Item it;
    // both halves of stage src (K into dst_k, V into dst_v) in one pass;
    // tok0 = the stage's first key, t_end = the item's end.  Chunk idx =
    // ct + 128 u of the stage's 1024 (K or V = u / 4, tile = u % 4): each
    // thread keeps its 8-row block, row j and chunk c for all eight, so the
    // addresses are a per-thread base plus constants, and all eight loads are
    // in flight before the first conversion.  (One pass per stage: each
    // barrier round trip and fence costs about as much as widening a half.)
    static_assert(!F8 || C::kConverters == 4, "the widening map assumes 128 converter threads");
    const int cj = ct & 7, cc = (ct >> 3) & 7, ctin = ((ct >> 6) & 1) * 8 + cj;
    const int c0 = (2 * cc) & 7;
    const int src_off = ctin * 128 + ((cc ^ cj) << 4);
    const int dst_off = (cc >> 2) * kWHalf + ctin * 128;
    const int st_lo = (c0 ^ cj) << 4, st_hi = ((c0 + 1) ^ cj) << 4;
    auto widen = [&](const uint8_t* src, uint8_t* dst_k, uint8_t* dst_v, int tok0, int t_end) {
      uint4 raw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        raw[u] = *reinterpret_cast<const uint4*>(src + (u >> 2) * kWTiles * kWF8Tile +
                                                 (u & 3) * kWF8Tile + src_off);
      const int v_rows = t_end - tok0;  // V rows at or past this are zeroed
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint8_t* row = (u >= 4 ? dst_v : dst_k) + dst_off + (u & 3) * kTileTokens * 128;
        uint4 lo, hi;
        e4m3x4_to_f16x4(raw[u].x, lo.x, lo.y);
        e4m3x4_to_f16x4(raw[u].y, lo.z, lo.w);
        e4m3x4_to_f16x4(raw[u].z, hi.x, hi.y);
        e4m3x4_to_f16x4(raw[u].w, hi.z, hi.w);
        if (u >= 4 && (u & 3) * kTileTokens + ctin >= v_rows) {
          lo = make_uint4(0u, 0u, 0u, 0u);
          hi = lo;
        }
        *reinterpret_cast<uint4*>(row + st_lo) = lo;
        *reinterpret_cast<uint4*>(row + st_hi) = hi;
      }
      fence_proxy_async_smem();  // the tensor core reads the widened halves
      __syncwarp();
    };
    for (int k = 0; ok && schedule_item(sched, a, k, &it); ++k) {
      for (int i = 0; i < it.n_iters; ++i, ++gs) {
        const int s = gs % C::kStages;
        const int ok_slot = gs % C::kOpK;
        const int ov_slot = gs % C::kOpV;
        ok = __all_sync(kFull, mbar_wait(&full_bar[s], (gs / C::kStages) & 1)) != 0;
        if (ok && gs >= C::kOpK)
          ok = __all_sync(kFull, mbar_wait(&convk_empty[ok_slot], ((gs / C::kOpK) - 1) & 1)) != 0;
        if (ok && gs >= C::kOpV)
          ok = __all_sync(kFull, mbar_wait(&convv_empty[ov_slot], ((gs / C::kOpV) - 1) & 1)) != 0;
        if (!ok) break;
        widen(smem + C::kOffLoad + s * C::kLoadBytes, smem + C::kOffOpK + ok_slot * C::kKSlotBytes,
              smem + C::kOffOpV + ov_slot * C::kVSlotBytes, it.t_begin + i * kWTok, it.t_end);
        if (lane == 0) {
          mbar_arrive(&convk_full[ok_slot]);
          mbar_arrive(&convv_full[ov_slot]);
          mbar_arrive(&empty_bar[s]);
        }
      }
    }
    if (!ok && lane == 0 && a.status != nullptr)
      atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
    return;
  }

  // ============================================================= MMA issuer
  // The whole warp runs this loop (all its values warp-uniform) and one
  // elected lane issues each MMA and commit.
  if (warp == C::kMmaWarp) {
    constexpr uint32_t kIdescQK = umma_idesc_bf16(kWRows, kWTok, false, false, F8);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(kWRows, kHeadDim, false, true, F8);
    // B-operand descriptors of stage 0: other stages and K-steps differ only
    // in the start-address field (16-byte units, no carry below 256 KB), so
    // each MMA adds a constant to one of these. A (Q, P) is read from TMEM.
    const uint64_t k_desc0 = umma_smem_desc(smem_base + C::kOffOpK, 16, 1024);
    // B = V [64 keys][2 x 64 d], MN-major: d-halves 8 KB apart (LBO), 8-key
    // groups 1 KB apart (SBO), 16 keys = 2 KB per K-step
    const uint64_t v_desc0 = umma_smem_desc(smem_base + C::kOffOpV, kWHalf, 1024);
    // O += P_jj . V_jj (ring stage gsj), then release the stage and the P buffer
    auto issue_pv = [&](int jj, int gsj) {
      tc_fence_after_sync();
      const uint32_t pa = tmem + kWColP + (jj & 1) * (kWTok / 2);
      const uint64_t vd = v_desc0 + static_cast<uint64_t>((gsj % C::kOpV) * (C::kVSlotBytes >> 4));
      const uint32_t d = tmem + kWColO + (jj & 1) * kHeadDim;
#pragma unroll
      for (int kk = 0; kk < kWTok / 16; ++kk)  // 16 keys = 8 P columns per K-step
        umma_bf16_ts_warp(d, pa + kk * 8, vd + kk * (2048 >> 4), kIdescPV,
                          (jj > 1 || kk > 0) ? 1u : 0u);
      umma_commit_warp(&pv_done[jj & 1]);
      umma_commit_warp(F8 ? &convv_empty[gsj % C::kOpV] : &empty_bar[gsj % C::kStages]);
    };
    // S_j = Q . K_j^T: 16 d per K-step (8 Q columns; K: d-half kk / 4, 32
    // bytes into its 128-byte swizzled rows)
    auto issue_qk = [&](int j, int gsj) {
      tc_fence_after_sync();
      const uint64_t kd = k_desc0 + static_cast<uint64_t>((gsj % C::kOpK) * (C::kKSlotBytes >> 4));
      const uint32_t d = tmem + (j & 1) * kWTok;
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        umma_bf16_ts_warp(d, tmem + kWColQ + kk * 8, kd + (((kk >> 2) * kWHalf + (kk & 3) * 32) >> 4),
                          kIdescQK, kk > 0 ? 1u : 0u);
      umma_commit_warp(&s_full[j & 1]);
      if constexpr (F8) umma_commit_warp(&convk_empty[gsj % C::kOpK]);  // its K slot is free
    };
    bool ok = true;
    int gs = 0;         // ring stages consumed so far (all items)
    int u0 = 0, u1 = 0; // tiles of each softmax group so far (all items)
    int go = 0;         // items with keys so far
    Item it;
    for (int k = 0; ok && schedule_item(sched, a, k, &it); ++k) {
      if (it.n_iters == 0) continue;  // an empty request: output written by the softmax warps
      // Q of this item in TMEM, the previous item's outputs read out
      ok = __any_sync(kFull, mbar_wait(item_go, go & 1)) != 0;
      ++go;
      if (!ok) break;
      // event loop: issue the next S = Q.K^T as soon as its stage has landed
      // and its score buffer is free, and the next O += P.V as soon as its
      // probabilities are ready -- neither waits on the other, so the two
      // softmax groups overlap. A phase seen complete by any lane is complete.
      const int n = it.n_iters;
      int next_qk = 0, next_pv = 0;
      unsigned long long idle_since = 0;
      while (next_pv < n) {
        bool progress = false;
        if (next_qk < n) {
          const int j = next_qk;
          const int gsj = gs + j;
          const int u = ((j & 1) ? u1 : u0) + (j >> 1);  // the group's use of its buffers
          const bool landed = F8 ? mbar_test(&convk_full[gsj % C::kOpK], (gsj / C::kOpK) & 1)
                                 : mbar_test(&full_bar[gsj % C::kStages], (gsj / C::kStages) & 1);
          const bool s_ready = u == 0 || mbar_test(&s_free[j & 1], (u - 1) & 1);
          if (__any_sync(kFull, landed) && __any_sync(kFull, s_ready)) {
            issue_qk(j, gsj);
            ++next_qk;
            progress = true;
          }
        }
        if (next_pv < next_qk) {
          const int jj = next_pv;
          const int u = ((jj & 1) ? u1 : u0) + (jj >> 1);
          const int gsv = gs + jj;  // (FP8: its V slot must be widened too)
          const bool v_ready = !F8 || mbar_test(&convv_full[gsv % C::kOpV], (gsv / C::kOpV) & 1);
          if (__any_sync(kFull, v_ready) && __any_sync(kFull, mbar_test(&p_full[jj & 1], u & 1))) {
            issue_pv(jj, gs + jj);
            ++next_pv;
            progress = true;
          }
        }
        if (progress) {
          idle_since = 0;
        } else {
          const unsigned long long now = __shfl_sync(kFull, global_timer_ns(), 0);
          if (idle_since == 0) {
            idle_since = now;
          } else if (now - idle_since > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
      }
      gs += n;
      u0 += (n + 1) >> 1;
      u1 += n >> 1;
    }
    // TMEM is released once the softmax warps are done with it.  Each of
    // their waits gives up after kWaitLimitNs, and after a failure a softmax
    // warp passes at most two more waits (its group's statistics exchange and
    // this arrival) before arriving here, so kTmemDoneWaits limits cover it
    // with room to spare; should even that run out, TMEM is released anyway
    // (a CTA that kept it would block the next allocation on this SM).
    constexpr unsigned long long kTmemDoneWaits = 5;
    ok = (__all_sync(kFull, mbar_wait_for(tmem_done, 0, kTmemDoneWaits * kWaitLimitNs)) != 0) && ok;
    if (!ok && lane == 0 && a.status != nullptr)
      atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
    tc_fence_after_sync();
    tmem_dealloc(tmem, kWTmemCols);
    return;
  }

  // ================================================ softmax groups (warps 0-7)
  const int grp = warp >> 2;       // softmax group: tiles j with j & 1 == grp
  const int r = tid & 127;         // TMEM lane
  // query row of the lane and (key split) the half of each tile it takes
  const int row = KS ? ((r >> 5) << 4) | (r & 15) : r;
  const int kh = KS ? (r >> 4) & 1 : 0;
  constexpr int kKeys = KS ? kWTok / 2 : kWTok;  // keys of a tile per thread
  const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const uint32_t o_col = kWColO + grp * kHeadDim;
  const uint8_t* q_stage = smem + C::kOffQ + row * 256;
  int gs = 0;      // ring stages of all previous items
  int u_base = 0;  // this group's tiles in all previous items
  bool ok = true;
  Item it;
  for (int k = 0; schedule_item(sched, a, k, &it); ++k) {
    const int t_end = it.t_end;
    int lim = 0;  // keys j < lim are visible to this row (0 for padding rows)
    if (row < a.rows) {
      const int t = row / a.group;
      lim = a.causal ? min(t_end, it.L - a.q_len + 1 + t) : t_end;
    }
    // ---- this item's query row (zeros for padding rows) into TMEM lane r:
    // the A operand of S = Q.K^T, d pairs packed in 64 columns (group 0: one
    // row per thread).  FP8: straight from global memory, all 16 chunks of the
    // row in flight at once, widened to f16 (the products run in f16).
    if (!C::kQStaged && grp == 0) {
      if (ok) {
        uint4 v[16];
        if (row < a.rows) {
          const int t = row / a.group;
          const uint4* qrow = reinterpret_cast<const uint4*>(
              a.q + static_cast<int64_t>(it.b) * a.q_sb + static_cast<int64_t>(t) * a.q_st +
              static_cast<int64_t>(it.kvh * a.group + (row - t * a.group)) * a.q_sh);
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) v[ch] = __ldg(qrow + ch);
        } else {
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) v[ch] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int qc = 0; qc < 4; ++qc) {  // 32 d = 16 columns per step
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 x = v[qc * 4 + c];
            w[4 * c] = bf16x2_to_f16x2(x.x);
            w[4 * c + 1] = bf16x2_to_f16x2(x.y);
            w[4 * c + 2] = bf16x2_to_f16x2(x.z);
            w[4 * c + 3] = bf16x2_to_f16x2(x.w);
          }
          tmem_st16(lane_base + kWColQ + qc * 16, w);
        }
        tmem_wait_st();
      }
    }
    // (or from the staging buffer the producers filled)
    if (C::kQStaged && grp == 0) {
      if (ok) ok = __all_sync(kFull, mbar_wait(q_full, k & 1)) != 0;
      if (ok) {
#pragma unroll 1
        for (int qc = 0; qc < 4; ++qc) {  // 32 d = 16 columns per step
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = qc * 4 + c;
            const uint4 v = row < a.rows
                                ? *reinterpret_cast<const uint4*>(q_stage + ((ch ^ (row & 15)) << 4))
                                : make_uint4(0, 0, 0, 0);
            // FP8 caches: the products run in f16, so Q is widened too
            w[4 * c] = F8 ? bf16x2_to_f16x2(v.x) : v.x;
            w[4 * c + 1] = F8 ? bf16x2_to_f16x2(v.y) : v.y;
            w[4 * c + 2] = F8 ? bf16x2_to_f16x2(v.z) : v.z;
            w[4 * c + 3] = F8 ? bf16x2_to_f16x2(v.w) : v.w;
          }
          tmem_st16(lane_base + kWColQ + qc * 16, w);
        }
        tmem_wait_st();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);
    }
    // item_go advances only on items with keys, so its phases cannot run two
    // ahead of the MMA warp: each such item's tiles need the MMAs
    if (it.n_iters > 0) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(item_go);
    }

    float m_used = -INFINITY;  // reference max of P (log2 domain), raised lazily
    float l = 0.f;             // sum of the fp32 probabilities (for the LSE)
    float lq = 0.f;            // sum of the probabilities as rounded into P (divides O)
    const int n_iters = it.n_iters;
    const int my_tiles = grp == 0 ? (n_iters + 1) >> 1 : n_iters >> 1;
    for (int j = grp; ok && j < n_iters; j += 2) {
      const int lu = j >> 1;          // use of this group's buffers within the item
      const int u = u_base + lu;      // ... and over all items (barrier phases)
      ok = __all_sync(kFull, mbar_wait(&s_full[grp], u & 1)) != 0;
      if (!ok) break;
      tc_fence_after_sync();
      // (tcgen05.ld and .st take one column address for the whole warp, so
      // a key-split lane reads the whole score row and keeps its half)
      float x[kKeys];
      {
        float lo[32], hi[32];
        tmem_ld32(lane_base + grp * kWTok, lo);
        tmem_ld32(lane_base + grp * kWTok + 32, hi);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if constexpr (KS) {
            x[i] = kh ? hi[i] : lo[i];
          } else {
            x[i] = lo[i];
            x[32 + i] = hi[i];
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[grp]);

      // ---- scale, masks (only on tiles that reach past this row's limit) and
      // the lazy running max
      // With a positive scale the max of the scaled scores is the scale times
      // the max of the raw ones, so the scores stay raw and the scale goes into
      // the exponent's multiply-add below (s_fma; one multiply less per score);
      // any other scale scales them here (s_fma = 1).
      const int tile0 = it.t_begin + j * kWTok;
      const int tok0 = tile0 + kh * kKeys;  // this thread's first key
      const bool raw = a.scale_log2 > 0.f;
      const float s_fma = raw ? a.scale_log2 : 1.f;
      float mt = -INFINITY;
      if (raw) {
        if (tok0 + kKeys <= lim) {
#pragma unroll
          for (int i = 0; i < kKeys; i += 2) mt = fmax3(mt, x[i], x[i + 1]);
        } else {
#pragma unroll
          for (int i = 0; i < kKeys; i += 2) {
            x[i] = tok0 + i < lim ? x[i] : -INFINITY;
            x[i + 1] = tok0 + i + 1 < lim ? x[i + 1] : -INFINITY;
            mt = fmax3(mt, x[i], x[i + 1]);
          }
        }
        mt *= a.scale_log2;
      } else {
#pragma unroll
        for (int i = 0; i < kKeys; i += 2) {
          x[i] = tok0 + i < lim ? x[i] * a.scale_log2 : -INFINITY;
          x[i + 1] = tok0 + i + 1 < lim ? x[i + 1] * a.scale_log2 : -INFINITY;
          mt = fmax3(mt, x[i], x[i + 1]);
        }
      }
      const bool raise = mt != -INFINITY && (m_used == -INFINITY || mt > m_used + kRescaleLog2);
      const float alpha = raise ? (m_used == -INFINITY ? 0.f : ex2(m_used - mt)) : 1.f;
      if (raise) m_used = mt;
      const float mref = m_used == -INFINITY ? 0.f : m_used;  // all masked so far: p = 0
      // (pairs of scores in the packed two-wide fp32 instructions: half the
      // issue slots for the exponent arguments and the running sums)
      uint32_t pk[kKeys / 2];
      float2 ps = make_float2(0.f, 0.f), qs = make_float2(0.f, 0.f);
      const float2 s2 = make_float2(s_fma, s_fma);
      const float2 nm2 = make_float2(-mref, -mref);
#pragma unroll
      for (int i = 0; i < kKeys; i += 2) {
        const float2 e = __ffma2_rn(make_float2(x[i], x[i + 1]), s2, nm2);
        const float p0 = ex2(e.x);
        const float p1 = ex2(e.y);
        ps = __fadd2_rn(ps, make_float2(p0, p1));
        pk[i / 2] = F8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
        // bf16 P: the sum of the rounded weights normalises O (f16 P of the
        // FP8 path rounds to 2^-11, well inside the bar: its fp32 sum serves)
        if constexpr (!F8)
          qs = __fadd2_rn(qs, make_float2(packed_lo(pk[i / 2], false), packed_hi(pk[i / 2], false)));
      }
      l = l * alpha + (ps.x + ps.y);
      lq = F8 ? l : lq * alpha + (qs.x + qs.y);

      // ---- this group's previous P.V (tile j - 2) must be done before its O
      // is rescaled and its P buffer rewritten (the previous use may belong to
      // the previous item: then only the wait, no rescale)
      if (u >= 1) {
        ok = __all_sync(kFull, mbar_wait(&pv_done[grp], (u - 1) & 1)) != 0;
        if (!ok) break;
        tc_fence_after_sync();
        if (lu >= 1 && __any_sync(kFull, raise && alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < kHeadDim / 32; ++c) {
            float o[32];
            tmem_ld32(lane_base + o_col + c * 32, o);
            tmem_wait_ld();
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 v = __fmul2_rn(make_float2(o[i], o[i + 1]), a2);
              o[i] = v.x;
              o[i + 1] = v.y;
            }
            tmem_st32(lane_base + o_col + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      // P row (64 bf16 packed in 32 columns) into TMEM: the A operand of P.V
      // (key split: zeros over the other half of the tile)
      {
        float w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if constexpr (KS) {
            const uint32_t v = i < 16 ? (kh ? 0u : pk[i]) : (kh ? pk[i - 16] : 0u);
            w[i] = __uint_as_float(v);
          } else {
            w[i] = __uint_as_float(pk[i]);
          }
        }
        tmem_st32(lane_base + kWColP + grp * (kWTok / 2), w);
      }
      // keys past the chunk end: their V rows may hold anything (NaN * 0 is
      // NaN), so zero them before the MMA reads the stage (FP8: the
      // converters already wrote those rows as zeros)
      const int n_valid = min(kWTok, t_end - tile0);
      if (!F8 && n_valid < kWTok) {
        uint8_t* vst = smem + C::kOffOpV + ((gs + j) % C::kOpV) * C::kVSlotBytes;
        for (int idx = r; idx < (kWTok - n_valid) * 16; idx += 128) {
          const int row = n_valid + (idx >> 4);
          const int c = idx & 15;  // 8 chunks per half, 2 halves
          *reinterpret_cast<uint4*>(vst + (c >> 3) * kWHalf + row * 128 + (c & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[grp]);
    }
    if (ok && my_tiles > 0) {
      ok = __all_sync(kFull, mbar_wait(&pv_done[grp], (u_base + my_tiles - 1) & 1)) != 0;
      tc_fence_after_sync();
    }
    gs += n_iters;
    u_base += my_tiles;

    // ---- merge the two groups (same recurrence as the combine) and write
    // O / l (final bf16 row or fp32 partial) and the LSE; group g writes the
    // d-columns [64 g, 64 g + 64) of every row
    // The exchange needs one barrier per item: the buffer (k & 1) was last
    // read before item k - 1's barrier, which every writer has passed; the
    // barrier also orders both groups' last P.V (each waited for its own)
    // before either reads the other's O columns.  It is an mbarrier (one
    // arrival per warp) with a bounded wait; a warp whose wait runs out
    // reports it through the flags and the item loop ends.
    float* stat = reinterpret_cast<float*>(smem + C::kOffStat + (k & 1) * kWStatBytes);
    stat[grp * 384 + r] = m_used;
    stat[grp * 384 + 128 + r] = l;
    stat[grp * 384 + 256 + r] = lq;
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
      stat[768 + warp] = ok ? 1.f : 0.f;
      mbar_arrive(grp_sync);
    }
    const bool synced = __all_sync(kFull, mbar_wait(grp_sync, k & 1)) != 0;
    tc_fence_after_sync();
    ok = synced;
#pragma unroll
    for (int w = 0; w < 8; ++w) ok = ok && stat[768 + w] != 0.f;  // (all 256 threads agree
                                                                  //  unless a wait ran out)
    const float m0 = stat[r], l0 = stat[128 + r], q0 = stat[256 + r];
    const float m1 = stat[384 + r], l1 = stat[512 + r], q1 = stat[640 + r];
    float M = fmaxf(m0, m1);
    // key split: the other half of this row is lane r ^ 16 of this warp
    float pm0 = -INFINITY, pl0 = 0.f, pq0 = 0.f, pm1 = -INFINITY, pl1 = 0.f, pq1 = 0.f;
    if constexpr (KS) {
      pm0 = __shfl_xor_sync(kFull, m0, 16);
      pl0 = __shfl_xor_sync(kFull, l0, 16);
      pq0 = __shfl_xor_sync(kFull, q0, 16);
      pm1 = __shfl_xor_sync(kFull, m1, 16);
      pl1 = __shfl_xor_sync(kFull, l1, 16);
      pq1 = __shfl_xor_sync(kFull, q1, 16);
      M = fmaxf(M, fmaxf(pm0, pm1));
    }
    const float Mu = M == -INFINITY ? 0.f : M;
    const float f0 = l0 > 0.f ? ex2(m0 - Mu) : 0.f;
    const float f1 = l1 > 0.f ? ex2(m1 - Mu) : 0.f;
    float Lt = l0 * f0 + l1 * f1;  // the LSE's sum
    float Qt = q0 * f0 + q1 * f1;  // the weights P.V actually used
    if constexpr (KS) {
      const float pf0 = pl0 > 0.f ? ex2(pm0 - Mu) : 0.f;
      const float pf1 = pl1 > 0.f ? ex2(pm1 - Mu) : 0.f;
      Lt += pl0 * pf0 + pl1 * pf1;
      Qt += pq0 * pf0 + pq1 * pf1;
    }
    const float inv = (Qt > 0.f ? 1.f / Qt : 0.f) * (F8 ? a.v_scale : 1.f);
    const bool have0 = ok && n_iters > 0;  // O[0] / O[1] were written
    const bool have1 = ok && n_iters > 1;
    const bool direct = it.nsplit == 1;
    const int S = a.num_splits;
    const int t = row < a.rows ? row / a.group : 0;
    const int h = it.kvh * a.group + (row - t * a.group);
    const int64_t prow = (static_cast<int64_t>(it.b) * a.q_len + t) * a.num_q_heads + h;
    // partial slot of this row: by item for a device-planned call (item =
    // pre[b] * Hkv + kvh * n_b + chunk), else by (row, chunk)
    const int64_t pidx =
        direct ? 0
        : listed ? (static_cast<int64_t>(a.pre[it.b]) * a.num_kv_heads +
                    static_cast<int64_t>(it.kvh) * it.nsplit + it.split) * a.rows + row
                 : prow * S + it.split;
    // (O is read out here, before this thread's next arrival on item_go lets
    // the next item's P.V overwrite it)
    // both buffers are read unconditionally (a buffer this item did not
    // write holds stale values that the selects below drop), 32 columns at a
    // time (two TMEM round trips; the tile loop's registers are free by now)
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      const int d0 = grp * 64 + c * 32;
      float o0[32], o1[32];
      tmem_ld32(lane_base + kWColO + d0, o0);
      tmem_ld32(lane_base + kWColO + kHeadDim + d0, o1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) o0[i] = (have0 ? o0[i] * f0 : 0.f) + (have1 ? o1[i] * f1 : 0.f);
      if constexpr (KS) {
        // this lane writes columns [d0 + 16 kh, d0 + 16 kh + 16) of the row:
        // its own sum there plus the other half's, which it receives for the
        // columns it sends (every lane of the warp takes part)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mine = kh ? o0[16 + i] : o0[i];
          const float theirs = __shfl_xor_sync(kFull, kh ? o0[i] : o0[16 + i], 16);
          o0[i] = (mine + theirs) * inv;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o0[i] *= inv;
      }
      constexpr int kCols = KS ? 16 : 32;  // columns this thread writes
      const int dw = d0 + kh * kCols;
      if (row < a.rows) {
        if (direct) {
          uint16_t* dst = a.out + static_cast<int64_t>(it.b) * a.o_sb +
                          static_cast<int64_t>(t) * a.o_st + static_cast<int64_t>(h) * a.o_sh + dw;
#pragma unroll
          for (int i = 0; i < kCols; i += 8)
            *reinterpret_cast<uint4*>(dst + i) =
                make_uint4(pack_bf16x2(o0[i], o0[i + 1]), pack_bf16x2(o0[i + 2], o0[i + 3]),
                           pack_bf16x2(o0[i + 4], o0[i + 5]), pack_bf16x2(o0[i + 6], o0[i + 7]));
        } else {
          float* dst = a.part_o + pidx * kHeadDim + dw;
          const uint64_t keep = l2_evict_last_policy();
#pragma unroll
          for (int i = 0; i < kCols; i += 4)
            st_global_hint(dst + i, make_float4(o0[i], o0[i + 1], o0[i + 2], o0[i + 3]), keep);
        }
      }
    }
    if (grp == 0 && kh == 0 && row < a.rows) {
      const float lse = Lt > 0.f ? (Mu + log2f(Lt)) * kLn2w : -INFINITY;
      if (direct)
        a.lse[prow] = lse;
      else
        st_global_hint(a.part_lse + pidx, lse, l2_evict_last_policy());
    }
    if (!ok) break;
  }
  if (!ok && lane == 0 && a.status != nullptr)
    atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive(tmem_done);  // the MMA warp releases TMEM after all 8
}

std::mutex g_wide_mu;
bool g_wide_attr[2][64];
int g_wide_sms[64];

template <bool F8>
cudaError_t ensure_wide_attrs(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_wide_mu);
  if (!g_wide_attr[F8][dev]) {
    e = cudaFuncSetAttribute(wide_kernel<F8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             WCfg<F8>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(wide_kernel<F8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             WCfg<F8>::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&g_wide_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_wide_attr[F8][dev] = true;
  }
  if (sms != nullptr) *sms = g_wide_sms[dev];
  return cudaSuccess;
}

template <bool F8>
cudaError_t launch_wide_t(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                          cudaStream_t stream) {
  int sms = 0;
  cudaError_t e = ensure_wide_attrs<F8>(&sms);
  if (e != cudaSuccess) return e;
  SplitArgs pa = a;
  pa.persistent = a.batch <= kWMaxSchedBatch ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  // persistent: one CTA per SM (at most one per possible item); otherwise one
  // CTA per item.  Device-planned calls (batch <= kWMaxSchedBatch, checked by
  // the host) are always persistent.
  const bool listed = a.items != nullptr;
  if (listed && !pa.persistent) return cudaErrorInvalidValue;
  const int64_t items = listed ? a.item_slots
                               : static_cast<int64_t>(a.num_splits) * a.num_kv_heads * a.batch;
  cfg.gridDim = pa.persistent ? dim3(static_cast<unsigned>(std::min<int64_t>(sms, items)))
                              : dim3(a.num_splits, a.num_kv_heads, a.batch);
  cfg.blockDim = dim3(WCfg<F8>::kThreads);
  cfg.dynamicSmemBytes = WCfg<F8>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // up to 64 query rows: the key-split form
  return a.rows <= kWRows / 2 ? cudaLaunchKernelEx(&cfg, wide_kernel<F8, true>, k_map, v_map, pa)
                              : cudaLaunchKernelEx(&cfg, wide_kernel<F8, false>, k_map, v_map, pa);
}

}  // namespace

cudaError_t launch_wide(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                        cudaStream_t stream) {
  return a.kv_fp8 ? launch_wide_t<true>(k_map, v_map, a, stream)
                  : launch_wide_t<false>(k_map, v_map, a, stream);
}

int wide_ctas_per_sm() {
  static int cached[64];  // per device, queried once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (ensure_wide_attrs<false>(nullptr) != cudaSuccess) return 1;
  {
    std::lock_guard<std::mutex> lk(g_wide_mu);
    if (cached[dev] > 0) return cached[dev];
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, wide_kernel<false, false>, WCfg<false>::kThreads,
                                                    WCfg<false>::kSmemBytes) != cudaSuccess ||
      n < 1)
    return 1;
  std::lock_guard<std::mutex> lk(g_wide_mu);
  cached[dev] = n;
  return n;
}

}  // namespace dattn
