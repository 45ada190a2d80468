// split_kernel.cu -- the per-chunk kernel of split-KV decode attention.
//
// One CTA owns one (chunk of KV tokens, kv head, request) work item (the
// FlashDecoding split of "Capstone FlashAttention", §2.3: with one query token
// the KV *sequence* is cut into chunks that run on different SMs).  Inside the
// CTA:
//   * a producer warp gathers the chunk's 16-token pages through the block
//     table and streams K and V into a ring of shared-memory stages with TMA
//     tensor loads (cp.async.bulk.tensor, 128-byte swizzle, completion counted
//     on an mbarrier), several stages ahead of the math -- the asynchronous,
//     multi-buffered prefetch of the pages' copy pipelines ("Capstone
//     FlashAttention", §2.2 TMA / producer-consumer warps; the CUDA-optimisation
//     article, §3.3 double buffering);
//   * each consumer warp takes one 16-token tile per stage and computes
//     S^T = K . Q^T on the tensor cores (mma.sync m16n8k16 bf16 -> fp32), with
//     the GQA group x q_len query rows as the 8- or 16-wide N side, so a tile
//     of keys against all rows that share its KV head is one dense product;
//     then the online-softmax update of running max m and running sum l
//     ("Capstone FlashAttention", §1.2 recurrence: m' = max(m, rowmax),
//     alpha = e^{m-m'}, l' = alpha l + sum p, O' = alpha O + P V), with the
//     division deferred to the end (§2.1), and O^T += V^T . P^T on the tensor
//     cores (P rounded to bf16; movmatrix turns the score fragment into the
//     B operand without a trip through shared memory);
//   * the consumer warps' states are merged with the same recurrence, and the
//     CTA writes either the final bf16 output and LSE (request fits one
//     chunk) or an fp32 partial output plus its natural-log LSE for the
//     combine kernel (the per-tile LSE buffer of the CUTLASS split-KV post,
//     §4.2).
// Exponentials are taken base 2 on scores pre-multiplied by log2(e).
// FP8 caches (F8): one TMA box carries all 128 E4M3 values of a 16-token tile
// (half the bytes of bf16), and the MMA operands are built from those bytes in
// registers (every E4M3 value is an f16 value; cvt.e4m3x2 widens pairs):
// ldmatrix (b16) on the FP8 K tile gives a thread 4 consecutive d of one key,
// used as the k pairs (2t4, 2t4+1) and (8+2t4, 9+2t4) of a 16-d step -- a
// permutation of d inside the step, applied to Q's fragment as well, which
// leaves the dot product unchanged; ldmatrix.trans (b16) on the FP8 V tile
// gives a thread 2 d x 2 keys, split by byte permutes into the V^T fragment
// rows d = 2g4 and 2g4 + 1 of the 16-d output tile (so the O^T accumulator's
// rows g4 / g4 + 8 are d = 16mt + 2g4 / + 1).  Both products run on f16
// operands (Q widened from bf16, P rounded to f16); k_scale is folded into the
// score scale and v_scale into the output.
// Keys at or past seq_len (and, with the causal mask, past a row's own
// position) are masked to -inf; V rows past seq_len in a request's last page
// are zeroed in shared memory first, since those slots may hold anything.

#include <mutex>

#include "decode_attn.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace dattn {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

#ifndef DATTN_Q_SMEM
#define DATTN_Q_SMEM 1
#endif
template <int NT, int STAGES, int TPS, bool F8 = false>
struct SplitCfg {
  static constexpr int kThreads = 32 * (TPS + 1);        // TPS consumer warps + 1 producer
  static constexpr int kHalfBytes = kTileTokens * 64 * 2;  // [16 tokens][64 d] bf16
  // one 16-token K (or V) tile: two bf16 halves, or 16 rows of 128 FP8 bytes
  static constexpr int kTileBytes = F8 ? kTileTokens * 128 : 2 * kHalfBytes;
  static constexpr int kStageBytes = 2 * TPS * kTileBytes;  // TPS K tiles, then TPS V tiles
  // Inside the K (or V) region of a stage the layout is d-half-major: the
  // 128-byte rows of the TPS tiles' first 64 d (bf16), then of their last 64
  // d -- [2 halves][16 TPS tokens][128 B] -- so one TMA box of 16 TPS tokens
  // fills a whole half (contiguous caches) and 16-token boxes (paged caches)
  // land in the same place.  FP8 tiles are whole 128-byte rows already.
  static constexpr int kRegionBytes = TPS * kTileBytes;    // K (or V) of a stage
  static constexpr int kTileStride = kTileTokens * 128;    // next tile, same d-half
  static constexpr int kHalfStride = F8 ? 0 : TPS * kTileStride;  // next d-half
  static constexpr int kPipeBytes = STAGES * kStageBytes;
  static constexpr int kRows = 8 * NT;                     // padded query rows
  static constexpr int kRedStride = kHeadDim + 4;          // floats per row (bank spread)
  static constexpr int kRedBytes = TPS * kRows * kRedStride * 4;
  static_assert(kRedBytes <= kPipeBytes, "merge scratch must fit in the stage ring");
  static_assert(4 * TPS <= 32, "one TMA box per producer lane");
  // cluster merge: this CTA's normalised output [kRows][128] fp32, after the
  // warp-merge scratch in the (idle) stage ring, and its per-row LSE
  static constexpr int kXoOffset = (kRedBytes + 127) / 128 * 128;
  static_assert(kXoOffset + kRows * kHeadDim * 4 <= kPipeBytes, "cluster output must fit");
  // 16-row variants read their Q fragments from shared memory each step
  // instead of holding all 32 in registers for the whole loop: [16 rows][16
  // chunks of 16 B], chunk c of row r at c ^ (r & 7) (FP8: d permuted within
  // each 16-d step to match the K fragments, in f16)
  static constexpr bool kQSmem = NT == 2 && DATTN_Q_SMEM;
  static constexpr int kQBytes = kQSmem ? kRows * 256 : 0;
  static constexpr int kBarBytes = 2 * STAGES * 8;
  static constexpr int kStatBytes = 3 * TPS * kRows * 4 + kRows * 4;
  // Cluster merge of the deep bf16 shape (4 tiles per stage; it runs at most
  // one CTA per SM, so shared memory is plentiful): every CTA pushes its
  // merged (row, 4 d) units and their rows' LSEs into the inbox of the CTA
  // that owns each unit.  Unit u of U = rows x 32 goes to CTA u mod S, slot
  // u / S, so an inbox holds S x ceil(U / S) <= U + 15 entries per array.
  static constexpr bool kPushMerge = TPS == 4 && !F8;
  static constexpr int kInboxUnits = kRows * 32 + 16;
  static constexpr int kOffInbox = (kPipeBytes + kQBytes + kBarBytes + kStatBytes + 15) / 16 * 16;
  static constexpr int kInboxBytes = kPushMerge ? kInboxUnits * (16 + 4) : 0;
  static constexpr int kSmemBytes = 1024 + kOffInbox + kInboxBytes;
};

// Byte address of 16-byte chunk `chunk` (0..15, i.e. d = 8*chunk) of token row
// `tok` inside one bf16 tile: d-half chunk / 8 at half_stride bytes per half,
// 128-byte rows, chunk index XOR-ed with (tok & 7) as the TMA 128-byte swizzle
// lays it out (every half starts on a 1024-byte boundary).
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int tok, int chunk,
                                              uint32_t half_stride) {
  return tile + (chunk >> 3) * half_stride + (tok << 7) + (((chunk & 7) ^ (tok & 7)) << 4);
}

__device__ __forceinline__ uint32_t load_u32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// CM (cluster merge): the num_splits CTAs of one (kv head, request) form one
// thread-block cluster; instead of writing fp32 partials for the combine
// kernel they merge their results through distributed shared memory and write
// the final output themselves.
// LS (listed): a device-planned call; CTA i takes item slot i of the device
// planner's list.  A separate instantiation, because a CTA's (chunk, kv head,
// request) read from memory is per-thread data to the compiler, while the
// grid-planned variants take them from blockIdx and the kernel parameters as
// warp-uniform values, so every index and address derived from them stays in
// the uniform datapath instead of costing a per-thread instruction each.
template <int NT, int STAGES, int TPS, bool CM, bool F8, bool LS>
__global__ void __launch_bounds__(SplitCfg<NT, STAGES, TPS, F8>::kThreads)
    split_kv_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const SplitArgs a) {
  static_assert(!(CM && LS), "a device-planned call writes partials");
  using C = SplitCfg<NT, STAGES, TPS, F8>;
  constexpr uint32_t kFull = 0xffffffffu;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr bool listed = LS;

  // launched early behind the previous kernel of the stream (or the device
  // planner): nothing it may write (q, caches, lengths, the plan, outputs)
  // is touched before this
  grid_dependency_wait();

  // ---- this CTA's work item and key range [t_begin, t_end)
  int split, kvh, b, L, chunk;
  if constexpr (listed) {
    // item slot blockIdx.x of the planner's list (slots past its count exit)
    const int n_items = a.plan[1];
    const int4 itm = a.items[blockIdx.x];
    chunk = a.plan[0];
    if (static_cast<int>(blockIdx.x) >= n_items) return;
    b = itm.x;
    kvh = itm.y;
    split = itm.z;
    L = itm.w;  // clamped (and reported) by the planner
  } else {
    split = blockIdx.x;
    kvh = blockIdx.y;
    b = blockIdx.z;
    L = a.seq_lens[b];  // (under the cluster merge its load overlaps the set-up)
    chunk = a.chunk_len;
  }
  // the request length, clamped, with its status bits (grid-planned calls)
  auto take_length = [&]() {
    if constexpr (listed) return;
    uint32_t bad = 0;
    if (L < 0 || L > a.max_seq_len) {
      bad |= DA_STATUS_SEQ_LEN;
      L = L < 0 ? 0 : a.max_seq_len;
    }
    if (a.causal && L > 0 && L < a.q_len) bad |= DA_STATUS_SHORT_CAUSAL;
    if (bad && a.status != nullptr && split == 0 && kvh == 0 && threadIdx.x == 0)
      atomicOr(a.status, static_cast<int32_t>(bad));
  };
  if constexpr (!CM) {
    // a CTA past its request's chunks exits before any set-up (with the
    // cluster merge every CTA stays: an empty chunk contributes 0 / -inf)
    take_length();
    if (split >= (L > 0 ? (L + chunk - 1) / chunk : 1)) return;
  }
  const int t_begin = split * chunk;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = smem + C::kPipeBytes;  // (16-row variants)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes + C::kQBytes);
  uint64_t* empty_bar = full_bar + STAGES;
  float* stat_m = reinterpret_cast<float*>(empty_bar + STAGES);
  float* stat_l = stat_m + TPS * C::kRows;
  float* stat_q = stat_l + TPS * C::kRows;
  float* xl = stat_q + TPS * C::kRows;  // cluster merge: this CTA's per-row LSE
  float4* inbox_v = reinterpret_cast<float4*>(smem + C::kOffInbox);  // (push merge)
  float* inbox_l = reinterpret_cast<float*>(smem + C::kOffInbox + C::kInboxUnits * 16);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], TPS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // push merge: the first phase of the cluster barrier, waited on just
  // before the pushes (every peer has started by then)
  if constexpr (CM && C::kPushMerge) cluster_arrive_relaxed();

  // Cluster merge with a contiguous cache: the first stage is one box per (K
  // or V, d-half) from t_begin, which does not depend on the request length,
  // so the producer issues it while the length's load is still in flight (a
  // chunk that turns out empty or short just leaves some of it unused; the
  // producer still waits for it before leaving).  (t_begin < max_seq_len for
  // every chunk of the grid, so the box starts inside the cache.)
  const bool early = CM && a.big_box != 0;
  if (CM && early && warp == TPS) {
    if (lane == 0) {
      prefetch_tensor_map(&k_map);
      prefetch_tensor_map(&v_map);
      mbar_arrive_expect_tx(&full_bar[0], static_cast<uint32_t>(C::kStageBytes));
    }
    __syncwarp();
    if (lane < (F8 ? 2 : 4)) {
      const bool is_v = F8 ? (lane & 1) != 0 : (lane & 2) != 0;
      const int half = F8 ? 0 : lane & 1;
      tma_load_4d(smem + (is_v ? C::kRegionBytes : 0) + half * C::kHalfStride,
                  is_v ? &v_map : &k_map, &full_bar[0], half * 64, kvh, t_begin, b,
                  l2_evict_first_policy());
    }
  }
  if constexpr (CM) take_length();
  const int nsplit_b = L > 0 ? (L + chunk - 1) / chunk : 1;
  const int t_end = min(L, t_begin + chunk);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTileTokens - 1) / kTileTokens : 0;
  const int n_iters = (n_tiles + TPS - 1) / TPS;

  // =========================================================== producer warp
  if (warp == TPS) {
    if (lane == 0 && !early) {
      prefetch_tensor_map(&k_map);
      prefetch_tensor_map(&v_map);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int32_t* bt_row = a.paged ? a.block_table + static_cast<int64_t>(b) * a.bt_stride : nullptr;
    // physical page of tile (it * TPS + lane); fetched one stage ahead
    PageWindow pw{bt_row, t_begin, n_tiles, a.page_size, a.num_pages, lane, a.status, 0, 0, 0};
    if (a.paged) pw.init();
    int issued = early ? 1 : 0;  // (the early first stage)
    bool ok = true;
    const bool withhold =
        a.test_withhold != 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    for (int it = issued; it < n_iters; ++it) {
      const int s = it % STAGES;
      const int use = it / STAGES;
      int good = 1;
      if (lane == 0 && use > 0) good = mbar_wait(&empty_bar[s], (use - 1) & 1) ? 1 : 0;
      good = __shfl_sync(kFull, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      const int tiles_here = min(TPS, n_tiles - it * TPS);
      // page id of the tile this lane loads, picked in registers
      const int my_tile = F8 ? lane >> 1 : lane >> 2;
      int my_pg = 0;
#pragma unroll
      for (int i = 0; i < TPS; ++i) {
        const int pg = a.paged ? pw.get(it * TPS + i) : 0;
        if (my_tile == i) my_pg = pg;
      }
      constexpr int kBoxBytes = C::kTileBytes;  // K or V of one tile
      // test hook (DA_FLAG_TEST_WITHHOLD_COPY): block (0, 0, 0) of a two-pass
      // launch never fills its first stage, so its consumers' bounded wait
      // runs out and reports DA_STATUS_TIMEOUT
      if (!CM && it == 0 && withhold) {
        ++issued;
        continue;
      }
      uint8_t* stage = smem + s * C::kStageBytes;
      if (a.big_box) {
        // contiguous cache: one box of 16 TPS tokens per (K or V, d-half)
        // fills the whole stage region (the last stage may read tokens past
        // the chunk, which no consumer uses; past the cache the box is
        // zero-filled), so its byte count is always the full stage
        constexpr int kBigBoxes = F8 ? 2 : 4;
        if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(C::kStageBytes));
        __syncwarp();
        if (lane < kBigBoxes) {
          const bool is_v = F8 ? (lane & 1) != 0 : (lane & 2) != 0;
          const int half = F8 ? 0 : lane & 1;
          tma_load_4d(stage + (is_v ? C::kRegionBytes : 0) + half * C::kHalfStride,
                      is_v ? &v_map : &k_map, &full_bar[s], half * 64, kvh,
                      t_begin + it * TPS * kTileTokens, b, policy);
        }
        ++issued;
        __syncwarp();
        continue;
      }
      if (lane == 0)
        mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(tiles_here * 2 * kBoxBytes));
      __syncwarp();
      if (F8 && lane < tiles_here * 2) {
        // one TMA box per lane: all 128 FP8 values of 16 tokens (tile =
        // lane / 2, K or V from lane % 2) into the first half of the tile slot
        const int i = lane >> 1;
        const int tok = t_begin + (it * TPS + i) * kTileTokens;
        const int grp = a.paged ? my_pg : b;
        const int tin = a.paged ? tok % a.page_size : tok;
        const bool is_v = (lane & 1) != 0;
        uint8_t* dst = stage + (is_v ? C::kRegionBytes : 0) + i * C::kTileStride;
        tma_load_4d(dst, is_v ? &v_map : &k_map, &full_bar[s], 0, kvh, tin, grp, policy);
      }
      // one TMA box per lane (tile = lane / 4; K or V, d-half from lane % 4)
      if (!F8 && lane < tiles_here * 4) {
        const int i = lane >> 2;
        const int tok = t_begin + (it * TPS + i) * kTileTokens;
        const int grp = a.paged ? my_pg : b;
        const int tin = a.paged ? tok % a.page_size : tok;
        const int half = lane & 1;
        const bool is_v = (lane & 2) != 0;
        uint8_t* dst = stage + (is_v ? C::kRegionBytes : 0) + half * C::kHalfStride +
                       i * C::kTileStride;
        tma_load_4d(dst, is_v ? &v_map : &k_map, &full_bar[s], half * 64, kvh, tin, grp, policy);
      }
      ++issued;
      __syncwarp();
    }
    if (lane == 0) {
      if (!ok && a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
      // do not leave while copies are in flight: wait (bounded) for the last
      // stages this warp issued
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        if (!(withhold && it == 0)) mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1);
    }
    if constexpr (CM) {
      // the consumers' two cluster-barrier phases need every thread of the cluster
      if constexpr (C::kPushMerge) cluster_wait();
      else cluster_sync();
      cluster_sync();
    }
    return;
  }

  // ========================================================= consumer warps
  const int g4 = lane >> 2;  // fragment row group
  const int t4 = lane & 3;   // thread in group
  // Q^T as the B operand: rows r = 8*nt + g4, d pairs 2*t4 (+8) of k-step ks
  // (FP8: 4*t4 and 4*t4 + 2, the d permutation of the FP8 K fragments)
  auto q_row = [&](int r) -> const uint16_t* {
    if (r >= a.rows) return nullptr;
    const int t = r / a.group;
    const int g = r - t * a.group;
    return a.q + static_cast<int64_t>(b) * a.q_sb + static_cast<int64_t>(t) * a.q_st +
           static_cast<int64_t>(kvh * a.group + g) * a.q_sh;
  };
  constexpr int kQfSteps = C::kQSmem ? 1 : 8;  // fragments held in registers
  uint32_t qf[kQfSteps][NT][2];
  const uint32_t q_lane_addr =
      smem_addr(q_smem) + ((lane & 7) + 8 * (lane >> 4)) * 256;  // ldmatrix row of this lane
  if constexpr (C::kQSmem) {
    // stage the 16 rows once: item (row, 16-d step) per thread
    for (int idx = threadIdx.x; idx < C::kRows * 8; idx += 32 * TPS) {
      const int r = idx >> 3, ks = idx & 7;
      const uint16_t* qr = q_row(r);
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (qr != nullptr) {
        lo = make_uint4(load_u32(qr + 16 * ks), load_u32(qr + 16 * ks + 2),
                        load_u32(qr + 16 * ks + 4), load_u32(qr + 16 * ks + 6));
        hi = make_uint4(load_u32(qr + 16 * ks + 8), load_u32(qr + 16 * ks + 10),
                        load_u32(qr + 16 * ks + 12), load_u32(qr + 16 * ks + 14));
      }
      if constexpr (F8) {  // f16; chunk 2ks: d pairs 0,4,8,12; chunk 2ks+1: 2,6,10,14
        const uint4 c0 = make_uint4(bf16x2_to_f16x2(lo.x), bf16x2_to_f16x2(lo.z),
                                    bf16x2_to_f16x2(hi.x), bf16x2_to_f16x2(hi.z));
        const uint4 c1 = make_uint4(bf16x2_to_f16x2(lo.y), bf16x2_to_f16x2(lo.w),
                                    bf16x2_to_f16x2(hi.y), bf16x2_to_f16x2(hi.w));
        lo = c0;
        hi = c1;
      }
      *reinterpret_cast<uint4*>(q_smem + r * 256 + (((2 * ks) ^ (r & 7)) << 4)) = lo;
      *reinterpret_cast<uint4*>(q_smem + r * 256 + (((2 * ks + 1) ^ (r & 7)) << 4)) = hi;
    }
    named_barrier_sync(1, 32 * TPS);
  }
  int lim[NT][2];  // keys j < lim are visible to this thread's two rows
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint16_t* qrow = q_row(nt * 8 + g4);
    if constexpr (!C::kQSmem) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int d = ks * 16 + 2 * t4;
        qf[ks][nt][0] = qrow ? load_u32(qrow + d) : 0u;
        qf[ks][nt][1] = qrow ? load_u32(qrow + d + 8) : 0u;
        if constexpr (F8) {
          const int dp = ks * 16 + 4 * t4;
          qf[ks][nt][0] = qrow ? bf16x2_to_f16x2(load_u32(qrow + dp)) : 0u;
          qf[ks][nt][1] = qrow ? bf16x2_to_f16x2(load_u32(qrow + dp + 2)) : 0u;
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = nt * 8 + 2 * t4 + rr;
      int lm = t_end;
      if (a.causal && row < a.rows) lm = min(lm, L - a.q_len + 1 + row / a.group);
      lim[nt][rr] = lm;
    }
  }

  // per row: running max m, the sum l of the fp32 probabilities (the LSE)
  // and the sum lq of the probabilities as rounded into the P operand (it
  // normalises O, so the weights P.V applied sum to one exactly)
  float m[NT][2], l[NT][2], lq[NT][2], acc[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      m[nt][rr] = -INFINITY;
      l[nt][rr] = 0.f;
      lq[nt][rr] = 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
  }

  const uint32_t smem_base = smem_addr(smem);
  bool ok = true;
  for (int it = 0; it < n_iters; ++it) {
    const int s = it % STAGES;
    ok = __all_sync(kFull, mbar_wait(&full_bar[s], (it / STAGES) & 1)) != 0;
    if (!ok) break;
    const int tile = it * TPS + warp;
    if (tile < n_tiles) {
      const uint32_t kt = smem_base + s * C::kStageBytes + warp * C::kTileStride;
      const uint32_t vt = kt + C::kRegionBytes;
      const int tok0 = t_begin + tile * kTileTokens;
      // ---- S^T[16 keys x 8*NT rows] = K . Q^T
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[nt][i] = 0.f;
      // Q fragments of 16-d step ks: from registers, or (16 rows) one
      // ldmatrix.x4 from shared memory -- matrices (rows 0-7, chunk 2ks),
      // (rows 0-7, 2ks + 1), (rows 8-15, 2ks), (rows 8-15, 2ks + 1)
      auto q_frag = [&](int ks, uint32_t (&f)[NT][2]) {
        if constexpr (C::kQSmem) {
          uint32_t r4[4];
          const int row = (lane & 7) + 8 * (lane >> 4);
          ldsm_x4(q_lane_addr + (((2 * ks + ((lane >> 3) & 1)) ^ (row & 7)) << 4), r4);
          f[0][0] = r4[0];
          f[0][1] = r4[1];
          f[NT - 1][0] = r4[2];
          f[NT - 1][1] = r4[3];
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            f[nt][0] = qf[ks % kQfSteps][nt][0];
            f[nt][1] = qf[ks % kQfSteps][nt][1];
          }
        }
      };
      if constexpr (F8) {
        // FP8 K tile: 16 rows of 128 bytes, 16-byte chunk c of row t at
        // (c ^ (t & 7)); one ldmatrix.x4 covers two 16-d steps
        const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t r[4];
          const int chunk = 2 * kp + (lane >> 4);
          ldsm_x4(kt + key * 128 + ((chunk ^ (key & 7)) << 4), r);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // r[2h]: key g4, d 4t4..4t4+3 of the step; r[2h+1]: key g4 + 8
            uint32_t af[4];  // (each word split into its 16-bit halves, no shift)
            e4m3x4_to_f16x4(r[2 * h], af[0], af[2]);
            e4m3x4_to_f16x4(r[2 * h + 1], af[1], af[3]);
            uint32_t qb[NT][2];
            q_frag(2 * kp + h, qb);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16_16816(sc[nt], af, qb[nt][0], qb[nt][1]);
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t af[4];
          ldsm_x4(tile_addr(kt, (lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4),
                            C::kHalfStride),
                  af);
          uint32_t qb[NT][2];
          q_frag(ks, qb);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], af, qb[nt][0], qb[nt][1]);
        }
      }

      // ---- online softmax over this tile (base-2 domain)
      const int j0 = tok0 + g4;
      const int j1 = j0 + 8;
      float p[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const float x0 = j0 < lim[nt][rr] ? sc[nt][rr] * a.scale_log2 : -INFINITY;
          const float x1 = j1 < lim[nt][rr] ? sc[nt][2 + rr] * a.scale_log2 : -INFINITY;
          float mx = fmaxf(x0, x1);
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
          const float m_new = fmaxf(m[nt][rr], mx);
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          const float alpha = ex2(m[nt][rr] - m_use);
          const float p0 = ex2(x0 - m_use);
          const float p1 = ex2(x1 - m_use);
          l[nt][rr] = l[nt][rr] * alpha + (p0 + p1);
          if constexpr (!F8) lq[nt][rr] *= alpha;
          m[nt][rr] = m_new;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            acc[mt][nt][rr] *= alpha;
            acc[mt][nt][2 + rr] *= alpha;
          }
          p[nt][rr] = p0;
          p[nt][2 + rr] = p1;
        }
      }
      // P^T as the B operand of the value product: transpose each 8x8 bf16
      // block of the score fragment (keys x rows -> rows x keys)
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // key j0 (rows rr = 0 low, 1 high), then key j1
        const uint32_t k0 = F8 ? pack_f16x2(p[nt][0], p[nt][1]) : pack_bf16x2(p[nt][0], p[nt][1]);
        const uint32_t k1 = F8 ? pack_f16x2(p[nt][2], p[nt][3]) : pack_bf16x2(p[nt][2], p[nt][3]);
        // bf16 P: the sums of the rounded weights normalise O (the FP8 path's
        // f16 P rounds to 2^-11, well inside the bar: its fp32 sums serve)
        if constexpr (!F8) {
          lq[nt][0] += packed_lo(k0, false) + packed_lo(k1, false);
          lq[nt][1] += packed_hi(k0, false) + packed_hi(k1, false);
        }
        pb[nt][0] = movmatrix_trans(k0);
        pb[nt][1] = movmatrix_trans(k1);
      }

      // ---- keys past seq_len: their V slots may hold anything (NaN * 0 is
      // NaN), so zero those rows of the tile before using it
      if (tok0 + kTileTokens > L) {
        const int first = L - tok0;  // >= 1 since tok0 < t_end <= L
        uint8_t* vgen = smem + s * C::kStageBytes + C::kRegionBytes + warp * C::kTileStride;
        if constexpr (F8) {  // whole 128-byte rows
          for (int idx = lane; idx < (kTileTokens - first) * 8; idx += 32)
            *reinterpret_cast<uint4*>(vgen + (first + (idx >> 3)) * 128 + (idx & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        } else {
          for (int idx = lane; idx < (kTileTokens - first) * 16; idx += 32) {
            const int row = first + (idx >> 4);
            const int c = idx & 15;
            *reinterpret_cast<uint4*>(vgen + (c >> 3) * C::kHalfStride + (row << 7) + ((c & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // ---- O^T[128 d x 8*NT rows] += V^T . P^T
      if constexpr (F8) {
        // FP8 V tile, transposed b16 loads: r[i] bytes = (key 2t4: d 2g4,
        // 2g4+1), (key 2t4+1: d 2g4, 2g4+1) of matrix i; matrices (keys 0-7,
        // chunk c), (keys 8-15, chunk c), then chunk c + 1
        const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int mp = 0; mp < 4; ++mp) {
          uint32_t r[4];
          const int chunk = 2 * mp + (lane >> 4);
          ldsm_x4_trans(vt + key * 128 + ((chunk ^ (key & 7)) << 4), r);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // one byte permute per word: (key 2t4, key 2t4 + 1) of d 2g4 in the
            // low half, of d 2g4 + 1 in the high half; then both halves widen
            uint32_t af[4];  // d 2g4 / 2g4 + 1 of keys 2t4, +1, then of keys 8 + 2t4, +1
            e4m3x4_to_f16x4(__byte_perm(r[2 * h], 0, 0x3120), af[0], af[1]);
            e4m3x4_to_f16x4(__byte_perm(r[2 * h + 1], 0, 0x3120), af[2], af[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_f16_16816(acc[2 * mp + h][nt], af, pb[nt][0], pb[nt][1]);
          }
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t af[4];
          ldsm_x4_trans(tile_addr(vt, (lane & 7) + (lane >> 4) * 8, 2 * mt + ((lane >> 3) & 1),
                                  C::kHalfStride),
                        af);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], af, pb[nt][0], pb[nt][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
  }
  if (!ok && lane == 0 && a.status != nullptr)
    atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));

  // the main loop is done: the combine kernel may start launching
  if (threadIdx.x == 0) allow_dependent_launch();

  // ---- merge the consumer warps' (m, l, O) with the same recurrence
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float v = l[nt][rr];
      v += __shfl_xor_sync(kFull, v, 4);
      v += __shfl_xor_sync(kFull, v, 8);
      v += __shfl_xor_sync(kFull, v, 16);
      l[nt][rr] = v;
      if constexpr (F8) {
        lq[nt][rr] = v;
      } else {
        float w = lq[nt][rr];
        w += __shfl_xor_sync(kFull, w, 4);
        w += __shfl_xor_sync(kFull, w, 8);
        w += __shfl_xor_sync(kFull, w, 16);
        lq[nt][rr] = w;
      }
    }
  if (g4 == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = nt * 8 + 2 * t4 + rr;
        stat_m[warp * C::kRows + row] = m[nt][rr];
        stat_l[warp * C::kRows + row] = l[nt][rr];
        stat_q[warp * C::kRows + row] = lq[nt][rr];
      }
  }
  // every consumer warp is done with the stage ring (a warp may still be
  // reading any of its last stages until then) ...
  named_barrier_sync(1, 32 * TPS);
  // ... so each warp writes its O rows, scaled by its weight f = e^{m_w - M}
  // / sum_w lq_w e^{m_w - M} (the rounded-P sums normalise O; v_scale for FP8
  // caches), into it; after a second barrier the rows of the warps are summed.
  float* red = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = nt * 8 + 2 * t4 + rr;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < TPS; ++w) M = fmaxf(M, stat_m[w * C::kRows + row]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float Qs = 0.f;  // the rounded weights' sum over the warps
#pragma unroll
      for (int w = 0; w < TPS; ++w)
        Qs += stat_q[w * C::kRows + row] * ex2(stat_m[w * C::kRows + row] - Mu);
      const float f = (Qs > 0.f ? ex2(m[nt][rr] - Mu) / Qs : 0.f) * (F8 ? a.v_scale : 1.f);
      // accumulator rows g4 / g4 + 8 of output tile mt hold d = 16mt + g4 /
      // + 8 (bf16 path) or d = 16mt + 2g4 / + 1 (FP8 path)
      float* dst = red + (warp * C::kRows + row) * C::kRedStride + (F8 ? 2 * g4 : g4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        dst[mt * 16] = acc[mt][nt][rr] * f;
        dst[mt * 16 + (F8 ? 1 : 8)] = acc[mt][nt][2 + rr] * f;
      }
    }
  named_barrier_sync(1, 32 * TPS);

  // the row's natural-log LSE from the warps' fp32 sums
  auto row_lse = [&](int row) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < TPS; ++w) M = fmaxf(M, stat_m[w * C::kRows + row]);
    const float Mu = M == -INFINITY ? 0.f : M;
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < TPS; ++w)
      Ls += stat_l[w * C::kRows + row] * ex2(stat_m[w * C::kRows + row] - Mu);
    return Ls > 0.f ? (Mu + log2f(Ls)) * kLn2 : -INFINITY;
  };
  // the merged (row, d..d+3) of the CTA's output: the warps' scaled rows summed
  auto merged = [&](int row, int d) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < TPS; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(red + (w * C::kRows + row) * C::kRedStride + d);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    return v;
  };

  if constexpr (CM && C::kPushMerge) {
    // ---- cluster merge by push: every CTA writes each merged (row, 4 d)
    // unit and its row's LSE into the inbox of the unit's owner (CTA u mod S,
    // slot u / S); one cluster barrier publishes them, and each owner reduces
    // its units from its own shared memory (the same max / weighted-sum merge
    // as the combine kernel) -- no remote loads, no second barrier
    const int S = gridDim.x;  // cluster = all chunks of this (kv head, request), <= 16
    const int units = a.rows * 32;
    const int slots = (units + S - 1) / S;
    cluster_wait();  // every peer has started: its inbox may be written
    for (int u = threadIdx.x; u < units; u += 32 * TPS) {
      const int row = u >> 5;
      const int owner = u % S;
      const int slot = u / S;
      const uint32_t dv = smem_addr(inbox_v + split * slots + slot);
      const uint32_t dl = smem_addr(inbox_l + split * slots + slot);
      st_cluster_f32x4(map_to_rank(dv, owner), merged(row, (u & 31) * 4));
      st_cluster_f32(map_to_rank(dl, owner), row_lse(row));
    }
    cluster_sync();  // every push has landed
    for (int slot = threadIdx.x; slot < slots; slot += 32 * TPS) {
      const int u = slot * S + split;
      if (u >= units) break;
      const int row = u >> 5;
      const int d = (u & 31) * 4;
      float M = -INFINITY;
      for (int r = 0; r < S; ++r) M = fmaxf(M, inbox_l[r * slots + slot]);
      float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
      if (M != -INFINITY) {
        for (int r = 0; r < S; ++r) {  // peers in rank order
          const float w = ex2((inbox_l[r * slots + slot] - M) * kLog2e);
          const float4 x = inbox_v[r * slots + slot];
          W += w;
          acc4.x += w * x.x;
          acc4.y += w * x.y;
          acc4.z += w * x.z;
          acc4.w += w * x.w;
        }
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      const int t = row / a.group;
      const int h = kvh * a.group + (row - t * a.group);
      *reinterpret_cast<uint2*>(a.out + static_cast<int64_t>(b) * a.o_sb +
                                static_cast<int64_t>(t) * a.o_st +
                                static_cast<int64_t>(h) * a.o_sh + d) =
          make_uint2(pack_bf16x2(acc4.x * inv, acc4.y * inv),
                     pack_bf16x2(acc4.z * inv, acc4.w * inv));
      if (d == 0) {
        const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
        a.lse[prow] = W > 0.f ? M + logf(W) : -INFINITY;
      }
    }
    return;
  } else if constexpr (CM) {
    // ---- cluster merge: publish this CTA's (O, lse), then the CTAs of the
    // cluster reduce the rows over all CTAs through distributed shared
    // memory (the same max / weighted-sum merge as the combine kernel)
    float* xo = reinterpret_cast<float*>(smem + C::kXoOffset);
    for (int idx = threadIdx.x; idx < a.rows * 32; idx += 32 * TPS) {
      const int row = idx >> 5;
      const int d = (idx & 31) * 4;
      *reinterpret_cast<float4*>(xo + row * kHeadDim + d) = merged(row, d);
    }
    if (threadIdx.x < a.rows) xl[threadIdx.x] = row_lse(threadIdx.x);
    cluster_sync();  // every CTA's (O, lse) is visible cluster-wide

    const int S = gridDim.x;  // cluster = all chunks of this (kv head, request), <= 16
    const uint32_t xo_addr = smem_addr(xo);
    const uint32_t xl_addr = smem_addr(xl);
    // (row, 4 d) units interleaved over the CTAs of the cluster (unit u goes
    // to CTA u mod S), so every CTA reduces an equal share
    for (int u = threadIdx.x * S + split; u < a.rows * 32; u += 32 * TPS * S) {
      const int row = u >> 5;
      const int d = (u & 31) * 4;
      // every peer's LSE and the first 8 peers' output slices in one round
      // trip of independent remote loads, the other 8 in a second (a load
      // consumed right after it is issued would cost a round trip per peer)
      constexpr int kPeers = 16, kHalf = 8;
      float lr[kPeers];
      float4 x[kHalf];
#pragma unroll
      for (int r = 0; r < kPeers; ++r)
        lr[r] = r < S ? ld_cluster_f32(map_to_rank(xl_addr + row * 4, r)) : -INFINITY;
#pragma unroll
      for (int j = 0; j < kHalf; ++j)
        x[j] = j < S ? ld_cluster_f32x4(map_to_rank(xo_addr + (row * kHeadDim + d) * 4, j))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kPeers; ++r) M = fmaxf(M, lr[r]);
      float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
      float W = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int r0 = 0; r0 < kPeers; r0 += kHalf) {
          if (r0 > 0 && r0 < S) {
#pragma unroll
            for (int j = 0; j < kHalf; ++j)
              x[j] = r0 + j < S
                         ? ld_cluster_f32x4(map_to_rank(xo_addr + (row * kHeadDim + d) * 4, r0 + j))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int j = 0; j < kHalf; ++j) {
            if (r0 + j < S) {  // peers in rank order
              const float w = ex2((lr[r0 + j] - M) * kLog2e);
              W += w;
              acc4.x += w * x[j].x;
              acc4.y += w * x[j].y;
              acc4.z += w * x[j].z;
              acc4.w += w * x[j].w;
            }
          }
        }
      }
      const float inv = W > 0.f ? 1.f / W : 0.f;
      const int t = row / a.group;
      const int h = kvh * a.group + (row - t * a.group);
      *reinterpret_cast<uint2*>(a.out + static_cast<int64_t>(b) * a.o_sb +
                                static_cast<int64_t>(t) * a.o_st +
                                static_cast<int64_t>(h) * a.o_sh + d) =
          make_uint2(pack_bf16x2(acc4.x * inv, acc4.y * inv),
                     pack_bf16x2(acc4.z * inv, acc4.w * inv));
      if (d == 0) {
        const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
        a.lse[prow] = W > 0.f ? M + logf(W) : -INFINITY;
      }
    }
    cluster_sync();  // no CTA leaves while another may still read its smem
    return;
  } else {
    const bool direct = nsplit_b == 1;
    const int S = a.num_splits;
    for (int idx = threadIdx.x; idx < a.rows * 32; idx += 32 * TPS) {
      const int row = idx >> 5;
      const int d = (idx & 31) * 4;
      const float4 v = merged(row, d);
      const int t = row / a.group;
      const int h = kvh * a.group + (row - t * a.group);
      if (direct) {
        uint2 pk = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
        *reinterpret_cast<uint2*>(a.out + static_cast<int64_t>(b) * a.o_sb +
                                  static_cast<int64_t>(t) * a.o_st +
                                  static_cast<int64_t>(h) * a.o_sh + d) = pk;
      } else {
        const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
        const int64_t pidx = listed ? static_cast<int64_t>(blockIdx.x) * a.rows + row
                                    : prow * S + split;
        st_global_hint(a.part_o + pidx * kHeadDim + d, v, l2_evict_last_policy());
      }
    }
    if (threadIdx.x < a.rows) {
      const int row = threadIdx.x;
      const float lse = row_lse(row);
      const int t = row / a.group;
      const int h = kvh * a.group + (row - t * a.group);
      const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
      if (direct)
        a.lse[prow] = lse;
      else
        st_global_hint(a.part_lse + (listed ? static_cast<int64_t>(blockIdx.x) * a.rows + row
                                            : prow * S + split),
                       lse, l2_evict_last_policy());
    }
  }
}

// Pipeline shape: kTilesPerStage consumer warps (one 16-token tile each per
// stage; 2 tiles = 32 tokens = 16 KB of K+V per stage), kStages stages in
// flight (48 KB of shared memory, 4 CTAs per SM).  Chosen by GB300 sweeps over
// (stages, tiles): shapes with 2-3 CTAs per SM beat one large CTA per SM by
// 1.5-2x on ragged paged batches.  Overridable at build time for sweeps.
#ifndef DATTN_STAGES
#define DATTN_STAGES 3
#endif
#ifndef DATTN_TILES_PER_STAGE
#define DATTN_TILES_PER_STAGE 2
#endif
constexpr int kStages = DATTN_STAGES;
constexpr int kTilesPerStage = DATTN_TILES_PER_STAGE;
// the 16-row bf16 variant (overridable for sweeps)
#ifndef DATTN_NT2_STAGES
#define DATTN_NT2_STAGES DATTN_STAGES
#endif
#ifndef DATTN_NT2_TILES_PER_STAGE
#define DATTN_NT2_TILES_PER_STAGE DATTN_TILES_PER_STAGE
#endif
// FP8 caches: tiles are half the bytes; 4 stages (32 KB) leave room for 5-6
// CTAs per SM, which the latency-bound 16-row FP8 variant needs (GB300: 4
// stages 150 us, 6 stages 156 us on 32 requests x q_len 4; B = 1 unchanged)
#ifndef DATTN_F8_STAGES
#define DATTN_F8_STAGES 4
#endif
#ifndef DATTN_F8_TILES_PER_STAGE
#define DATTN_F8_TILES_PER_STAGE 2
#endif
// the 16-row FP8 variant takes three tiles (three consumer warps) per stage:
// 12 consumer warps per SM for its latency-bound loop (GB300: 152 -> 136 us
// on 32 requests x q_len 4; the 8-row variant stays at two, 1 % faster there)
#ifndef DATTN_F8_NT2_TILES_PER_STAGE
#define DATTN_F8_NT2_TILES_PER_STAGE 3
#endif
constexpr int kF8Stages = DATTN_F8_STAGES;
constexpr int kF8TilesPerStage = DATTN_F8_TILES_PER_STAGE;
// Grids of at most one CTA per SM (one short call, e.g. B = 1 at 4K tokens):
// occupancy no longer hides a CTA's copy latency, so each CTA keeps more
// bytes in flight -- 3 stages of 4 tiles (96 KB) and four consumer warps
// (GB300: 17 -> 15 us on B = 1, 32/8 heads, 4096 tokens).
constexpr int kDeepStages = 3;
constexpr int kDeepTilesPerStage = 4;

template <int NT, bool CM, bool F8, bool DP = false, bool LS = false>
struct Variant {
  static_assert(!(F8 && DP), "the deep shape serves bf16 caches");
  static constexpr int kSt = F8 ? kF8Stages : DP ? kDeepStages
                                           : NT == 2 ? DATTN_NT2_STAGES : kStages;
  static constexpr int kTps = F8 ? (NT == 2 ? DATTN_F8_NT2_TILES_PER_STAGE : kF8TilesPerStage)
                              : DP ? kDeepTilesPerStage
                                   : NT == 2 ? DATTN_NT2_TILES_PER_STAGE : kTilesPerStage;
  using C = SplitCfg<NT, kSt, kTps, F8>;
  static constexpr auto kernel = split_kv_kernel<NT, kSt, kTps, CM, F8, LS>;
};

constexpr int kMaxDev = 64;
constexpr int kMaxCluster = 16;  // non-portable cluster size limit
std::mutex g_attr_mu;
bool g_attr_done[2][2][2][2][2][kMaxDev];
// cached cudaOccupancyMaxActiveClusters per (NT, FP8, deep, cluster size, device); -1 unknown
int g_max_clusters[2][2][2][kMaxCluster + 1][kMaxDev];
bool g_max_clusters_init = false;
int g_sm_count[kMaxDev];

template <int NT, bool CM, bool F8, bool DP = false, bool LS = false>
cudaError_t ensure_attrs(int* dev_out = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  if (dev_out) *dev_out = dev;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (!g_attr_done[NT - 1][CM][F8][DP][LS][dev]) {
    e = cudaFuncSetAttribute(Variant<NT, CM, F8, DP, LS>::kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Variant<NT, CM, F8, DP, LS>::C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (CM) {
      e = cudaFuncSetAttribute(Variant<NT, CM, F8, DP, LS>::kernel,
                               cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    if (g_sm_count[dev] == 0) {
      e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
    }
    g_attr_done[NT - 1][CM][F8][DP][LS][dev] = true;
  }
  return cudaSuccess;
}

// True when a grid of `ctas` CTAs takes the deep shape: bf16 caches and at
// most one CTA per SM.
bool deep_grid(bool fp8, int64_t ctas) {
  if (fp8) return false;
  int dev = 0;
  if (ensure_attrs<1, false, false>(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  return ctas <= g_sm_count[dev];
}

template <int NT, bool CM, bool F8, bool DP, bool LS>
void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], const SplitArgs& a,
                 cudaStream_t st) {
  cfg = {};
  cfg.gridDim = LS ? dim3(static_cast<unsigned>(a.item_slots))
                   : dim3(a.num_splits, a.num_kv_heads, a.batch);
  cfg.blockDim = dim3(Variant<NT, CM, F8, DP, LS>::C::kThreads);
  cfg.dynamicSmemBytes = Variant<NT, CM, F8, DP, LS>::C::kSmemBytes;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (CM) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.num_splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
}

template <int NT, bool CM, bool F8, bool DP, bool LS>
cudaError_t launch_variant(const CUtensorMap& km, const CUtensorMap& vm, const SplitArgs& a,
                           cudaStream_t st) {
  cudaError_t e = ensure_attrs<NT, CM, F8, DP, LS>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  fill_config<NT, CM, F8, DP, LS>(cfg, attr, a, st);
  return cudaLaunchKernelEx(&cfg, Variant<NT, CM, F8, DP, LS>::kernel, km, vm, a);
}

// the cluster-merge, listed (device-planned) or grid-planned variant
template <int NT, bool CM, bool F8, bool DP = false>
cudaError_t launch_nt(const CUtensorMap& km, const CUtensorMap& vm, const SplitArgs& a,
                      cudaStream_t st) {
  if constexpr (CM) return launch_variant<NT, true, F8, DP, false>(km, vm, a, st);
  else if (a.items != nullptr) return launch_variant<NT, false, F8, DP, true>(km, vm, a, st);
  else return launch_variant<NT, false, F8, DP, false>(km, vm, a, st);
}

// Resident CTAs per SM of a variant (queried once per device, then cached).
int g_ctas_per_sm[2][2][kMaxDev];

template <int NT, bool F8>
int ctas_per_sm_nt() {
  int dev = 0;
  if (ensure_attrs<NT, false, F8>(&dev) != cudaSuccess) return 1;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_ctas_per_sm[NT - 1][F8][dev] > 0) return g_ctas_per_sm[NT - 1][F8][dev];
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Variant<NT, false, F8>::kernel,
                                                    Variant<NT, false, F8>::C::kThreads,
                                                    Variant<NT, false, F8>::C::kSmemBytes) !=
          cudaSuccess ||
      n < 1)
    return 1;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  g_ctas_per_sm[NT - 1][F8][dev] = n;
  return n;
}

// How many clusters of `splits` CTAs the device can hold at once.
template <int NT, bool F8, bool DP = false>
int max_active_clusters(int splits) {
  int dev = 0;
  if (ensure_attrs<NT, true, F8, DP>(&dev) != cudaSuccess) return 0;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (!g_max_clusters_init) {
      for (auto& x : g_max_clusters)
        for (auto& y : x)
          for (auto& z : y)
            for (auto& u : z)
              for (int& w : u) w = -1;
      g_max_clusters_init = true;
    }
    if (g_max_clusters[NT - 1][F8][DP][splits][dev] >= 0)
      return g_max_clusters[NT - 1][F8][DP][splits][dev];
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(splits), 1, 1);
  cfg.blockDim = dim3(Variant<NT, true, F8, DP>::C::kThreads);
  cfg.dynamicSmemBytes = Variant<NT, true, F8, DP>::C::kSmemBytes;
  cudaLaunchAttribute cl[1];
  cl[0].id = cudaLaunchAttributeClusterDimension;
  cl[0].val.clusterDim.x = static_cast<unsigned>(splits);
  cl[0].val.clusterDim.y = 1;
  cl[0].val.clusterDim.z = 1;
  cfg.attrs = cl;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, Variant<NT, true, F8, DP>::kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear the (non-sticky) error of a rejected query
    n = 0;
  }
  std::lock_guard<std::mutex> lk(g_attr_mu);
  g_max_clusters[NT - 1][F8][DP][splits][dev] = n;
  return n;
}

}  // namespace

cudaError_t launch_split(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                         bool cluster_merge, cudaStream_t stream) {
  if (a.rows > kMaxNarrowRows) return launch_wide(k_map, v_map, a, stream);
  if (a.kv_fp8) {
    if (a.rows <= 8)
      return cluster_merge ? launch_nt<1, true, true>(k_map, v_map, a, stream)
                           : launch_nt<1, false, true>(k_map, v_map, a, stream);
    return cluster_merge ? launch_nt<2, true, true>(k_map, v_map, a, stream)
                         : launch_nt<2, false, true>(k_map, v_map, a, stream);
  }
  const int64_t ctas = a.items != nullptr
                           ? a.item_slots
                           : static_cast<int64_t>(a.num_splits) * a.num_kv_heads * a.batch;
  if (deep_grid(false, ctas)) {
    if (a.rows <= 8)
      return cluster_merge ? launch_nt<1, true, false, true>(k_map, v_map, a, stream)
                           : launch_nt<1, false, false, true>(k_map, v_map, a, stream);
    return cluster_merge ? launch_nt<2, true, false, true>(k_map, v_map, a, stream)
                         : launch_nt<2, false, false, true>(k_map, v_map, a, stream);
  }
  if (a.rows <= 8)
    return cluster_merge ? launch_nt<1, true, false>(k_map, v_map, a, stream)
                         : launch_nt<1, false, false>(k_map, v_map, a, stream);
  return cluster_merge ? launch_nt<2, true, false>(k_map, v_map, a, stream)
                       : launch_nt<2, false, false>(k_map, v_map, a, stream);
}

int split_box_tokens(int rows, bool fp8, bool paged, int64_t ctas) {
  if (paged || rows > kMaxNarrowRows) return kTileTokens;  // pages, or the tcgen05 kernel
  if (fp8) return kTileTokens * (rows <= 8 ? Variant<1, false, true>::kTps
                                           : Variant<2, false, true>::kTps);
  return kTileTokens * (deep_grid(false, ctas) ? Variant<1, false, false, true>::kTps
                                               : Variant<1, false, false>::kTps);
}

int split_ctas_per_sm(int rows, bool fp8) {
  if (rows > kMaxNarrowRows) return wide_ctas_per_sm();
  if (fp8) return rows <= 8 ? ctas_per_sm_nt<1, true>() : ctas_per_sm_nt<2, true>();
  return rows <= 8 ? ctas_per_sm_nt<1, false>() : ctas_per_sm_nt<2, false>();
}

bool split_cluster_merge_fits(int rows, bool fp8, int num_splits, int64_t num_clusters) {
  if (num_splits < 2 || num_splits > kMaxCluster || num_clusters < 1 || rows > kMaxNarrowRows)
    return false;
  const bool deep = deep_grid(fp8, num_splits * num_clusters);  // as launch_split decides
  const int n = fp8 ? (rows <= 8 ? max_active_clusters<1, true>(num_splits)
                                 : max_active_clusters<2, true>(num_splits))
                    : deep ? (rows <= 8 ? max_active_clusters<1, false, true>(num_splits)
                                        : max_active_clusters<2, false, true>(num_splits))
                           : (rows <= 8 ? max_active_clusters<1, false>(num_splits)
                                        : max_active_clusters<2, false>(num_splits));
  // all clusters resident at once: in multi-wave grids the idle CTAs of short
  // requests hold slots (GB300 sweeps: 1.5-2x slower than partials + combine)
  return n >= num_clusters;
}

}  // namespace dattn
