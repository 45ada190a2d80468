// wide_kernel.cu -- split-KV decode attention for wide query groups (GQA group
// x speculative tokens = 17..128 query rows per KV head) on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// With many query rows per KV head the per-chunk work is a dense attention
// tile ("Capstone FlashAttention", §2.3 speculative verify of several draft
// tokens at once, §4.5; the CUTLASS split-KV post, §6: 4-token speculation):
// arithmetic intensity reaches G*q_len FLOP per KV byte, far beyond what the
// legacy warp-level MMA sustains at HBM rate.  One CTA per (chunk, kv head,
// request), like the narrow kernel, with three roles:
//   * warp 4 streams K/V stages with TMA (64 tokens = four 16-token page tiles
//     per stage, 128-byte swizzle, mbarrier byte counts), as in split_kernel.cu
//     but laid out as [2 d-halves][64 tokens][64 d] so that each half is a
//     canonical swizzled operand tile;
//   * one thread of warp 5 issues the MMAs: S = Q.K^T (M = 128 rows padded,
//     N = 64 keys, K = 128 d; A = Q and B = K both K-major in shared memory)
//     into one of two TMEM score buffers, and O += P.V (N = 128 d, K = 64 keys;
//     B = V read MN-major straight from the TMA tile) into a TMEM accumulator;
//     tcgen05.commit signals completion on mbarriers;
//   * warps 0-3 own one query row per thread (TMEM lane = row): they read the
//     score row, apply the masks, keep the running max / running sum of the
//     online softmax ("Capstone FlashAttention", §1.2), write P in bf16 to
//     shared memory, and rescale the O row in TMEM only when the running max
//     has grown by more than 2^8 since the last rescale (P stays <= 256, exact
//     in the deferred normalisation, §2.1).
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
#ifndef DATTN_WIDE_STAGES
#define DATTN_WIDE_STAGES 6
#endif
constexpr int kWStages = DATTN_WIDE_STAGES;  // K/V stages in flight
#ifndef DATTN_WIDE_PRODUCERS
#define DATTN_WIDE_PRODUCERS 4
#endif
// TMA copies issued by one warp are serialised (~130 cycles per box), so
// several producer warps share each stage's boxes.
constexpr int kWProducers = DATTN_WIDE_PRODUCERS;
constexpr int kWProducerWarp = 8;            // warps 0-7 softmax (2 groups), then TMA, then MMA
constexpr int kWMmaWarp = kWProducerWarp + kWProducers;
constexpr int kWThreads = 32 * (kWMmaWarp + 1);
constexpr int kWBoxes = 4 * kWTiles;         // per stage: tiles x {K, V} x 2 d-halves, 2 KB each
constexpr int kWBoxesPerWarp = (kWBoxes + kWProducers - 1) / kWProducers;
static_assert(kWProducers >= 1 && kWBoxesPerWarp <= 32, "boxes per producer warp");
constexpr int kWSoftmaxThreads = 256;
constexpr int kWHalf = kWTok * 128;          // [64 tokens][64 d] bf16 = 8 KB
constexpr int kWStageBytes = 4 * kWHalf;     // K halves, then V halves
constexpr int kWOffStage = 0;                // shared memory holds only the K/V ring
constexpr int kWOffBar = kWOffStage + kWStages * kWStageBytes;
constexpr int kWNumBars = 2 * kWStages + 2 + 2 + 2 + 2;  // full, empty, s_full, s_free, p_full, pv_done
constexpr int kWSmemBytes = 1024 + kWOffBar + kWNumBars * 8 + 16;
static_assert(kWSmemBytes <= 227 * 1024, "K/V ring exceeds shared memory");
// Tensor memory (512 columns x 128 lanes, lane = query row): fp32 scores
// S[g] at 64 g, fp32 outputs O[g] at 128 + 128 g, bf16 probabilities P[g]
// (64 keys packed in 32 columns) at 384 + 32 g, and the bf16 query rows Q
// (128 d packed in 64 columns) at 448 -- the A operands of both MMAs.
constexpr uint32_t kWTmemCols = 512;
constexpr uint32_t kWColO = 128;
constexpr uint32_t kWColP = 384;
constexpr uint32_t kWColQ = 448;
constexpr float kRescaleLog2 = 8.f;          // lazy rescale threshold (log2 units)

// Tile j of a chunk goes to softmax group g = j & 1 (warps 4g..4g+3): its
// scores land in TMEM buffer S[g], its probabilities in TMEM buffer P[g], and
// P.V accumulates into O[g]; the two groups alternate, so one group's softmax
// overlaps the other's, and their (m, l, O) merge exactly at the end.
__global__ void __launch_bounds__(kWThreads, 1)
    wide_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                const SplitArgs a) {
  constexpr uint32_t kFull = 0xffffffffu;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  grid_dependency_wait();

  int L = a.seq_lens[b];
  uint32_t bad = 0;
  if (L < 0 || L > a.max_seq_len) {
    bad |= DA_STATUS_SEQ_LEN;
    L = L < 0 ? 0 : a.max_seq_len;
  }
  if (a.causal && L > 0 && L < a.q_len) bad |= DA_STATUS_SHORT_CAUSAL;
  if (bad && a.status != nullptr && split == 0 && kvh == 0 && tid == 0)
    atomicOr(a.status, static_cast<int32_t>(bad));
  const int chunk = a.chunk_len;
  const int nsplit_b = L > 0 ? (L + chunk - 1) / chunk : 1;
  if (split >= nsplit_b) return;  // before any TMEM is allocated
  const int t_begin = split * chunk;
  const int t_end = min(L, t_begin + chunk);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTileTokens - 1) / kTileTokens : 0;
  const int n_iters = (n_tiles + kWTiles - 1) / kWTiles;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWOffBar);
  uint64_t* full_bar = bars;                   // [kWStages] TMA bytes landed
  uint64_t* empty_bar = bars + kWStages;       // [kWStages] stage consumed by the MMAs
  uint64_t* s_full = bars + 2 * kWStages;      // [2] scores in TMEM buffer
  uint64_t* s_free = s_full + 2;               // [2] score buffer read by softmax
  uint64_t* p_full = s_free + 2;               // [2] P buffer (and O rescale) ready for PV
  uint64_t* pv_done = p_full + 2;              // [2] PV of that P buffer finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kWNumBars);

  if (tid == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&full_bar[s], kWProducers);
      mbar_init(&empty_bar[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == kWMmaWarp) {
    tmem_alloc(tmem_slot, kWTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  // ============================================================ TMA producer
  if (warp >= kWProducerWarp && warp < kWMmaWarp) {
    const int pw_idx = warp - kWProducerWarp;
    if (lane == 0 && pw_idx == 0) {
      prefetch_tensor_map(&k_map);
      prefetch_tensor_map(&v_map);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int32_t* bt_row =
        a.paged ? a.block_table + static_cast<int64_t>(b) * a.bt_stride : nullptr;
    PageWindow pw{bt_row, t_begin, n_tiles, a.page_size, a.num_pages, lane, a.status, 0, 0, 0};
    if (a.paged) pw.init();
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < n_iters; ++it) {
      const int s = it % kWStages;
      const int use = it / kWStages;
      int good = 1;
      if (lane == 0 && use > 0) good = mbar_wait_spin(&empty_bar[s], (use - 1) & 1) ? 1 : 0;
      good = __shfl_sync(kFull, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      const int tiles_here = min(kWTiles, n_tiles - it * kWTiles);
      // this lane's box: bx = lane * kWProducers + pw_idx (tile bx / 4; K or
      // V and the d-half from bx % 4); page id of its tile picked in registers
      const int bx = lane * kWProducers + pw_idx;
      int my_pg = 0;
#pragma unroll
      for (int i = 0; i < kWTiles; ++i) {
        const int pg = a.paged ? pw.get(it * kWTiles + i) : 0;
        if ((bx >> 2) == i) my_pg = pg;
      }
      // boxes of this warp that hold data (tiles past the chunk end are skipped)
      int mine = 0;
      for (int c = pw_idx; c < tiles_here * 4; c += kWProducers) ++mine;
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(mine * 2048));
      __syncwarp();
      if (lane < kWBoxesPerWarp && bx < tiles_here * 4) {
        const int i = bx >> 2;
        const int tok = t_begin + (it * kWTiles + i) * kTileTokens;
        const int grp = a.paged ? my_pg : b;
        const int tin = a.paged ? tok % a.page_size : tok;
        const int half = bx & 1;
        const bool is_v = (bx & 2) != 0;
        uint8_t* dst = smem + kWOffStage + s * kWStageBytes + (is_v ? 2 * kWHalf : 0) +
                       half * kWHalf + i * 2048;
        tma_load_4d(dst, is_v ? &v_map : &k_map, &full_bar[s], half * 64, kvh, tin, grp, policy);
      }
      ++issued;
      __syncwarp();
    }
    if (lane == 0) {
      if (!ok && a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
      for (int it = max(0, issued - kWStages); it < issued; ++it)
        mbar_wait(&full_bar[it % kWStages], (it / kWStages) & 1);
    }
    return;
  }

  // ============================================================= MMA issuer
  // The whole warp runs this loop (all its values warp-uniform) and one
  // elected lane issues each MMA and commit.
  if (warp == kWMmaWarp) {
    named_barrier_sync(2, kWSoftmaxThreads + 32);  // Q is in tensor memory
    constexpr uint32_t kIdescQK = umma_idesc_bf16(kWRows, kWTok, false, false);
    constexpr uint32_t kIdescPV = umma_idesc_bf16(kWRows, kHeadDim, false, true);
    // B-operand descriptors of stage 0: other stages and K-steps differ only
    // in the start-address field (16-byte units, no carry below 256 KB), so
    // each MMA adds a constant to one of these. A (Q, P) is read from TMEM.
    const uint64_t k_desc0 = umma_smem_desc(smem_base + kWOffStage, 16, 1024);
    // B = V [64 keys][2 x 64 d], MN-major: d-halves 8 KB apart (LBO), 8-key
    // groups 1 KB apart (SBO), 16 keys = 2 KB per K-step
    const uint64_t v_desc0 = umma_smem_desc(smem_base + kWOffStage + 2 * kWHalf, kWHalf, 1024);
    // O += P_jj . V_jj, then release the stage and the P buffer
    auto issue_pv = [&](int jj) {
      tc_fence_after_sync();
      const uint32_t pa = tmem + kWColP + (jj & 1) * (kWTok / 2);
      const uint64_t vd = v_desc0 + static_cast<uint64_t>((jj % kWStages) * (kWStageBytes >> 4));
      const uint32_t d = tmem + kWColO + (jj & 1) * kHeadDim;
#pragma unroll
      for (int kk = 0; kk < kWTok / 16; ++kk)  // 16 keys = 8 P columns per K-step
        umma_bf16_ts_warp(d, pa + kk * 8, vd + kk * (2048 >> 4), kIdescPV,
                          (jj > 1 || kk > 0) ? 1u : 0u);
      umma_commit_warp(&pv_done[jj & 1]);
      umma_commit_warp(&empty_bar[jj % kWStages]);
    };
    // S_j = Q . K_j^T: 16 d per K-step (8 Q columns; K: d-half kk / 4, 32
    // bytes into its 128-byte swizzled rows)
    auto issue_qk = [&](int j) {
      tc_fence_after_sync();
      const uint64_t kd = k_desc0 + static_cast<uint64_t>((j % kWStages) * (kWStageBytes >> 4));
      const uint32_t d = tmem + (j & 1) * kWTok;
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        umma_bf16_ts_warp(d, tmem + kWColQ + kk * 8, kd + (((kk >> 2) * kWHalf + (kk & 3) * 32) >> 4),
                          kIdescQK, kk > 0 ? 1u : 0u);
      umma_commit_warp(&s_full[j & 1]);
    };
    // event loop: issue the next S = Q.K^T as soon as its stage has landed
    // and its score buffer is free, and the next O += P.V as soon as its
    // probabilities are ready -- neither waits on the other, so the two
    // softmax groups overlap. A phase seen complete by any lane is complete.
    bool ok = true;
    int next_qk = 0, next_pv = 0;
    unsigned long long idle_since = 0;
    while (next_pv < n_iters) {
      bool progress = false;
      if (next_qk < n_iters) {
        const int j = next_qk;
        const bool landed = mbar_test(&full_bar[j % kWStages], (j / kWStages) & 1);
        const bool s_ready = j < 2 || mbar_test(&s_free[j & 1], ((j >> 1) - 1) & 1);
        if (__any_sync(kFull, landed) && __any_sync(kFull, s_ready)) {
          issue_qk(j);
          ++next_qk;
          progress = true;
        }
      }
      if (next_pv < next_qk &&
          __any_sync(kFull, mbar_test(&p_full[next_pv & 1], (next_pv >> 1) & 1))) {
        issue_pv(next_pv);
        ++next_pv;
        progress = true;
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
    if (!ok && lane == 0 && a.status != nullptr)
      atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
    __syncwarp();
    named_barrier_sync(3, kWSoftmaxThreads + 32);  // softmax warps are done with TMEM
    tc_fence_after_sync();
    tmem_dealloc(tmem, kWTmemCols);
    return;
  }

  // ================================================ softmax groups (warps 0-7)
  const int grp = warp >> 2;       // softmax group: tiles j with j & 1 == grp
  const int r = tid & 127;         // query row = TMEM lane
  const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const uint32_t o_col = kWColO + grp * kHeadDim;
  int lim = 0;  // keys j < lim are visible to this row (0 for padding rows)
  if (r < a.rows) {
    const int t = r / a.group;
    lim = a.causal ? min(t_end, L - a.q_len + 1 + t) : t_end;
  }
  // ---- this thread's query row (zeros for padding rows) into TMEM lane r:
  // the A operand of S = Q.K^T, d pairs packed in 64 columns
  if (grp == 0) {
    const uint16_t* qrow = nullptr;
    if (r < a.rows) {
      const int t = r / a.group;
      const int g = r - t * a.group;
      qrow = a.q + static_cast<int64_t>(b) * a.q_sb + static_cast<int64_t>(t) * a.q_st +
             static_cast<int64_t>(kvh * a.group + g) * a.q_sh;
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float w[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = qrow ? *reinterpret_cast<const uint4*>(qrow + half * 64 + c * 8)
                             : make_uint4(0, 0, 0, 0);
        w[4 * c] = __uint_as_float(v.x);
        w[4 * c + 1] = __uint_as_float(v.y);
        w[4 * c + 2] = __uint_as_float(v.z);
        w[4 * c + 3] = __uint_as_float(v.w);
      }
      tmem_st32(lane_base + kWColQ + half * 32, w);
    }
    tmem_wait_st();
  }
  tc_fence_before_sync();
  named_barrier_sync(2, kWSoftmaxThreads + 32);

  float m_used = -INFINITY;  // reference max of P (log2 domain), raised lazily
  float l = 0.f;
  bool ok = true;
  int last_j = -1;
  for (int j = grp; j < n_iters; j += 2) {
    const int use = j >> 1;  // this group's use count of its buffers
    ok = __all_sync(kFull, mbar_wait(&s_full[grp], use & 1)) != 0;
    if (!ok) break;
    tc_fence_after_sync();
    float x[kWTok];
    {
      float lo[32], hi[32];
      tmem_ld32(lane_base + grp * kWTok, lo);
      tmem_ld32(lane_base + grp * kWTok + 32, hi);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = lo[i];
        x[32 + i] = hi[i];
      }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_free[grp]);

    // ---- scale, masks (only on tiles that reach past this row's limit) and
    // the lazy running max
    const int tok0 = t_begin + j * kWTok;
    float mt = -INFINITY;
    if (tok0 + kWTok <= lim) {
#pragma unroll
      for (int i = 0; i < kWTok; ++i) {
        x[i] *= a.scale_log2;
        mt = fmaxf(mt, x[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kWTok; ++i) {
        x[i] = tok0 + i < lim ? x[i] * a.scale_log2 : -INFINITY;
        mt = fmaxf(mt, x[i]);
      }
    }
    const bool raise = mt != -INFINITY && (m_used == -INFINITY || mt > m_used + kRescaleLog2);
    const float alpha = raise ? (m_used == -INFINITY ? 0.f : ex2(m_used - mt)) : 1.f;
    if (raise) m_used = mt;
    const float mref = m_used == -INFINITY ? 0.f : m_used;  // all masked so far: p = 0
    uint32_t pk[kWTok / 2];
    float psum = 0.f;
#pragma unroll
    for (int i = 0; i < kWTok; i += 2) {
      const float p0 = ex2(x[i] - mref);
      const float p1 = ex2(x[i + 1] - mref);
      psum += p0 + p1;
      pk[i / 2] = pack_bf16x2(p0, p1);
    }
    l = l * alpha + psum;

    // ---- this group's previous P.V (tile j - 2) must be done before its O
    // is rescaled and its P buffer rewritten
    if (use >= 1) {
      ok = __all_sync(kFull, mbar_wait(&pv_done[grp], (use - 1) & 1)) != 0;
      if (!ok) break;
      tc_fence_after_sync();
      if (__any_sync(kFull, raise && alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < kHeadDim / 32; ++c) {
          float o[32];
          tmem_ld32(lane_base + o_col + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_base + o_col + c * 32, o);
        }
        tmem_wait_st();
      }
    }
    // P row (64 bf16 packed in 32 columns) into TMEM: the A operand of P.V
    {
      float w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = __uint_as_float(pk[i]);
      tmem_st32(lane_base + kWColP + grp * (kWTok / 2), w);
    }
    // keys past the chunk end: their V rows may hold anything (NaN * 0 is
    // NaN), so zero them before the MMA reads the stage
    const int n_valid = min(kWTok, t_end - tok0);
    if (n_valid < kWTok) {
      uint8_t* vst = smem + kWOffStage + (j % kWStages) * kWStageBytes + 2 * kWHalf;
      for (int idx = r; idx < (kWTok - n_valid) * 16; idx += 128) {
        const int row = n_valid + (idx >> 4);
        const int c = idx & 15;  // 8 chunks per half, 2 halves
        *reinterpret_cast<uint4*>(vst + (c >> 3) * kWHalf + row * 128 + (c & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      }
    }
    if (n_valid < kWTok) fence_proxy_async_smem();
    tmem_wait_st();
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&p_full[grp]);
    last_j = j;
  }
  if (ok && last_j >= 0) {
    ok = __all_sync(kFull, mbar_wait(&pv_done[grp], (last_j >> 1) & 1)) != 0;
    tc_fence_after_sync();
  }
  if (!ok && lane == 0 && a.status != nullptr)
    atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));

  // ---- merge the two groups (same recurrence as the combine) and write
  // O / l (final bf16 row or fp32 partial) and the LSE; group g writes the
  // d-columns [64 g, 64 g + 64) of every row
  float* stat = reinterpret_cast<float*>(smem + kWOffStage);  // the K/V ring is idle now
  tc_fence_before_sync();
  named_barrier_sync(4, kWSoftmaxThreads);  // both groups' last P.V are done
  stat[grp * 256 + r] = m_used;
  stat[grp * 256 + 128 + r] = l;
  named_barrier_sync(4, kWSoftmaxThreads);
  tc_fence_after_sync();
  const float m0 = stat[r], l0 = stat[128 + r];
  const float m1 = stat[256 + r], l1 = stat[384 + r];
  const float M = fmaxf(m0, m1);
  const float Mu = M == -INFINITY ? 0.f : M;
  const float f0 = l0 > 0.f ? ex2(m0 - Mu) : 0.f;
  const float f1 = l1 > 0.f ? ex2(m1 - Mu) : 0.f;
  const float Lt = l0 * f0 + l1 * f1;
  const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
  const bool have0 = ok && n_iters > 0;  // O[0] / O[1] were written
  const bool have1 = ok && n_iters > 1;
  const bool direct = nsplit_b == 1;
  const int S = a.num_splits;
  const int t = r < a.rows ? r / a.group : 0;
  const int h = kvh * a.group + (r - t * a.group);
  const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int d0 = grp * 64 + c * 32;
    float o0[32], o1[32];
    if (have0) {
      tmem_ld32(lane_base + kWColO + d0, o0);
    }
    if (have1) {
      tmem_ld32(lane_base + kWColO + kHeadDim + d0, o1);
    }
    if (have0 || have1) tmem_wait_ld();
    if (r < a.rows) {
      float o[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        o[i] = ((have0 ? o0[i] * f0 : 0.f) + (have1 ? o1[i] * f1 : 0.f)) * inv;
      if (direct) {
        uint16_t* dst = a.out + static_cast<int64_t>(b) * a.o_sb + static_cast<int64_t>(t) * a.o_st +
                        static_cast<int64_t>(h) * a.o_sh + d0;
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          *reinterpret_cast<uint4*>(dst + i) =
              make_uint4(pack_bf16x2(o[i], o[i + 1]), pack_bf16x2(o[i + 2], o[i + 3]),
                         pack_bf16x2(o[i + 4], o[i + 5]), pack_bf16x2(o[i + 6], o[i + 7]));
      } else {
        float* dst = a.part_o + (prow * S + split) * kHeadDim + d0;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
      }
    }
  }
  if (grp == 0 && r < a.rows) {
    const float lse = Lt > 0.f ? (Mu + log2f(Lt)) * kLn2w : -INFINITY;
    if (direct)
      a.lse[prow] = lse;
    else
      a.part_lse[prow * S + split] = lse;
  }
  tc_fence_before_sync();
  named_barrier_sync(3, kWSoftmaxThreads + 32);  // the MMA warp releases TMEM after this
}

std::mutex g_wide_mu;
bool g_wide_attr[64];

cudaError_t ensure_wide_attrs() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_wide_mu);
  if (!g_wide_attr[dev]) {
    e = cudaFuncSetAttribute(wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmemBytes);
    if (e != cudaSuccess) return e;
    g_wide_attr[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_wide(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                        cudaStream_t stream) {
  cudaError_t e = ensure_wide_attrs();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_splits, a.num_kv_heads, a.batch);
  cfg.blockDim = dim3(kWThreads);
  cfg.dynamicSmemBytes = kWSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wide_kernel, k_map, v_map, a);
}

int wide_ctas_per_sm() {
  if (ensure_wide_attrs() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, wide_kernel, kWThreads, kWSmemBytes) !=
          cudaSuccess ||
      n < 1)
    return 1;
  return n;
}

}  // namespace dattn
