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

template <int NT, int STAGES, int TPS>
struct SplitCfg {
  static constexpr int kThreads = 32 * (TPS + 1);        // TPS consumer warps + 1 producer
  static constexpr int kHalfBytes = kTileTokens * 64 * 2;  // [16 tokens][64 d] bf16
  static constexpr int kTileBytes = 2 * kHalfBytes;        // one 16-token K (or V) tile
  static constexpr int kStageBytes = 2 * TPS * kTileBytes;  // TPS K tiles, then TPS V tiles
  static constexpr int kPipeBytes = STAGES * kStageBytes;
  static constexpr int kRows = 8 * NT;                     // padded query rows
  static constexpr int kRedStride = kHeadDim + 4;          // floats per row (bank spread)
  static constexpr int kRedBytes = TPS * kRows * kRedStride * 4;
  static_assert(kRedBytes <= kPipeBytes, "merge scratch must fit in the stage ring");
  static constexpr int kBarBytes = 2 * STAGES * 8;
  static constexpr int kStatBytes = 2 * TPS * kRows * 4;
  static constexpr int kSmemBytes = 1024 + kPipeBytes + kBarBytes + kStatBytes;
};

// Byte address of 16-byte chunk `chunk` (0..15, i.e. d = 8*chunk) of token row
// `tok` inside one tile: two 2048-byte halves [16 tokens][64 d], 128-byte rows,
// chunk index XOR-ed with (tok & 7) as the TMA 128-byte swizzle lays it out.
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int tok, int chunk) {
  return tile + ((chunk >> 3) << 11) + (tok << 7) + (((chunk & 7) ^ (tok & 7)) << 4);
}

__device__ __forceinline__ uint32_t load_u32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

template <int NT, int STAGES, int TPS>
__global__ void __launch_bounds__(SplitCfg<NT, STAGES, TPS>::kThreads)
    split_kv_kernel(const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const SplitArgs a) {
  using C = SplitCfg<NT, STAGES, TPS>;
  constexpr uint32_t kFull = 0xffffffffu;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // launched early behind the previous kernel of the stream: nothing that
  // kernel may write (q, caches, lengths, outputs) is touched before this
  grid_dependency_wait();

  // ---- this CTA's key range [t_begin, t_end)
  int L = a.seq_lens[b];
  uint32_t bad = 0;
  if (L < 0 || L > a.max_seq_len) {
    bad |= DA_STATUS_SEQ_LEN;
    L = L < 0 ? 0 : a.max_seq_len;
  }
  if (a.causal && L > 0 && L < a.q_len) bad |= DA_STATUS_SHORT_CAUSAL;
  if (bad && a.status != nullptr && split == 0 && kvh == 0 && threadIdx.x == 0)
    atomicOr(a.status, static_cast<int32_t>(bad));
  const int chunk = a.chunk_len;
  const int nsplit_b = L > 0 ? (L + chunk - 1) / chunk : 1;
  if (split >= nsplit_b) return;
  const int t_begin = split * chunk;
  const int t_end = min(L, t_begin + chunk);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTileTokens - 1) / kTileTokens : 0;
  const int n_iters = (n_tiles + TPS - 1) / TPS;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kPipeBytes);
  uint64_t* empty_bar = full_bar + STAGES;
  float* stat_m = reinterpret_cast<float*>(empty_bar + STAGES);
  float* stat_l = stat_m + TPS * C::kRows;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], TPS);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // =========================================================== producer warp
  if (warp == TPS) {
    if (lane == 0) {
      prefetch_tensor_map(&k_map);
      prefetch_tensor_map(&v_map);
    }
    const uint64_t policy = l2_evict_first_policy();
    const int32_t* bt_row = a.paged ? a.block_table + static_cast<int64_t>(b) * a.bt_stride : nullptr;
    // physical page of tile (it * TPS + lane); fetched one stage ahead
    auto page_of = [&](int it) -> int {
      const int tile = it * TPS + lane;
      if (!a.paged || lane >= TPS || tile >= n_tiles) return 0;
      const int tok = t_begin + tile * kTileTokens;
      int pg = __ldg(bt_row + tok / a.page_size);
      if (pg < 0 || pg >= a.num_pages) {
        if (a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(DA_STATUS_BAD_PAGE));
        pg = 0;
      }
      return pg;
    };
    int pg_next = n_iters > 0 ? page_of(0) : 0;
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < n_iters; ++it) {
      const int pg_cur = pg_next;
      if (it + 1 < n_iters) pg_next = page_of(it + 1);
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
      int pgs[TPS];
#pragma unroll
      for (int i = 0; i < TPS; ++i) pgs[i] = __shfl_sync(kFull, pg_cur, i);
      if (lane == 0) {
        mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(tiles_here * 2 * C::kTileBytes));
        uint8_t* stage = smem + s * C::kStageBytes;
        for (int i = 0; i < tiles_here; ++i) {
          const int tok = t_begin + (it * TPS + i) * kTileTokens;
          const int grp = a.paged ? pgs[i] : b;
          const int tin = a.paged ? tok % a.page_size : tok;
          uint8_t* kd = stage + i * C::kTileBytes;
          uint8_t* vd = stage + (TPS + i) * C::kTileBytes;
          tma_load_4d(kd, &k_map, &full_bar[s], 0, kvh, tin, grp, policy);
          tma_load_4d(kd + C::kHalfBytes, &k_map, &full_bar[s], 64, kvh, tin, grp, policy);
          tma_load_4d(vd, &v_map, &full_bar[s], 0, kvh, tin, grp, policy);
          tma_load_4d(vd + C::kHalfBytes, &v_map, &full_bar[s], 64, kvh, tin, grp, policy);
        }
      }
      ++issued;
      __syncwarp();
    }
    if (lane == 0) {
      if (!ok && a.status != nullptr) atomicOr(a.status, static_cast<int32_t>(DA_STATUS_TIMEOUT));
      // do not leave while copies are in flight: wait (bounded) for the last
      // stages this warp issued
      for (int it = max(0, issued - STAGES); it < issued; ++it)
        mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1);
    }
    return;
  }

  // ========================================================= consumer warps
  const int g4 = lane >> 2;  // fragment row group
  const int t4 = lane & 3;   // thread in group
  // Q^T as the B operand: rows r = 8*nt + g4, d pairs 2*t4 (+8) of k-step ks
  uint32_t qf[8][NT][2];
  int lim[NT][2];  // keys j < lim are visible to this thread's two rows
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = nt * 8 + g4;
    const uint16_t* qrow = nullptr;
    if (r < a.rows) {
      const int t = r / a.group;
      const int g = r - t * a.group;
      qrow = a.q + static_cast<int64_t>(b) * a.q_sb + static_cast<int64_t>(t) * a.q_st +
             static_cast<int64_t>(kvh * a.group + g) * a.q_sh;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d = ks * 16 + 2 * t4;
      qf[ks][nt][0] = qrow ? load_u32(qrow + d) : 0u;
      qf[ks][nt][1] = qrow ? load_u32(qrow + d + 8) : 0u;
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = nt * 8 + 2 * t4 + rr;
      int lm = t_end;
      if (a.causal && row < a.rows) lm = min(lm, L - a.q_len + 1 + row / a.group);
      lim[nt][rr] = lm;
    }
  }

  float m[NT][2], l[NT][2], acc[8][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      m[nt][rr] = -INFINITY;
      l[nt][rr] = 0.f;
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
      const uint32_t kt = smem_base + s * C::kStageBytes + warp * C::kTileBytes;
      const uint32_t vt = kt + TPS * C::kTileBytes;
      const int tok0 = t_begin + tile * kTileTokens;

      // ---- S^T[16 keys x 8*NT rows] = K . Q^T
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[nt][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t af[4];
        ldsm_x4(tile_addr(kt, (lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4)), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], af, qf[ks][nt][0], qf[ks][nt][1]);
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
        pb[nt][0] = movmatrix_trans(pack_bf16x2(p[nt][0], p[nt][1]));
        pb[nt][1] = movmatrix_trans(pack_bf16x2(p[nt][2], p[nt][3]));
      }

      // ---- keys past seq_len: their V slots may hold anything (NaN * 0 is
      // NaN), so zero those rows of the tile before using it
      if (tok0 + kTileTokens > L) {
        const int first = L - tok0;  // >= 1 since tok0 < t_end <= L
        uint8_t* vgen = smem + s * C::kStageBytes + (TPS + warp) * C::kTileBytes;
        for (int idx = lane; idx < (kTileTokens - first) * 16; idx += 32) {
          const int row = first + (idx >> 4);
          const int c = idx & 15;
          *reinterpret_cast<uint4*>(vgen + ((c >> 3) << 11) + (row << 7) + ((c & 7) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // ---- O^T[128 d x 8*NT rows] += V^T . P^T
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t af[4];
        ldsm_x4_trans(tile_addr(vt, (lane & 7) + (lane >> 4) * 8, 2 * mt + ((lane >> 3) & 1)), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[mt][nt], af, pb[nt][0], pb[nt][1]);
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
    }
  if (g4 == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = nt * 8 + 2 * t4 + rr;
        stat_m[warp * C::kRows + row] = m[nt][rr];
        stat_l[warp * C::kRows + row] = l[nt][rr];
      }
  }
  named_barrier_sync(1, 32 * TPS);

  float* red = reinterpret_cast<float*>(smem);  // the stage ring is idle now
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = nt * 8 + 2 * t4 + rr;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < TPS; ++w) M = fmaxf(M, stat_m[w * C::kRows + row]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float Ls = 0.f;
#pragma unroll
      for (int w = 0; w < TPS; ++w)
        Ls += stat_l[w * C::kRows + row] * ex2(stat_m[w * C::kRows + row] - Mu);
      const float f = Ls > 0.f ? ex2(m[nt][rr] - Mu) / Ls : 0.f;
      float* dst = red + (warp * C::kRows + row) * C::kRedStride + g4;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        dst[mt * 16] = acc[mt][nt][rr] * f;
        dst[mt * 16 + 8] = acc[mt][nt][2 + rr] * f;
      }
    }
  named_barrier_sync(1, 32 * TPS);

  const bool direct = nsplit_b == 1;
  const int S = a.num_splits;
  for (int idx = threadIdx.x; idx < a.rows * 32; idx += 32 * TPS) {
    const int row = idx >> 5;
    const int d = (idx & 31) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < TPS; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(red + (w * C::kRows + row) * C::kRedStride + d);
      v.x += x.x;
      v.y += x.y;
      v.z += x.z;
      v.w += x.w;
    }
    const int t = row / a.group;
    const int h = kvh * a.group + (row - t * a.group);
    if (direct) {
      uint2 pk = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      *reinterpret_cast<uint2*>(a.out + static_cast<int64_t>(b) * a.o_sb +
                                static_cast<int64_t>(t) * a.o_st +
                                static_cast<int64_t>(h) * a.o_sh + d) = pk;
    } else {
      const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
      *reinterpret_cast<float4*>(a.part_o + (prow * S + split) * kHeadDim + d) = v;
    }
  }
  if (threadIdx.x < a.rows) {
    const int row = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < TPS; ++w) M = fmaxf(M, stat_m[w * C::kRows + row]);
    const float Mu = M == -INFINITY ? 0.f : M;
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < TPS; ++w)
      Ls += stat_l[w * C::kRows + row] * ex2(stat_m[w * C::kRows + row] - Mu);
    const float lse = Ls > 0.f ? (Mu + log2f(Ls)) * kLn2 : -INFINITY;
    const int t = row / a.group;
    const int h = kvh * a.group + (row - t * a.group);
    const int64_t prow = (static_cast<int64_t>(b) * a.q_len + t) * a.num_q_heads + h;
    if (direct)
      a.lse[prow] = lse;
    else
      a.part_lse[prow * S + split] = lse;
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

template <int NT>
struct Variant {
  using C = SplitCfg<NT, kStages, kTilesPerStage>;
  static constexpr auto kernel = split_kv_kernel<NT, kStages, kTilesPerStage>;
};

std::mutex g_attr_mu;
bool g_attr_done[2][64];

template <int NT>
cudaError_t ensure_attrs() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (!g_attr_done[NT - 1][dev]) {
    e = cudaFuncSetAttribute(Variant<NT>::kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Variant<NT>::C::kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_done[NT - 1][dev] = true;
  }
  return cudaSuccess;
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap& km, const CUtensorMap& vm, const SplitArgs& a,
                      cudaStream_t st) {
  cudaError_t e = ensure_attrs<NT>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_splits, a.num_kv_heads, a.batch);
  cfg.blockDim = dim3(Variant<NT>::C::kThreads);
  cfg.dynamicSmemBytes = Variant<NT>::C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, Variant<NT>::kernel, km, vm, a);
}

template <int NT>
int ctas_per_sm_nt() {
  if (ensure_attrs<NT>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Variant<NT>::kernel, Variant<NT>::C::kThreads,
                                                    Variant<NT>::C::kSmemBytes) != cudaSuccess ||
      n < 1)
    return 1;
  return n;
}

}  // namespace

cudaError_t launch_split(const CUtensorMap& k_map, const CUtensorMap& v_map, const SplitArgs& a,
                         cudaStream_t stream) {
  if (a.rows <= 8) return launch_nt<1>(k_map, v_map, a, stream);
  return launch_nt<2>(k_map, v_map, a, stream);
}

int split_ctas_per_sm(int rows) { return rows <= 8 ? ctas_per_sm_nt<1>() : ctas_per_sm_nt<2>(); }

}  // namespace dattn
