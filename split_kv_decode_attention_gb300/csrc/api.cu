// api.cu -- the C ABI of libdecode_attn.so (declared in include/decode_attn.h):
// argument validation, the split planner, TMA tensor-map construction and the
// launches of the split and combine kernels.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "decode_attn.h"
#include "kernels.cuh"
#include "plan_rule.cuh"

namespace {

using dattn::kHeadDim;
using dattn::kTileTokens;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sm_count = 0;
  int major = 0;
  int minor = 0;
  bool valid = false;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

int current_device_info(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.valid) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return DA_ERR_NO_DEVICE;
    d.valid = true;
  }
  *out = d;
  return DA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

int rows_of(const decode_attn_params* p) {
  return (p->num_q_heads / p->num_kv_heads) * p->q_len;
}

bool kv_fp8(const decode_attn_params* p) { return (p->flags & DA_FLAG_KV_FP8_E4M3) != 0; }

// Shape checks shared by every entry point.
int check_shape(const decode_attn_params* p) {
  if (p == nullptr) return DA_ERR_NULL_POINTER;
  if (p->batch < 0 || p->batch > 65535 || p->q_len < 1 || p->num_q_heads < 1 ||
      p->num_kv_heads < 1 || p->num_kv_heads > 65535 || p->max_seq_len < 0 ||
      p->num_q_heads % p->num_kv_heads != 0 ||
      (p->flags & ~(DA_FLAG_TWO_PASS | DA_FLAG_KV_FP8_E4M3 | DA_FLAG_TEST_WITHHOLD_COPY)) != 0 ||
      !std::isfinite(p->scale))
    return DA_ERR_BAD_SHAPE;
  if (kv_fp8(p) && (!std::isfinite(p->k_scale) || !std::isfinite(p->v_scale)))
    return DA_ERR_BAD_SHAPE;
  if (p->head_dim != DECODE_ATTN_HEAD_DIM) return DA_ERR_HEAD_DIM;
  if (static_cast<int64_t>(p->num_q_heads / p->num_kv_heads) * p->q_len > DECODE_ATTN_MAX_ROWS)
    return DA_ERR_ROWS;
  return DA_OK;
}

int check_paged(const decode_attn_params* p, bool paged) {
  if (!paged) return DA_OK;
  if (p->page_size <= 0 || p->page_size % kTileTokens != 0) return DA_ERR_PAGE_SIZE;
  if (p->max_pages_per_seq < 1 || p->num_pages < 1 ||
      p->block_table_stride < p->max_pages_per_seq ||
      static_cast<int64_t>(p->max_seq_len) >
          static_cast<int64_t>(p->max_pages_per_seq) * p->page_size)
    return DA_ERR_BAD_SHAPE;
  return DA_OK;
}

int chunk_for_splits(const decode_attn_params* p, int32_t num_splits, int32_t* chunk,
                     int32_t* splits_eff) {
  return dattn::plan_chunk_for_splits(p->max_seq_len, num_splits, chunk, splits_eff)
             ? DA_OK
             : DA_ERR_SPLITS;
}

// The planner proper (the rule of plan_rule.cuh, shared with the device
// planner kernel): a function of the shape, the host lengths and the number
// of CTAs the split launch keeps resident at once (SMs x CTAs per SM).
int plan_for_slots(const decode_attn_params* p, const int32_t* host_seq_lens, int64_t slots,
                   int32_t* num_splits, int32_t* chunk_len) {
  dattn::PlanShape shape;
  shape.slots = slots;
  shape.batch = p->batch;
  shape.num_kv_heads = p->num_kv_heads;
  shape.rows = rows_of(p);
  shape.max_seq_len = p->max_seq_len;
  bool uniform = true;
  int64_t work_tokens = 0;
  auto clamped = [&](int32_t b) {
    return std::min<int64_t>(std::max(host_seq_lens[b], 0), p->max_seq_len);
  };
  if (host_seq_lens != nullptr) {
    for (int32_t b = 0; b < p->batch; ++b) {
      work_tokens += clamped(b);
      if (host_seq_lens[b] != host_seq_lens[0]) uniform = false;
    }
  }
  auto chunks_of = [&](int64_t c) {
    int64_t n = 0;
    for (int32_t b = 0; b < p->batch; ++b) {
      const int64_t Lb = clamped(b);
      n += Lb > 0 ? ceil_div64(Lb, c) : 1;
    }
    return n * p->num_kv_heads;
  };
  const int64_t splits = dattn::plan_splits(shape, uniform, work_tokens, chunks_of);
  int32_t chunk = 0, eff = 0;
  const int rc = chunk_for_splits(p, static_cast<int32_t>(splits), &chunk, &eff);
  if (rc != DA_OK) return rc;
  *num_splits = eff;
  *chunk_len = chunk;
  return DA_OK;
}

// The planner on the current device: its SM count times the split launch's
// resident CTAs per SM for this shape (occupancy of the kernel it will run).
int plan_impl(const decode_attn_params* p, const int32_t* host_seq_lens, int32_t* num_splits,
              int32_t* chunk_len) {
  DeviceInfo di;
  const int rc = current_device_info(&di);
  if (rc != DA_OK) return rc;
  const int64_t slots =
      static_cast<int64_t>(di.sm_count) * dattn::split_ctas_per_sm(rows_of(p), kv_fp8(p));
  return plan_for_slots(p, host_seq_lens, slots, num_splits, chunk_len);
}

// box_tokens: token rows per box (16; a whole stage for contiguous caches
// on the warp-MMA kernel)
// Encoded tensor maps of recent calls: a serving loop passes the same caches
// every step, so the map of (base, layout, box) is encoded once and reused.
struct MapKey {
  const void* base;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box;
  int fp8;
  bool operator==(const MapKey& o) const {
    return base == o.base && std::memcmp(dims, o.dims, sizeof(dims)) == 0 &&
           std::memcmp(strides, o.strides, sizeof(strides)) == 0 && box == o.box && fp8 == o.fp8;
  }
};
constexpr int kMapCacheSize = 16;
std::mutex g_map_mu;
struct {
  MapKey key;
  CUtensorMap map;
  bool valid;
} g_map_cache[kMapCacheSize];
int g_map_next = 0;

int make_kv_map(CUtensorMap* map, const void* base, const decode_attn_params* p, bool paged,
                int box_tokens) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return DA_ERR_CUDA;
  // dims, innermost first: d (128), kv head, token-in-group, group
  //   paged: group = physical page, token-in-group = slot in page
  //   contiguous: group = request, token-in-group = token position
  const cuuint64_t dims[4] = {
      static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(p->num_kv_heads),
      static_cast<cuuint64_t>(paged ? p->page_size : std::max(p->max_seq_len, 1)),
      static_cast<cuuint64_t>(paged ? p->num_pages : std::max(p->batch, 1))};
  // element bytes: 2 (bf16) or 1 (FP8); a box row is 128 bytes either way
  // (the 128-byte swizzle span): 64 bf16 (two boxes per 16-token tile) or all
  // 128 FP8 values of a token (one box)
  const cuuint64_t eb = kv_fp8(p) ? 1 : 2;
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(p->kv_stride_head) * eb,
                                 static_cast<cuuint64_t>(p->kv_stride_token) * eb,
                                 static_cast<cuuint64_t>(p->kv_stride_page) * eb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), 1,
                             static_cast<cuuint32_t>(box_tokens), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = base;
  std::memcpy(key.dims, dims, sizeof(dims));
  std::memcpy(key.strides, strides, sizeof(strides));
  key.box = box[2];
  key.fp8 = kv_fp8(p) ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (auto& e : g_map_cache)
      if (e.valid && e.key == key) {
        *map = e.map;
        return DA_OK;
      }
  }
  CUresult r = enc(map, kv_fp8(p) ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return DA_ERR_ALIGNMENT;
  std::lock_guard<std::mutex> lk(g_map_mu);
  auto& e = g_map_cache[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCacheSize;
  e.key = key;
  e.map = *map;
  e.valid = true;
  return DA_OK;
}

bool stride_ok(int64_t s) { return s > 0 && s % 8 == 0 && s * 2 < (1LL << 40); }

// FP8 caches: strides in bytes, multiples of 16 (the TMA stride rule)
bool kv_stride_ok(const decode_attn_params* p, int64_t s) {
  return kv_fp8(p) ? (s > 0 && s % 16 == 0 && s < (1LL << 40)) : stride_ok(s);
}

// The split pass merges through thread-block clusters (no partials, no
// combine) when allowed by the flags and when the splits_eff CTAs of every
// (request, kv head) form a supported cluster and all clusters fit at once.
bool use_cluster_merge(const decode_attn_params* p, int32_t splits_eff) {
  if ((p->flags & DA_FLAG_TWO_PASS) != 0 || splits_eff < 2 || p->batch < 1) return false;
  return dattn::split_cluster_merge_fits(rows_of(p), kv_fp8(p), splits_eff,
                                         static_cast<int64_t>(p->batch) * p->num_kv_heads);
}

// ---- device-planned calls
// decode_attn(num_splits <= 0) with two or more requests plans on the device:
// the lengths may exist only in device memory (and change between replays of
// a captured graph), so a planner kernel applies the planner's rule to them
// and writes a work list; the split launch has one CTA per item slot of a
// host-sized capacity and the partials are indexed by item, so nothing the
// host sizes depends on the lengths.  A single request keeps the host plan
// (its only length is bounded by max_seq_len), with the cluster merge.
// Capacity: at most B * Hkv items of one chunk each, plus about 2 x
// kRaggedWaves waves of resident CTAs (the rule aims at kRaggedWaves; its
// rounding can double that); the planner grows the chunk if a plan would
// exceed it.
constexpr int64_t kListWaveSlack = 2 * dattn::kRaggedWaves;

struct ListLayout {
  size_t plan, pre, items, part_o, part_lse, total;
  int64_t cap, slots;
};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool device_planned(const decode_attn_params* p, int32_t num_splits) {
  // (the tcgen05 kernel walks its items persistently, from tables of at most
  // kWideMaxPlannedBatch requests)
  return num_splits <= 0 && p->batch >= 2 && p->max_seq_len <= (1 << 30) &&
         (rows_of(p) <= dattn::kMaxNarrowRows || p->batch <= dattn::kWideMaxPlannedBatch);
}

// Resident CTAs of the split launch for this shape on the current device.
int split_slots(const decode_attn_params* p, int64_t* slots) {
  DeviceInfo di;
  const int rc = current_device_info(&di);
  if (rc != DA_OK) return rc;
  *slots = static_cast<int64_t>(di.sm_count) * dattn::split_ctas_per_sm(rows_of(p), kv_fp8(p));
  return DA_OK;
}

// Workspace of a device-planned call (offsets 256-byte aligned): plan[4],
// pre[B + 1], items[cap] (int4), partial outputs [cap, rows, D] and partial
// LSEs [cap, rows] (fp32).
int list_layout(const decode_attn_params* p, ListLayout* l) {
  int rc = split_slots(p, &l->slots);
  if (rc != DA_OK) return rc;
  l->cap = static_cast<int64_t>(p->batch) * p->num_kv_heads + kListWaveSlack * l->slots;
  if (l->cap > 0x7fffffff) return DA_ERR_BAD_SHAPE;
  const size_t rows = static_cast<size_t>(rows_of(p));
  const size_t cap = static_cast<size_t>(l->cap);
  size_t off = 0;
  l->plan = off;
  off = round256(off + 16);
  l->pre = off;
  off = round256(off + (static_cast<size_t>(p->batch) + 1) * 4);
  l->items = off;
  off = round256(off + cap * 16);
  l->part_o = off;
  off = round256(off + cap * rows * kHeadDim * 4);
  l->part_lse = off;
  l->total = off + cap * rows * 4;
  return DA_OK;
}

// Arguments of the planner kernel for a device-planned call whose workspace
// starts at w.
dattn::PlanArgs plan_args(const decode_attn_params* p, const int32_t* seq_lens, int32_t* status,
                          uint8_t* w, const ListLayout& lay) {
  dattn::PlanArgs pa;
  std::memset(&pa, 0, sizeof(pa));
  pa.seq_lens = seq_lens;
  pa.status = status;
  pa.plan = reinterpret_cast<int32_t*>(w + lay.plan);
  pa.pre = reinterpret_cast<int32_t*>(w + lay.pre);
  pa.items = reinterpret_cast<int4*>(w + lay.items);
  pa.slots = lay.slots;
  pa.cap = lay.cap;
  pa.batch = p->batch;
  pa.num_kv_heads = p->num_kv_heads;
  pa.rows = rows_of(p);
  pa.max_seq_len = p->max_seq_len;
  pa.q_len = p->q_len;
  pa.causal = p->causal ? 1 : 0;
  return pa;
}

}  // namespace

extern "C" {

void decode_attn_params_init(decode_attn_params* p, int32_t batch, int32_t q_len,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t page_size, int32_t max_pages_per_seq, int32_t num_pages,
                             int32_t max_seq_len, int32_t causal) {
  if (p == nullptr) return;
  std::memset(p, 0, sizeof(*p));
  p->batch = batch;
  p->q_len = q_len;
  p->num_q_heads = num_q_heads;
  p->num_kv_heads = num_kv_heads;
  p->head_dim = head_dim;
  p->page_size = page_size;
  p->max_pages_per_seq = max_pages_per_seq;
  p->num_pages = num_pages;
  p->max_seq_len = max_seq_len;
  p->causal = causal;
  p->scale = head_dim > 0 ? 1.0f / std::sqrt(static_cast<float>(head_dim)) : 0.f;
  p->q_stride_head = head_dim;
  p->q_stride_token = static_cast<int64_t>(num_q_heads) * head_dim;
  p->q_stride_batch = p->q_stride_token * q_len;
  p->o_stride_head = p->q_stride_head;
  p->o_stride_token = p->q_stride_token;
  p->o_stride_batch = p->q_stride_batch;
  p->kv_stride_head = head_dim;
  p->kv_stride_token = static_cast<int64_t>(num_kv_heads) * head_dim;
  p->kv_stride_page = p->kv_stride_token * (page_size > 0 ? page_size : max_seq_len);
  p->block_table_stride = max_pages_per_seq;
  p->k_scale = 1.f;
  p->v_scale = 1.f;
}

int decode_attn_plan(const decode_attn_params* p, const int32_t* host_seq_lens,
                     int32_t* num_splits, int32_t* chunk_len) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (num_splits == nullptr || chunk_len == nullptr) return DA_ERR_NULL_POINTER;
  return plan_impl(p, host_seq_lens, num_splits, chunk_len);
}

int decode_attn_plan_slots(const decode_attn_params* p, const int32_t* host_seq_lens,
                           int64_t resident_ctas, int32_t* num_splits, int32_t* chunk_len) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (num_splits == nullptr || chunk_len == nullptr) return DA_ERR_NULL_POINTER;
  if (resident_ctas < 1 || resident_ctas > (int64_t{1} << 31)) return DA_ERR_BAD_SHAPE;
  return plan_for_slots(p, host_seq_lens, resident_ctas, num_splits, chunk_len);
}

int decode_attn_chunk_len(const decode_attn_params* p, int32_t num_splits, int32_t* chunk_len) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (chunk_len == nullptr) return DA_ERR_NULL_POINTER;
  int32_t eff = 0;
  return chunk_for_splits(p, num_splits, chunk_len, &eff);
}

int decode_attn_workspace_bytes(const decode_attn_params* p, int32_t num_splits, size_t* bytes) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (bytes == nullptr) return DA_ERR_NULL_POINTER;
  if (device_planned(p, num_splits)) {
    ListLayout l;
    rc = list_layout(p, &l);
    if (rc != DA_OK) return rc;
    *bytes = l.total;
    return DA_OK;
  }
  int32_t chunk = 0, eff = 0;
  if (num_splits <= 0) {  // one request (or none): the host plan
    rc = plan_impl(p, nullptr, &num_splits, &chunk);
    if (rc != DA_OK) return rc;
  }
  rc = chunk_for_splits(p, num_splits, &chunk, &eff);
  if (rc != DA_OK) return rc;
  if (eff <= 1) {
    *bytes = 0;
    return DA_OK;
  }
  const size_t rows = static_cast<size_t>(p->batch) * p->q_len * p->num_q_heads;
  *bytes = rows * static_cast<size_t>(eff) * (kHeadDim + 1) * sizeof(float);
  return DA_OK;
}

int decode_attn_launch_count(const decode_attn_params* p, int32_t num_splits) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (p->batch == 0) return 0;
  if (device_planned(p, num_splits)) return 3;  // planner, split, combine
  int32_t chunk = 0, eff = 0;
  if (num_splits <= 0) {
    rc = plan_impl(p, nullptr, &num_splits, &chunk);
    if (rc != DA_OK) return rc;
  }
  rc = chunk_for_splits(p, num_splits, &chunk, &eff);
  if (rc != DA_OK) return rc;
  return eff > 1 && !use_cluster_merge(p, eff) ? 2 : 1;
}

}  // extern "C"

namespace {

// The whole path (run_combine) or the split pass alone.
int run_decode(const decode_attn_params* p, const void* q, const void* k_cache,
               const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
               void* out, float* lse, int32_t num_splits, void* workspace,
               size_t workspace_bytes, int32_t* status, void* stream, bool run_combine) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  const bool paged = block_table != nullptr;
  rc = check_paged(p, paged);
  if (rc != DA_OK) return rc;
  if (p->batch == 0) return DA_OK;
  // with max_seq_len == 0 no key is ever read: the caches may be empty
  const bool no_keys = p->max_seq_len == 0;
  if (q == nullptr || (!no_keys && (k_cache == nullptr || v_cache == nullptr)) ||
      seq_lens == nullptr || out == nullptr || lse == nullptr)
    return DA_ERR_NULL_POINTER;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0 ||
      (paged && (reinterpret_cast<uintptr_t>(block_table) & 3u) != 0))
    return DA_ERR_ALIGNMENT;
  if (!stride_ok(p->q_stride_batch) || !stride_ok(p->q_stride_token) ||
      !stride_ok(p->q_stride_head) || !stride_ok(p->o_stride_batch) ||
      !stride_ok(p->o_stride_token) || !stride_ok(p->o_stride_head) ||
      (!no_keys && (!kv_stride_ok(p, p->kv_stride_page) || !kv_stride_ok(p, p->kv_stride_token) ||
                    !kv_stride_ok(p, p->kv_stride_head))))
    return DA_ERR_ALIGNMENT;

  DeviceInfo di;
  rc = current_device_info(&di);
  if (rc != DA_OK) return rc;
  if (di.major * 10 + di.minor < 100) return DA_ERR_NO_DEVICE;

  const bool listed = device_planned(p, num_splits);
  ListLayout lay;
  int32_t chunk = 0, eff = 0;
  bool cluster_merge = false;
  if (listed) {
    rc = list_layout(p, &lay);
    if (rc != DA_OK) return rc;
    if (workspace == nullptr || workspace_bytes < lay.total || !aligned16(workspace))
      return DA_ERR_WORKSPACE;
  } else {
    if (num_splits <= 0) {
      rc = plan_impl(p, nullptr, &num_splits, &chunk);
      if (rc != DA_OK) return rc;
    }
    rc = chunk_for_splits(p, num_splits, &chunk, &eff);
    if (rc != DA_OK) return rc;
    cluster_merge = use_cluster_merge(p, eff);
    size_t need = 0;
    decode_attn_workspace_bytes(p, num_splits, &need);
    if (!cluster_merge && need > 0 &&
        (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
      return DA_ERR_WORKSPACE;
  }

  // the split launch's grid (it picks the pipeline shape, and with it the box
  // height for contiguous caches)
  const int64_t ctas =
      listed ? lay.cap : static_cast<int64_t>(eff) * p->num_kv_heads * p->batch;
  const int box_tokens = dattn::split_box_tokens(rows_of(p), kv_fp8(p), paged, ctas);
  CUtensorMap kmap, vmap;
  std::memset(&kmap, 0, sizeof(kmap));
  std::memset(&vmap, 0, sizeof(vmap));
  if (!no_keys) {
    rc = make_kv_map(&kmap, k_cache, p, paged, box_tokens);
    if (rc != DA_OK) return rc;
    rc = make_kv_map(&vmap, v_cache, p, paged, box_tokens);
    if (rc != DA_OK) return rc;
  }

  dattn::SplitArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const uint16_t*>(q);
  a.q_sb = p->q_stride_batch;
  a.q_st = p->q_stride_token;
  a.q_sh = p->q_stride_head;
  a.out = static_cast<uint16_t*>(out);
  a.o_sb = p->o_stride_batch;
  a.o_st = p->o_stride_token;
  a.o_sh = p->o_stride_head;
  a.lse = lse;
  const size_t rows_total = static_cast<size_t>(p->batch) * p->q_len * p->num_q_heads;
  a.part_o = eff > 1 && !cluster_merge ? static_cast<float*>(workspace) : nullptr;
  a.part_lse = a.part_o != nullptr ? a.part_o + rows_total * eff * kHeadDim : nullptr;
  a.block_table = block_table;
  a.bt_stride = p->block_table_stride;
  a.seq_lens = seq_lens;
  a.status = status;
  a.batch = p->batch;
  a.q_len = p->q_len;
  a.num_q_heads = p->num_q_heads;
  a.num_kv_heads = p->num_kv_heads;
  a.group = p->num_q_heads / p->num_kv_heads;
  a.rows = rows_of(p);
  a.page_size = paged ? p->page_size : 0;
  a.num_pages = paged ? p->num_pages : 0;
  a.paged = paged ? 1 : 0;
  a.max_seq_len = p->max_seq_len;
  a.chunk_len = chunk;
  a.num_splits = eff;
  a.causal = p->causal ? 1 : 0;
  a.scale_log2 = p->scale * (kv_fp8(p) ? p->k_scale : 1.f) * 1.4426950408889634f;
  a.kv_fp8 = kv_fp8(p) ? 1 : 0;
  a.test_withhold = (p->flags & DA_FLAG_TEST_WITHHOLD_COPY) != 0 ? 1 : 0;
  a.v_scale = kv_fp8(p) ? p->v_scale : 1.f;
  // (no keys: no tensor map was encoded and no copy may be issued)
  a.big_box = box_tokens > kTileTokens && !no_keys ? 1 : 0;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  if (listed) {
    // the planner writes the plan, prefixes and items; the split launch has
    // one CTA per item slot and stores partials by item
    a.plan = reinterpret_cast<const int32_t*>(w + lay.plan);
    a.pre = reinterpret_cast<const int32_t*>(w + lay.pre);
    a.items = reinterpret_cast<const int4*>(w + lay.items);
    a.item_slots = static_cast<int>(lay.cap);
    a.part_o = reinterpret_cast<float*>(w + lay.part_o);
    a.part_lse = reinterpret_cast<float*>(w + lay.part_lse);
    a.chunk_len = 0;
    a.num_splits = 1;
    if (dattn::launch_plan(plan_args(p, seq_lens, status, w, lay), st) != cudaSuccess)
      return DA_ERR_CUDA;
  }
  if (dattn::launch_split(kmap, vmap, a, cluster_merge, st) != cudaSuccess) return DA_ERR_CUDA;
  if (run_combine && (listed || (eff > 1 && !cluster_merge))) {
    dattn::CombineArgs c = {};
    c.plan = a.plan;
    c.pre = a.pre;
    c.num_kv_heads = p->num_kv_heads;
    c.part_o = a.part_o;
    c.part_lse = a.part_lse;
    c.seq_lens = seq_lens;
    c.out = a.out;
    c.o_sb = a.o_sb;
    c.o_st = a.o_st;
    c.o_sh = a.o_sh;
    c.lse = lse;
    c.batch = p->batch;
    c.q_len = p->q_len;
    c.num_q_heads = p->num_q_heads;
    c.max_seq_len = p->max_seq_len;
    c.chunk_len = chunk;
    c.num_splits = eff;
    if (dattn::launch_combine(c, st) != cudaSuccess) return DA_ERR_CUDA;
  }
  return DA_OK;
}

}  // namespace

extern "C" {

int decode_attn(const decode_attn_params* p, const void* q, const void* k_cache,
                const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                void* out, float* lse, int32_t num_splits, void* workspace,
                size_t workspace_bytes, int32_t* status, void* stream) {
  return run_decode(p, q, k_cache, v_cache, block_table, seq_lens, out, lse, num_splits,
                    workspace, workspace_bytes, status, stream, true);
}

int decode_attn_split(const decode_attn_params* p, const void* q, const void* k_cache,
                      const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                      void* out, float* lse, int32_t num_splits, void* workspace,
                      size_t workspace_bytes, int32_t* status, void* stream) {
  return run_decode(p, q, k_cache, v_cache, block_table, seq_lens, out, lse, num_splits,
                    workspace, workspace_bytes, status, stream, false);
}

int decode_attn_combine(const decode_attn_params* p, const int32_t* seq_lens, int32_t num_splits,
                        int32_t chunk_len, const void* workspace, size_t workspace_bytes,
                        void* out, float* lse, void* stream) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (p->batch == 0) return DA_OK;
  if (seq_lens == nullptr || out == nullptr || lse == nullptr) return DA_ERR_NULL_POINTER;
  const bool listed = device_planned(p, num_splits);
  if (!listed && (num_splits < 1 || chunk_len < 1 || chunk_len % kTileTokens != 0 ||
                  ceil_div64(std::max(p->max_seq_len, 1), chunk_len) != num_splits))
    return DA_ERR_SPLITS;
  if (!listed && use_cluster_merge(p, num_splits)) return DA_OK;  // the split pass merged
  if (!aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 ||
      !stride_ok(p->o_stride_batch) || !stride_ok(p->o_stride_token) ||
      !stride_ok(p->o_stride_head))
    return DA_ERR_ALIGNMENT;
  const size_t rows_total = static_cast<size_t>(p->batch) * p->q_len * p->num_q_heads;
  dattn::CombineArgs c = {};
  if (listed) {
    // the plan, prefixes and item-indexed partials a device-planned split
    // pass left in the workspace (num_splits <= 0 there too)
    ListLayout lay;
    rc = list_layout(p, &lay);
    if (rc != DA_OK) return rc;
    if (workspace == nullptr || workspace_bytes < lay.total || !aligned16(workspace))
      return DA_ERR_WORKSPACE;
    const uint8_t* w = static_cast<const uint8_t*>(workspace);
    c.plan = reinterpret_cast<const int32_t*>(w + lay.plan);
    c.pre = reinterpret_cast<const int32_t*>(w + lay.pre);
    c.part_o = reinterpret_cast<const float*>(w + lay.part_o);
    c.part_lse = reinterpret_cast<const float*>(w + lay.part_lse);
    c.num_kv_heads = p->num_kv_heads;
  } else {
    const size_t need =
        rows_total * static_cast<size_t>(num_splits) * (kHeadDim + 1) * sizeof(float);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
      return DA_ERR_WORKSPACE;
    c.part_o = static_cast<const float*>(workspace);
    c.part_lse = c.part_o + rows_total * num_splits * kHeadDim;
  }
  c.seq_lens = seq_lens;
  c.out = static_cast<uint16_t*>(out);
  c.o_sb = p->o_stride_batch;
  c.o_st = p->o_stride_token;
  c.o_sh = p->o_stride_head;
  c.lse = lse;
  c.batch = p->batch;
  c.q_len = p->q_len;
  c.num_q_heads = p->num_q_heads;
  c.max_seq_len = p->max_seq_len;
  c.chunk_len = chunk_len;
  c.num_splits = num_splits;
  if (dattn::launch_combine(c, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}

}  // extern "C"

namespace {

// Staging layout of decode_attn_host's workspace: the partials of
// decode_attn(), then q, out, lse, seq_lens, the block table and the status
// word, each at a 256-byte boundary.
struct HostLayout {
  size_t part, q, out, lse, lens, bt, status, total;
};


int host_layout(const decode_attn_params* p, int32_t num_splits, bool paged, HostLayout* h) {
  size_t part = 0;
  int rc = decode_attn_workspace_bytes(p, num_splits, &part);
  if (rc != DA_OK) return rc;
  const size_t rows = static_cast<size_t>(p->batch) * p->q_len * p->num_q_heads;
  size_t off = round256(part);
  h->part = 0;
  h->q = off;
  off = round256(off + rows * kHeadDim * 2);
  h->out = off;
  off = round256(off + rows * kHeadDim * 2);
  h->lse = off;
  off = round256(off + rows * 4);
  h->lens = off;
  off = round256(off + static_cast<size_t>(p->batch) * 4);
  h->bt = off;
  if (paged) off = round256(off + static_cast<size_t>(p->batch) * p->block_table_stride * 4);
  h->status = off;
  h->total = off + 16;
  return DA_OK;
}

// The device's address of a page-locked host buffer (cudaHostAlloc /
// cudaHostRegister; also what torch's pin_memory gives), or false for
// pageable memory and anything else.
bool device_view(const void* host, const void** dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    cudaGetLastError();  // (an unknown pointer is not an error here)
    return false;
  }
  if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return false;
  *dev = at.devicePointer;
  return true;
}

// Element (b, t, h, d) at ((b * q_len + t) * Hq + h) * 128 + d (strides of
// dimensions of extent 1 do not matter).
bool dense_rows(int64_t sb, int64_t st, int64_t sh, const decode_attn_params* p) {
  const int64_t row = static_cast<int64_t>(p->num_q_heads) * kHeadDim;
  return (p->num_q_heads == 1 || sh == kHeadDim) && (p->q_len == 1 || st == row) &&
         (p->batch == 1 || sb == static_cast<int64_t>(p->q_len) * row);
}

}  // namespace

extern "C" {

int decode_attn_host_workspace_bytes(const decode_attn_params* p, int32_t num_splits,
                                     size_t* bytes) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (bytes == nullptr) return DA_ERR_NULL_POINTER;
  HostLayout h;
  rc = host_layout(p, num_splits, p->page_size > 0, &h);
  if (rc != DA_OK) return rc;
  *bytes = h.total;
  return DA_OK;
}

int decode_attn_host(const decode_attn_params* p, const void* q_host, const void* k_cache,
                     const void* v_cache, const int32_t* block_table_host,
                     const int32_t* seq_lens_host, void* out_host, float* lse_host,
                     int32_t num_splits, void* workspace, size_t workspace_bytes,
                     int32_t* status_host, void* stream) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  const bool paged = block_table_host != nullptr;
  rc = check_paged(p, paged);
  if (rc != DA_OK) return rc;
  if (p->batch == 0) {
    if (status_host != nullptr) *status_host = 0;
    return DA_OK;
  }
  if (q_host == nullptr || seq_lens_host == nullptr || out_host == nullptr ||
      lse_host == nullptr)
    return DA_ERR_NULL_POINTER;
  if (!dense_rows(p->q_stride_batch, p->q_stride_token, p->q_stride_head, p) ||
      !dense_rows(p->o_stride_batch, p->o_stride_token, p->o_stride_head, p))
    return DA_ERR_BAD_SHAPE;
  // the cache checks of decode_attn(), before anything is queued
  const bool no_keys = p->max_seq_len == 0;
  if (!no_keys && (k_cache == nullptr || v_cache == nullptr)) return DA_ERR_NULL_POINTER;
  if (!aligned16(k_cache) || !aligned16(v_cache) ||
      (!no_keys && (!kv_stride_ok(p, p->kv_stride_page) || !kv_stride_ok(p, p->kv_stride_token) ||
                    !kv_stride_ok(p, p->kv_stride_head))))
    return DA_ERR_ALIGNMENT;
  if (num_splits > 0) {  // the planner below reads the device itself
    HostLayout h0;
    rc = host_layout(p, num_splits, paged, &h0);
    if (rc != DA_OK) return rc;
    if (workspace == nullptr || workspace_bytes < h0.total || !aligned16(workspace))
      return DA_ERR_WORKSPACE;
  }
  DeviceInfo di;
  rc = current_device_info(&di);
  if (rc != DA_OK) return rc;
  if (di.major * 10 + di.minor < 100) return DA_ERR_NO_DEVICE;
  if (num_splits <= 0) {
    int32_t chunk = 0;
    rc = plan_impl(p, seq_lens_host, &num_splits, &chunk);
    if (rc != DA_OK) return rc;
  }
  HostLayout h;
  rc = host_layout(p, num_splits, paged, &h);
  if (rc != DA_OK) return rc;
  if (workspace == nullptr || workspace_bytes < h.total || !aligned16(workspace))
    return DA_ERR_WORKSPACE;

  uint8_t* w = static_cast<uint8_t*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(p->batch) * p->q_len * p->num_q_heads;
  const size_t bt_bytes = paged ? static_cast<size_t>(p->batch) * p->block_table_stride * 4 : 0;
  auto finish = [&](int code) {
    // the queued work reads or writes the caller's host buffers: it must be
    // done before the call returns, whatever the outcome
    if (cudaStreamSynchronize(st) != cudaSuccess && code == DA_OK) code = DA_ERR_CUDA;
    return code;
  };

  // Page-locked buffers: the kernels read q and the lengths and write out and
  // lse in host memory directly (over NVLink-C2C on Grace systems).  Two
  // inputs are read too often or too late for that: the block table, whose
  // entries the producers fetch one stage ahead of each copy, and q for the
  // tcgen05 kernel, which stages each work item's rows while the previous one
  // runs -- both go to the workspace first with one copy each (GB300, end to
  // end: w64 278 -> 259 us, w128 192 -> 162 us; the warp-MMA kernel reads
  // each query row once per CTA and keeps q in place).  A page-locked status
  // word is zeroed and written in place; any other one goes through a
  // workspace word.
  const void *q_d = nullptr, *lens_d = nullptr, *bt_d = nullptr, *out_d = nullptr,
             *lse_d = nullptr, *st_d = nullptr;
  if (device_view(q_host, &q_d) && device_view(seq_lens_host, &lens_d) &&
      (!paged || device_view(block_table_host, &bt_d)) && device_view(out_host, &out_d) &&
      device_view(lse_host, &lse_d)) {
    int32_t* status_dev = nullptr;
    if (status_host != nullptr) {
      if (device_view(status_host, &st_d)) {
        *status_host = 0;
        status_dev = static_cast<int32_t*>(const_cast<void*>(st_d));
      } else {
        status_dev = reinterpret_cast<int32_t*>(w + h.status);
        if (cudaMemsetAsync(status_dev, 0, 4, st) != cudaSuccess) return finish(DA_ERR_CUDA);
      }
    }
    const int32_t* bt_use = static_cast<const int32_t*>(bt_d);
    if (paged) {
      if (cudaMemcpyAsync(w + h.bt, block_table_host, bt_bytes, cudaMemcpyHostToDevice, st) !=
          cudaSuccess)
        return finish(DA_ERR_CUDA);
      bt_use = reinterpret_cast<const int32_t*>(w + h.bt);
    }
    const void* q_use = q_d;
    if (rows_of(p) > dattn::kMaxNarrowRows) {
      if (cudaMemcpyAsync(w + h.q, q_host, rows * kHeadDim * 2, cudaMemcpyHostToDevice, st) !=
          cudaSuccess)
        return finish(DA_ERR_CUDA);
      q_use = w + h.q;
    }
    rc = run_decode(p, q_use, k_cache, v_cache, bt_use, static_cast<const int32_t*>(lens_d),
                    const_cast<void*>(out_d), static_cast<float*>(const_cast<void*>(lse_d)),
                    num_splits, w + h.part, h.q, status_dev, stream, true);
    if (rc != DA_OK) return finish(rc);
    if (status_host != nullptr && st_d == nullptr &&
        cudaMemcpyAsync(status_host, w + h.status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return finish(DA_ERR_CUDA);
    return finish(DA_OK);
  }
  if (cudaMemcpyAsync(w + h.q, q_host, rows * kHeadDim * 2, cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(w + h.lens, seq_lens_host, static_cast<size_t>(p->batch) * 4,
                      cudaMemcpyHostToDevice, st) != cudaSuccess ||
      (paged && cudaMemcpyAsync(w + h.bt, block_table_host, bt_bytes, cudaMemcpyHostToDevice,
                                st) != cudaSuccess) ||
      cudaMemsetAsync(w + h.status, 0, 4, st) != cudaSuccess)
    return finish(DA_ERR_CUDA);
  rc = run_decode(p, w + h.q, k_cache, v_cache,
                  paged ? reinterpret_cast<const int32_t*>(w + h.bt) : nullptr,
                  reinterpret_cast<const int32_t*>(w + h.lens), w + h.out,
                  reinterpret_cast<float*>(w + h.lse), num_splits, w + h.part, h.q,
                  reinterpret_cast<int32_t*>(w + h.status), stream, true);
  if (rc != DA_OK) return finish(rc);
  if (cudaMemcpyAsync(out_host, w + h.out, rows * kHeadDim * 2, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(lse_host, w + h.lse, rows * 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      (status_host != nullptr &&
       cudaMemcpyAsync(status_host, w + h.status, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess))
    return finish(DA_ERR_CUDA);
  return finish(DA_OK);
}

int decode_attn_device_plan(const decode_attn_params* p, const int32_t* seq_lens,
                            void* workspace, size_t workspace_bytes, int32_t* status,
                            void* stream) {
  int rc = check_shape(p);
  if (rc != DA_OK) return rc;
  if (!device_planned(p, 0)) return DA_ERR_BAD_SHAPE;
  if (seq_lens == nullptr) return DA_ERR_NULL_POINTER;
  if ((reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0) return DA_ERR_ALIGNMENT;
  DeviceInfo di;
  rc = current_device_info(&di);
  if (rc != DA_OK) return rc;
  if (di.major * 10 + di.minor < 100) return DA_ERR_NO_DEVICE;
  ListLayout lay;
  rc = list_layout(p, &lay);
  if (rc != DA_OK) return rc;
  if (workspace == nullptr || workspace_bytes < lay.total || !aligned16(workspace))
    return DA_ERR_WORKSPACE;
  if (dattn::launch_plan(plan_args(p, seq_lens, status, static_cast<uint8_t*>(workspace), lay),
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}

const char* decode_attn_status_string(int code) {
  switch (code) {
    case DA_OK: return "ok";
    case DA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case DA_ERR_BAD_SHAPE: return "invalid sizes (batch, heads, q_len, lengths or paging)";
    case DA_ERR_HEAD_DIM: return "head_dim must be 128";
    case DA_ERR_PAGE_SIZE: return "page_size must be a positive multiple of 16";
    case DA_ERR_ROWS: return "(num_q_heads / num_kv_heads) * q_len exceeds 128";
    case DA_ERR_ALIGNMENT: return "pointer or stride misaligned (16-byte bases, strides multiple of 8 elements)";
    case DA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case DA_ERR_NO_DEVICE: return "no usable sm_100-class device is current";
    case DA_ERR_SPLITS: return "num_splits / chunk_len out of range";
    case DA_ERR_UNSUPPORTED:
      return "a flag combination this library does not run";
    case DA_ERR_STATIC_WORKSPACE_LIMIT:
      return "the call's partials exceed the 16 MiB static workspace (use fewer splits or decode_attn with a workspace)";
    default: return "unknown status code";
  }
}

}  // extern "C"
