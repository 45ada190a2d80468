/*
 * decode_attn.h -- C ABI of libdecode_attn.so: split-KV decode attention
 * (Flash-Decoding) for GB300 / sm_103a.
 *
 * The operation.  For every request b < batch, new token t < q_len and query
 * head h < num_q_heads, with key/value head kvh = h / G and G = Hq / Hkv
 * (contiguous GQA groups: "Capstone FlashAttention", §4.2; the inference-engine
 * chapter "12. attention kernels", decode section):
 *
 *     s_j   = scale * q[b,t,h,:] . K[b, j, kvh, :]
 *     out   = sum_j softmax(s)_j * V[b, j, kvh, :]          (bf16)
 *     lse   = ln sum_j exp(s_j)                              (fp32)
 *
 * exact attention softmax(QK^T/sqrt(d))V ("Capstone FlashAttention", §1.1),
 * over the keys j < L = seq_lens[b]; with `causal`, token t (at position
 * L - q_len + t) only sees keys j <= L - q_len + t.  A row with no visible key
 * gives out = 0 and lse = -inf.
 *
 * How.  The KV sequence of each (request, kv head) is cut into chunks of
 * `chunk_len` tokens that run on different SMs; each chunk keeps a running
 * max / running sum (online softmax, "Capstone FlashAttention", §1.2) and
 * writes an fp32 partial output plus its log-sum-exp; a combine kernel merges
 * the partials exactly ("Capstone FlashAttention", §2.3 FlashDecoding; the
 * per-tile LSE buffer of the CUTLASS split-KV post, §4.2).  Requests whose
 * keys fit one chunk skip the partials and the combine.  When the call needs
 * 2..16 chunks per (request, kv head) and all of them fit on the GPU at once,
 * the chunks of one head run as a thread-block cluster and merge through
 * distributed shared memory instead: one launch, no partials in memory (the
 * workspace is then unused; DA_FLAG_TWO_PASS turns this off).
 *
 * Cache layouts.  K and V share one layout; head_dim is contiguous.
 *   paged (block_table != NULL): element (page, slot, head, d) of a cache is at
 *       page*kv_stride_page + slot*kv_stride_token + head*kv_stride_head + d;
 *       logical token j of request b is page block_table[b*block_table_stride
 *       + j/page_size], slot j%page_size (PagedAttention, "Capstone
 *       FlashAttention", §4.1).
 *   contiguous (block_table == NULL): token j of request b is at
 *       b*kv_stride_page + j*kv_stride_token + head*kv_stride_head + d, for
 *       j < max_seq_len.
 * Strides are in elements; K and V base pointers must be 16-byte aligned and
 * every KV stride a multiple of 8 elements (16 bytes).
 *
 * FP8 caches (flags & DA_FLAG_KV_FP8_E4M3).  K and V hold one byte per element
 * in the OCP FP8 E4M3 format (1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits, subnormals, no infinities, S.1111.111 = NaN) with one fp32
 * scale per cache: the keys and values are k_scale * K and v_scale * V
 * (quantisation with explicit scaling factors rather than a plain cast:
 * "Capstone FlashAttention", §2.2 FP8 with scaling; the CUTLASS split-KV post,
 * §5.8).  q, out and lse keep their types.  Strides are then in bytes and must
 * be multiples of 16.
 *
 * Ownership and errors.  The caller owns every buffer (device memory unless
 * stated otherwise), including the workspace.  The library allocates nothing
 * on the device, never synchronises the stream and may be captured in a CUDA
 * graph.  Every function returns DA_OK (0) or a negative DA_ERR_* code; an
 * argument error is detected on the host before anything is launched.  Data
 * errors found on the device (a block-table entry outside [0, num_pages), a
 * seq_len outside [0, max_seq_len], a causal request shorter than q_len) are
 * OR-ed as DA_STATUS_* bits into *status when status != NULL; the caller reads
 * it after synchronising.  Faulty entries never fault the GPU: a bad page id
 * reads page 0 instead, an out-of-range length is clamped.
 *
 * Threading: all functions are thread-safe; calls on different streams may
 * overlap.
 */
#ifndef DECODE_ATTN_H_
#define DECODE_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DECODE_ATTN_HEAD_DIM 128   /* the only supported head_dim */
#define DECODE_ATTN_MAX_ROWS 128   /* (Hq / Hkv) * q_len must not exceed this;
                                      above 16 rows the tcgen05 kernel runs */
#define DECODE_ATTN_TOKEN_TILE 16  /* chunk_len and page_size are multiples */

/* return codes */
#define DA_OK 0
#define DA_ERR_NULL_POINTER -1     /* a required pointer is NULL */
#define DA_ERR_BAD_SHAPE -2        /* negative/zero sizes, Hq % Hkv != 0, ... */
#define DA_ERR_HEAD_DIM -3         /* head_dim != 128 */
#define DA_ERR_PAGE_SIZE -4        /* page_size not a positive multiple of 16 */
#define DA_ERR_ROWS -5             /* (Hq/Hkv)*q_len > DECODE_ATTN_MAX_ROWS */
#define DA_ERR_ALIGNMENT -6        /* pointer or stride misaligned */
#define DA_ERR_WORKSPACE -7        /* workspace NULL or smaller than required */
#define DA_ERR_CUDA -8             /* a CUDA runtime call or launch failed */
#define DA_ERR_NO_DEVICE -9        /* no usable sm_103 device is current */
#define DA_ERR_SPLITS -10          /* num_splits out of range */
#define DA_ERR_STATIC_WORKSPACE_LIMIT -11 /* partials exceed the static workspace */
#define DA_ERR_UNSUPPORTED -12     /* a flag combination this library does not run
                                      (reserved: no combination returns it at present) */

/* size of the device array behind decode_attn_static_workspace() */
#define DECODE_ATTN_STATIC_WORKSPACE_BYTES (16u << 20)

/* params.flags */
#define DA_FLAG_TWO_PASS 1u        /* always write fp32 partials to the workspace and
                                      merge them with the combine kernel (no
                                      cluster merge); needed to read partials */
#define DA_FLAG_KV_FP8_E4M3 2u     /* K and V caches are FP8 E4M3 bytes scaled by
                                      k_scale / v_scale (see "FP8 caches" above) */
#define DA_FLAG_TEST_WITHHOLD_COPY 0x100u /* test hook for failure detection:
                                      block (0, 0, 0) of the split launch never
                                      fills its first pipeline stage (at most 16
                                      rows per kv head: with DA_FLAG_TWO_PASS; above
                                      16, the tcgen05 kernel: the first stage of
                                      its first work item), so the bounded waits
                                      on it run out (~2 s each) and
                                      DA_STATUS_TIMEOUT is set; no fault, the
                                      context stays usable */

/* device status bits (OR-ed into *status) */
#define DA_STATUS_BAD_PAGE 1u      /* block-table entry outside [0, num_pages) */
#define DA_STATUS_SEQ_LEN 2u       /* seq_len < 0 or > max_seq_len (clamped) */
#define DA_STATUS_SHORT_CAUSAL 4u  /* causal and 0 < seq_len < q_len */
#define DA_STATUS_TIMEOUT 8u       /* an internal pipeline wait gave up */

typedef struct decode_attn_params {
  int32_t batch;              /* B >= 0 requests */
  int32_t q_len;              /* new tokens per request, >= 1 */
  int32_t num_q_heads;        /* Hq */
  int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0 */
  int32_t head_dim;           /* must be DECODE_ATTN_HEAD_DIM */
  int32_t page_size;          /* paged: tokens per page (multiple of 16);
                                 contiguous: ignored */
  int32_t max_pages_per_seq;  /* paged: usable columns of block_table */
  int32_t num_pages;          /* paged: physical pages in each cache (>= 1) */
  int32_t max_seq_len;        /* upper bound of seq_lens in this call; the
                                 contiguous cache holds this many tokens per
                                 request; paged: <= max_pages_per_seq*page_size */
  int32_t causal;             /* nonzero: causal mask among the q_len tokens */
  float scale;                /* softmax scale, e.g. 1/sqrt(head_dim) */
  int32_t flags;              /* DA_FLAG_* bits; 0 for the default path */
  int64_t q_stride_batch;     /* q [B, q_len, Hq, D] element strides; */
  int64_t q_stride_token;     /*   D contiguous, strides multiples of 8 */
  int64_t q_stride_head;
  int64_t o_stride_batch;     /* out [B, q_len, Hq, D] element strides */
  int64_t o_stride_token;
  int64_t o_stride_head;
  int64_t kv_stride_page;     /* see "Cache layouts" above */
  int64_t kv_stride_token;
  int64_t kv_stride_head;
  int64_t block_table_stride; /* elements between rows of block_table */
  float k_scale;              /* FP8 caches: keys = k_scale * K (1 by default) */
  float v_scale;              /* FP8 caches: values = v_scale * V (1 by default) */
} decode_attn_params;

/*
 * Fill *p with the strides of densely packed tensors:
 *   q, out [B, q_len, Hq, D]; paged caches [num_pages, page_size, Hkv, D];
 *   contiguous caches [B, max_seq_len, Hkv, D]; block_table [B, max_pages].
 * scale = 1/sqrt(head_dim), k_scale = v_scale = 1, flags = 0 (bf16 caches).
 * Pass page_size = 0 for a contiguous cache.
 */
void decode_attn_params_init(decode_attn_params *p, int32_t batch, int32_t q_len,
                             int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t page_size,
                             int32_t max_pages_per_seq, int32_t num_pages,
                             int32_t max_seq_len, int32_t causal);

/*
 * Split planner (host only; reads the current device's SM count once).
 * Picks the number of KV chunks per (request, kv head) and their length from
 * batch x kv heads x sequence length against the SM count, so that the split
 * kernel fills the GPU ("Capstone FlashAttention", §2.3: too few heads leave
 * SMs idle; chunks of a few hundred tokens or more).
 *   host_seq_lens  optional host copy of seq_lens (NULL: plan for max_seq_len)
 *   *num_splits    out: chunks per request at max_seq_len (>= 1)
 *   *chunk_len     out: tokens per chunk (multiple of 16)
 */
int decode_attn_plan(const decode_attn_params *p, const int32_t *host_seq_lens,
                     int32_t *num_splits, int32_t *chunk_len);

/*
 * The same planner for an explicit device shape (host only; needs no GPU and
 * touches no CUDA state), e.g. to plan ahead for another device:
 *   resident_ctas  CTAs of the split launch resident at once: SMs x CTAs per
 *                  SM of the kernel this shape runs (decode_attn_plan takes
 *                  the current device's SM count and the CUDA occupancy of
 *                  that kernel; on GB300, 152 SMs x 4 for bf16 caches with at
 *                  most 16 query rows per kv head, x 1 above 16 rows)
 * Equal lengths (or host_seq_lens NULL): one wave of equal chunks, at most 16
 * per (request, kv head).  Ragged lengths: chunks for about eight waves of
 * the real work, at least max(256, 64 x rows) tokens (256 x rows above 16
 * rows), shrunk (not below 256) while that leaves fewer chunks than resident
 * CTAs.  Returns DA_ERR_BAD_SHAPE unless 1 <= resident_ctas <= 2^31.
 */
int decode_attn_plan_slots(const decode_attn_params *p, const int32_t *host_seq_lens,
                           int64_t resident_ctas, int32_t *num_splits, int32_t *chunk_len);

/*
 * Chunk length used for a given num_splits: the smallest multiple of 16 that
 * covers max_seq_len in num_splits chunks.  Request b uses
 * ceil(seq_lens[b] / chunk_len) chunks (at least 1).
 */
int decode_attn_chunk_len(const decode_attn_params *p, int32_t num_splits,
                          int32_t *chunk_len);

/*
 * Workspace bytes decode_attn() needs for num_splits (0 when num_splits == 1;
 * unused when the cluster merge applies, see above).
 * Layout (fp32): partial outputs [B, q_len, Hq, num_splits, D], followed by
 * partial log-sum-exps [B, q_len, Hq, num_splits] (natural log).  Partial s of
 * a row is normalised (sum of weights 1) over its chunk's keys; an empty
 * chunk has lse -inf.  Entries of requests that use a single chunk are not
 * written.
 * num_splits <= 0: the need of the planned call -- for a device-planned call
 * (see "Device planning" at decode_attn) a bound that does not depend on the
 * lengths, for one request the host plan's need.  Reads the current device.
 */
int decode_attn_workspace_bytes(const decode_attn_params *p, int32_t num_splits,
                                size_t *bytes);

/*
 * Decode attention (the whole path: split kernel, then combine when a request
 * spans more than one chunk).
 *   q            bf16 [B, q_len, Hq, 128] (strides in *p)
 *   k_cache      bf16 cache, layout per *p (16-byte aligned)
 *   v_cache      bf16 cache, same layout as k_cache
 *   block_table  int32 [B, block_table_stride] or NULL (contiguous cache)
 *   seq_lens     int32 [B]: keys per request, including the q_len new tokens
 *   out          bf16 [B, q_len, Hq, 128] (strides in *p)
 *   lse          fp32 [B, q_len, Hq], contiguous
 *   num_splits   chunks per request at max_seq_len; <= 0 asks the planner
 *   workspace    device buffer of >= decode_attn_workspace_bytes() bytes
 *                (may be NULL when that is 0)
 *   status       optional int32 device word; DA_STATUS_* bits are OR-ed in
 *   stream       cudaStream_t to launch on (NULL: legacy default stream)
 * Device pointers only.  Asynchronous with respect to the host.
 *
 * Device planning (num_splits <= 0 with two or more requests; for the
 * tcgen05 kernel, above 16 rows per kv head, at most 1024 requests).  The
 * lengths may exist only on the device -- and change between replays of a
 * captured graph -- so the call plans there: a planner kernel applies
 * decode_attn_plan()'s rule to the current seq_lens (the same plan the host
 * planner gives for those lengths), then the split kernel runs one CTA per
 * item slot of a capacity fixed by the shape (B x Hkv + 16 waves of resident
 * CTAs), then the combine kernel merges: three launches, no host
 * synchronisation, graph capturable.  If the rule's chunk would make more
 * (request, kv head, chunk) items than the capacity, the chunk grows until
 * they fit.  Workspace layout (offsets rounded up to 256 bytes): int32
 * plan[4] = {chunk_len, items, chunks of the longest request, capacity};
 * int32 pre[B + 1], the exclusive prefix over requests of their chunk
 * counts; int4 items[capacity] = (b, kv head, chunk, clamped length) in
 * (request, kv head, chunk) order; fp32 partial outputs [capacity, rows, D]
 * and partial LSEs [capacity, rows], item i = pre[b] * Hkv + kvh * n_b + s
 * holding row r = t * G + g of that (b, kvh) (n_b = max(1, ceil(L_b /
 * chunk_len)) chunks).  One request keeps the host plan (from max_seq_len)
 * and, where it fits, the cluster merge.
 */
int decode_attn(const decode_attn_params *p, const void *q, const void *k_cache,
                const void *v_cache, const int32_t *block_table,
                const int32_t *seq_lens, void *out, float *lse,
                int32_t num_splits, void *workspace, size_t workspace_bytes,
                int32_t *status, void *stream);

/*
 * The split pass alone: the same arguments and the same first launch as
 * decode_attn().  Rows of requests that fit one chunk get their final out/lse;
 * rows of longer requests get partials in `workspace` (layout above), which
 * decode_attn_combine() with the same num_splits and the chunk length from
 * decode_attn_chunk_len() then merges.  decode_attn() == decode_attn_split()
 * followed by decode_attn_combine().
 */
int decode_attn_split(const decode_attn_params *p, const void *q, const void *k_cache,
                      const void *v_cache, const int32_t *block_table,
                      const int32_t *seq_lens, void *out, float *lse,
                      int32_t num_splits, void *workspace, size_t workspace_bytes,
                      int32_t *status, void *stream);

/*
 * The combine step alone: merges the partials that a split pass left in
 * `workspace` (layout above) into out/lse, for every row whose request uses
 * two or more chunks of `chunk_len` tokens.  M = max_s lse_s,
 * w_s = exp(lse_s - M), out = sum_s w_s O_s / sum_s w_s, lse = M + ln sum w_s
 * (the two-block merge of "Capstone FlashAttention", §1.2, applied to all
 * chunks).  decode_attn() calls it itself; it is exported so that the merge
 * can be run and checked on its own.
 */
/*   num_splits / chunk_len: the values the split pass used (num_splits ==
 *   ceil(max_seq_len / chunk_len)).  Launches nothing when that split pass
 *   merged through clusters (same params, same num_splits).  num_splits <= 0:
 *   the split pass was device-planned; the chunk length, prefixes and
 *   item-indexed partials are read from `workspace` (chunk_len is ignored). */
int decode_attn_combine(const decode_attn_params *p, const int32_t *seq_lens,
                        int32_t num_splits, int32_t chunk_len,
                        const void *workspace, size_t workspace_bytes, void *out,
                        float *lse, void *stream);

/*
 * decode_attn() for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for callers such as
 * plugin hosts that pass only input and output buffers, runtimes whose device
 * memory is owned by another allocator, and deployments that forbid device
 * allocation after start-up.  Same arguments as decode_attn() minus the
 * workspace: the partials go to a DECODE_ATTN_STATIC_WORKSPACE_BYTES (16 MiB)
 * array in the library's own device memory, which every GPU that loads the
 * library holds until the process exits.
 *   - A call needing more than that returns DA_ERR_STATIC_WORKSPACE_LIMIT and
 *     launches nothing (decode_attn_workspace_bytes() gives the need).
 *   - All calls on a device share the array, and it keeps the last call's
 *     contents (nothing in it needs clearing).  Calls that overlap on the GPU
 *     race on it: serialise them.
 *   - The first call in each CUDA context looks up the array's address with
 *     that device current (once per device; again after cudaDeviceReset, or
 *     in another context a driver-API caller made current); make it before
 *     any stream capture in that context.
 *   - Only calls that write partials (decode_attn_launch_count() == 2) use
 *     the array and count against the limit; single-chunk and cluster-merged
 *     calls never do.
 * Allocates nothing (no cudaMalloc/cudaFree or allocating library call).
 */
int decode_attn_static_workspace(const decode_attn_params *p, const void *q,
                                 const void *k_cache, const void *v_cache,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 void *out, float *lse, int32_t num_splits,
                                 int32_t *status, void *stream);

/*
 * decode_attn() with the per-call inputs and outputs in host memory: the call
 * a serving loop makes when q, seq_lens and the block table arrive from the
 * host and out / lse go back to it, while the K/V cache stays resident on the
 * device.  It runs the same kernels as decode_attn() and returns once
 * `stream` has finished the call's work.  When q, seq_lens, the block table,
 * out and lse are all page-locked (cudaHostAlloc / cudaHostRegister), the
 * kernels read seq_lens and write out and lse in place through the GPU's
 * mapping of host memory (NVLink-C2C on Grace systems), and read q in place
 * too when there are at most 16 query rows per KV head; the block table (and
 * q above 16 rows) is first copied into `workspace` with one copy each,
 * because the kernels read them many times or late.  A page-locked status
 * word is zeroed and written in place too.  Otherwise the call copies
 * q, seq_lens and the block table into device staging buffers carved from
 * `workspace` and copies out and lse (and the status word) back.  Unlike every
 * other entry it synchronises the stream, so it cannot be captured in a CUDA
 * graph.
 *   q_host            bf16 [B, q_len, Hq, 128] in host memory, dense: the
 *                     params' q strides must be the packed ones
 *   k_cache, v_cache  the device caches, as for decode_attn()
 *   block_table_host  int32 [B, block_table_stride] in host memory, or NULL
 *                     (contiguous cache)
 *   seq_lens_host     int32 [B] in host memory
 *   out_host          bf16 [B, q_len, Hq, 128] in host memory, dense (the
 *                     params' out strides must be the packed ones)
 *   lse_host          fp32 [B, q_len, Hq] in host memory
 *   num_splits        chunks per request; <= 0 asks the planner, which here
 *                     sees the actual lengths (decode_attn_plan() with
 *                     seq_lens_host gives the same count, for sizing the
 *                     workspace)
 *   workspace         device buffer of >= decode_attn_host_workspace_bytes()
 *                     bytes for that split count (16-byte aligned): the
 *                     partials of decode_attn(), then the staging buffers
 *   status_host       optional int32 host word: the call's DA_STATUS_* bits
 *   stream            cudaStream_t (NULL: legacy default stream)
 * Page-locked host buffers (cudaHostAlloc / cudaHostRegister) take the
 * direct path above; pageable memory works through staging copies.
 * Argument errors return before anything is copied or launched; a failure
 * after the copies were queued waits for the stream, then returns the code.
 */
int decode_attn_host_workspace_bytes(const decode_attn_params *p, int32_t num_splits,
                                     size_t *bytes);
int decode_attn_host(const decode_attn_params *p, const void *q_host, const void *k_cache,
                     const void *v_cache, const int32_t *block_table_host,
                     const int32_t *seq_lens_host, void *out_host, float *lse_host,
                     int32_t num_splits, void *workspace, size_t workspace_bytes,
                     int32_t *status_host, void *stream);

/*
 * The device planner alone: writes the plan, prefixes and item list that a
 * device-planned decode_attn() call with these params would compute from
 * seq_lens (layout under "Device planning" above) into `workspace`, without
 * running the kernels that follow, so the plan can be read back and checked.
 * The params must be ones decode_attn() plans on the device (two or more
 * requests; tcgen05 shapes up to 1024 requests), else DA_ERR_BAD_SHAPE.
 * DA_STATUS_SEQ_LEN / DA_STATUS_SHORT_CAUSAL are OR-ed into *status as the
 * full call would.  Asynchronous; graph capturable.
 */
int decode_attn_device_plan(const decode_attn_params *p, const int32_t *seq_lens,
                            void *workspace, size_t workspace_bytes, int32_t *status,
                            void *stream);

/* Static description of a return code. */
const char *decode_attn_status_string(int code);

/* Number of kernel launches decode_attn() makes for these arguments (1 or 2;
 * 1 with the cluster merge; 3 for a device-planned call: planner, split,
 * combine). */
int decode_attn_launch_count(const decode_attn_params *p, int32_t num_splits);

#ifdef __cplusplus
}
#endif

#endif /* DECODE_ATTN_H_ */
