/*
 * pa.h -- C ABI of libpa: attention forward over a paged KV cache on GB300 (sm_103a).
 *
 *   out[i, h] = sum_j softmax_j(scale * <q[i, h], k_j>) * v_j      (bf16)
 *   lse[i, h] = ln sum_j exp(scale * <q[i, h], k_j>)               (fp32, natural log)
 *
 * Keys and values live in 64-row pages.  Logical key j of sequence b is row
 * j % 64 of physical page block_table[b, j / 64] (FlashMLA "Tensor Shapes
 * Reference", diagram "Prefill to Cache Mapping"); query head h reads KV head
 * h / (Hq / Hk), contiguous groups (same page, diagram "Grouped-Query
 * Attention").  Keys at or past seq_len are never read ("unused slots ignored
 * via seq_lens", section 1 notes).  An empty key set yields out = 0 and
 * lse = -inf.
 *
 * Conventions shared by every call:
 *  - Ownership: the caller allocates and owns every buffer.  The library never
 *    allocates device memory and never synchronises inside pa_decode /
 *    pa_prefill; work is enqueued on `stream` and runs asynchronously.
 *  - Pointers named *_host are host memory; every other pointer is device
 *    memory on the current device, 16-byte aligned, contiguous in the layout
 *    given.
 *  - Errors: arguments are validated on the host before anything is enqueued;
 *    a failing check returns a non-zero pa_status and leaves a message for
 *    pa_last_error().  Faults the kernels detect themselves (a page id out of
 *    range, a wait that ran past its time limit) are recorded in the status
 *    word at the start of the caller's workspace and reported by
 *    pa_check_status().  Nothing traps.
 *  - Page size is 64 ("Blk: block size for paged cache (always 64)").
 *  - The pool layout is [num_pool_pages, Hk, 64, D] ("HND"): each (page, KV
 *    head) is one contiguous 64 x D slab (the "64 rows x D cols (contiguous
 *    slab)" of the paged-cache diagram).
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* a pointer, shape or value check failed on the host */
    PA_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels implement */
    PA_ERR_WORKSPACE = 3,     /* metadata or workspace buffer too small */
    PA_ERR_CUDA = 4,          /* a CUDA runtime call failed */
    PA_ERR_TIMEOUT = 5,       /* (device) a wait ran past its time limit */
    PA_ERR_DEVICE_BOUNDS = 6  /* (device) a page id or length was out of range */
} pa_status;

/* Element type of the KV pools.  With PA_KV_FP16 the query, the pools and the
 * output are all fp16 (q, k, v share one type, as MATE's forward requires);
 * otherwise the query and output are bf16. */
typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1, PA_KV_FP16 = 2 } pa_kv_dtype;

#define PA_PAGE_SIZE 64
#define PA_MAX_SPLITS 64
#define PA_MAX_GROUP 16     /* Hq / Hk supported by the decode kernels */
#define PA_STATUS_BYTES 256 /* status word region at the start of every workspace */

/* ----------------------------------------------------------------- decode */

typedef struct {
    int32_t batch;             /* B */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hk; Hq % Hk == 0 and Hq / Hk <= 16 */
    int32_t head_dim;          /* D: 64 or 128 */
    int32_t page_size;         /* must be 64 */
    int32_t max_pages_per_seq; /* row stride of block_table */
    int32_t num_pool_pages;    /* pages in k_pool / v_pool */
    int32_t kv_dtype;          /* pa_kv_dtype */
    int32_t num_sms;           /* SMs of the device (cudaDevAttrMultiProcessorCount) */
    int32_t ctas_per_sm;       /* persistent decode CTAs per SM; 0 = library default (1) */
    int32_t forced_splits;     /* split-KV count per sequence; 0 = choose automatically */
} pa_decode_shapes;

typedef struct {
    int32_t total_splits;   /* sum over sequences of the split count */
    int32_t num_items;      /* (sequence, split, KV head) work items */
    int32_t grid;           /* decode CTAs the schedule was built for */
    int32_t meta_ints;      /* int32 entries of the packed metadata */
    int32_t ctas_per_sm;    /* resolved value */
    int32_t reserved;
    size_t workspace_bytes; /* device workspace pa_decode needs */
} pa_decode_plan;

/*
 * pa_get_metadata -- choose the split-KV count of every sequence and the
 * persistent CTAs' work lists (the scheduler-metadata step: FlashMLA
 * get_mla_metadata, "Tensor Shapes Reference" section 2; MATE
 * get_scheduler_metadata with num_splits 0 = automatic).  Pure host code.
 *
 *   seq_lens_host     int32 [B] keys per sequence, 0 <= len <= max_pages * 64
 *   block_table_host  int32 [B, max_pages] or NULL; when given, every live slot
 *                     (column < ceil(len / 64)) is checked to hold a page id in
 *                     [0, num_pool_pages)
 *   shapes            see pa_decode_shapes
 *   meta_host         int32 [meta_capacity_ints] output, or NULL to only size
 *   plan              output: sizes and counts (always filled on PA_OK)
 *
 * Split rule (integers only, deterministic):
 *   pages_b = ceil(len_b / 64); units = sum_b pages_b * Hk;
 *   cap = num_sms * ctas_per_sm; chunk = max(4, ceil(units / (2 * cap)));
 *   n_b = 1 if pages_b <= 1, else min(forced, pages_b, 64) if forced > 0,
 *   else min(ceil(pages_b / chunk), 64).  Split s of b covers pages
 *   [floor(s * pages_b / n_b), floor((s + 1) * pages_b / n_b)).
 * Work items (b, s, kv head), cost = pages + 1, are dealt longest first to the
 * least-loaded of grid = min(#items, cap) CTAs (ties: lowest index).
 *
 * Packed layout (int32): [0] 0x50414D31 [1] B [2] Hk [3] total_splits
 * [4] num_items [5] grid [6] chunk [7] ctas_per_sm, then n_splits[B],
 * split_indptr[B+1], cta_indptr[grid+1], items[2*num_items] = (b, s<<16 | kvh).
 *
 * Returns PA_ERR_WORKSPACE (plan filled) if meta_capacity_ints < plan->meta_ints.
 */
pa_status pa_get_metadata(const int32_t* seq_lens_host, const int32_t* block_table_host,
                          const pa_decode_shapes* shapes, int32_t* meta_host, size_t meta_capacity_ints,
                          pa_decode_plan* plan);

/*
 * Device-side scheduling, for decode steps captured once in a CUDA graph and
 * replayed with new lengths (MATE's static plans: a plan built from
 * capacities, per-call lengths in device buffers, no host reads while
 * capturing).
 *
 * pa_get_static_plan (host, no lengths): a plan that covers every length mix
 * of `batch` sequences -- the split rule yields at most
 * batch + ceil(2 * num_sms * ctas_per_sm / Hk) splits (batch * min(forced, 64)
 * with forced splits).  Use it for pa_decode and for sizing the metadata
 * buffer (plan->meta_ints) and the workspace.  Limits: batch <= 8192, at most
 * 16384 work items (splits * Hk); PA_ERR_UNSUPPORTED beyond.
 *
 * pa_get_metadata_device (device, async on `stream`): one CTA reads
 * seq_lens_dev int32 [B] and writes the packed metadata of pa_get_metadata to
 * meta_dev int32 [plan->meta_ints] -- the same split rule, but the items,
 * sorted longest first, are dealt to the CTAs in snake order (0..grid-1, then
 * grid-1..0, ...) instead of least-loaded first.  Lengths above
 * max_pages_per_seq * 64 are clamped.
 */
pa_status pa_get_static_plan(const pa_decode_shapes* shapes, pa_decode_plan* plan);

pa_status pa_get_metadata_device(const pa_decode_shapes* shapes, const pa_decode_plan* static_plan,
                                 const int32_t* seq_lens_dev, int32_t* meta_dev, cudaStream_t stream);

/*
 * pa_decode -- single-token decode over the paged cache (FlashMLA
 * flash_mla_with_kvcache, "Tensor Shapes Reference" section 1; MATE paged mode,
 * flash_attn_with_kvcache), with split-KV partials merged by a log-sum-exp
 * combine when any sequence has more than one split.
 *
 *   q            bf16 [B, Hq, D] (fp16 with PA_KV_FP16)
 *   k_pool       [num_pool_pages, Hk, 64, D], bf16, e4m3 or fp16 per shapes->kv_dtype
 *   v_pool       same layout and type as k_pool
 *   k_scale      fp32 [Hk] per-KV-head dequantisation scale (e4m3 only, else NULL)
 *   v_scale      fp32 [Hk] (e4m3 only, else NULL); an e4m3 element x of head g
 *                stands for x * k_scale[g] (keys) or x * v_scale[g] (values)
 *   block_table  int32 [B, max_pages_per_seq]; slots past ceil(len/64) never read
 *   seq_lens     int32 [B] (device copy of the lengths given to pa_get_metadata)
 *   meta_dev     int32 [plan->meta_ints], device copy of pa_get_metadata's output
 *   scale        softmax scale (e.g. 1/sqrt(D))
 *   out          bf16 [B, Hq, D] (fp16 with PA_KV_FP16)
 *   lse          fp32 [B, Hq] or NULL
 *   workspace    >= plan->workspace_bytes device bytes; the first 256 bytes hold
 *                the status word, then the split partials, then one arrival
 *                counter per (sequence, KV head) for the in-kernel merge.
 *                Zero-fill it once before first use; on success the library
 *                leaves the status word and the counters at zero.  After a
 *                call that returned an error or left a device status (see
 *                pa_check_status), zero-fill it again: an aborted launch can
 *                leave counters part-way.  A workspace must not be used by two
 *                calls that may overlap.
 *
 * With fp8 KV the query is used in fp16 (exact for |q| in [2^-14, 65504];
 * smaller magnitudes round to fp16 subnormals).
 *
 * Stream order: the call is asynchronous on `stream`.  For every page type
 * but e4m3 at D = 128 (which has a kernel of its own, launched plainly) the
 * kernel is launched with programmatic stream serialization: its CTAs may
 * start their shared-memory set-up while the
 * previous kernel in the stream finishes, and touch no global memory until
 * that kernel has completed, so every input written and every buffer read by
 * earlier work in the stream is ordered as for a plain launch.  Under stream
 * capture that dependency becomes a programmatic edge of the graph.
 */
pa_status pa_decode(const pa_decode_shapes* shapes, const pa_decode_plan* plan, const void* q,
                    const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                    const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev,
                    float scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/*
 * The two steps pa_decode runs, callable on their own (same arguments and
 * rules as pa_decode):
 *   pa_decode_attend   the decode kernel alone: sequences with one split get
 *                      their final out / lse; split sequences leave fp32
 *                      partials (output normalised by its split's own sum, and
 *                      the split's log-sum-exp) in the workspace;
 *   pa_decode_combine  merges those partials: with m = max_s lse_s,
 *                      lse = m + ln sum_s exp(lse_s - m) and
 *                      out = sum_s exp(lse_s - lse) * o_s.
 *                      A no-op when plan->total_splits == batch.
 */
pa_status pa_decode_attend(const pa_decode_shapes* shapes, const pa_decode_plan* plan, const void* q,
                           const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                           const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev,
                           float scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

pa_status pa_decode_combine(const pa_decode_shapes* shapes, const pa_decode_plan* plan, const int32_t* meta_dev,
                            void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory, for instance code whose host framework owns every byte of device
 * memory through its own pool, or a loop that cannot afford the device-wide
 * synchronisation an allocation may cause.  (The pages have no counterpart to
 * this call; it exists for such callers.)
 *
 * Same arguments as pa_decode without the workspace: the split partials and
 * the status word live in one scratch array of 16 MiB in this library's own
 * device memory, which every GPU that loads the library keeps until the
 * process exits.  The call allocates nothing and frees nothing.
 *   - plan->workspace_bytes above 16 MiB is rejected with PA_ERR_WORKSPACE.
 *   - The first call on a device looks up the scratch array's device address
 *     (with that device current) and keeps it for later calls; make that
 *     first call before any stream capture.  The address belongs to the
 *     device's context: after cudaDeviceReset the next call (again outside
 *     any capture) looks it up anew in the new context.
 *   - All calls share the one array, which keeps the last call's contents;
 *     the status word is cleared at the start of each call.  Calls that may
 *     overlap on the GPU (other streams, other host threads) race on it.
 *   - Every host-side check (the same as pa_decode's) runs before anything
 *     is enqueued; a rejected call leaves the stream untouched.
 *   - status_host: NULL, or a host int32 that receives the device status word
 *     (PA_OK or the first device-detected fault: PA_ERR_DEVICE_BOUNDS,
 *     PA_ERR_TIMEOUT); the call then waits for `stream` before returning.
 *     With NULL the call does not wait, and a device-detected fault is not
 *     reported: the status word sits in the private scratch array, and the
 *     next call clears it.
 */
pa_status pa_decode_noalloc(const pa_decode_shapes* shapes, const pa_decode_plan* plan, const void* q,
                            const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev,
                            float scale, void* out, float* lse, int32_t* status_host, cudaStream_t stream);

/*
 * pa_page_table_from_flat -- block table rows from a flat list of page ids, on
 * the device (MATE msa_interface, _build_page_table_from_flat_kv_indices, page
 * counts as in _page_counts).  Sequence b owns the next ceil(kv_lens[b] / 64)
 * ids of kv_indices, in order; they fill the first columns of row b of
 * block_table and every other entry of the row is written 0.  Capture-safe:
 * no allocation, no synchronisation, lengths read on the device, so a CUDA
 * graph can replay it with new lengths and ids.
 *   kv_indices  int32 [num_indices] (device; may be NULL when num_indices is 0)
 *   kv_lens     int32 [batch] (device)
 *   block_table int32 [batch, max_pages_per_seq] (device, written in full)
 *   workspace   >= PA_STATUS_BYTES device bytes (status word), zero-filled once
 * Host checks: 1 <= batch <= 8192, max_pages_per_seq > 0, num_indices >= 0,
 * pointers.  Device checks, recorded as PA_ERR_DEVICE_BOUNDS in the status
 * word (pa_check_status): a negative length (counted as 0 pages), a sequence
 * with more pages than max_pages_per_seq (its row keeps its first ids), or a
 * list whose length differs from the page total the lengths imply (ids past
 * num_indices are not read; their entries are 0).
 */
pa_status pa_page_table_from_flat(const int32_t* kv_indices, int64_t num_indices, const int32_t* kv_lens,
                                  int32_t batch, int32_t max_pages_per_seq, int32_t* block_table, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/* ----------------------------------------------------------------- prefill */

typedef struct {
    int32_t batch;             /* B sequences */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hk, Hq % Hk == 0 */
    int32_t head_dim_qk;       /* q depth: 128, or 192 with rope_dim 64 */
    int32_t head_dim_v;        /* 128 */
    int32_t rope_dim;          /* 0, or 64: last 64 q entries pair with k_rope */
    int32_t max_seqlen_q;      /* upper bound on every q segment length */
    int32_t total_q;           /* cu_seqlens_q[B] */
    int32_t total_k;           /* cu_seqlens_k[B] (ragged keys); for paged keys the
                                  sum of kv lengths */
    int32_t page_size;         /* 64 when block_table is given */
    int32_t max_pages_per_seq; /* block_table row stride (paged) */
    int32_t num_pool_pages;    /* pages in the pools (paged) */
    int32_t num_sms;           /* informational: the prefill launch queries the current device */
    int32_t dtype;             /* PA_KV_BF16 or PA_KV_FP16: q, k, v, k_rope and out */
} pa_prefill_shapes;

/*
 * pa_prefill -- causal (or full) attention for a ragged batch of query
 * segments: chunked prefill against a paged cache (FlashMLA mha_fwd_kvcache,
 * section 4), ragged prefill (MATE dense mode, flash_attn_varlen_func) and the
 * MLA shape with one 64-wide rope key shared by all heads (Modular
 * flare_mla_prefill).
 *
 *   q            bf16 [total_q, Hq, head_dim_qk]
 *   k, v         paged (block_table != NULL): bf16 pools [num_pool_pages, Hk, 64, Dk]
 *                and [num_pool_pages, Hk, 64, Dv]; ragged: bf16 [total_k, Hk, Dk]
 *                and [total_k, Hk, Dv]; Dk = head_dim_qk - rope_dim
 *   k_rope       bf16 [total_k, 1, rope_dim] (ragged keys only) or NULL
 *   cu_seqlens_q int32 [B+1] running offsets of the query segments
 *   cu_seqlens_k int32 [B+1] running offsets of the key segments (kv lengths)
 *   qo_offset    int32 [B] or NULL (= kv_len - q_len): with causal != 0 query row
 *                i of segment b sees key j iff j <= qo_offset[b] + i (MATE
 *                _normalize_qo_offset / _resolve_seqused_k)
 *   out          bf16 [total_q, Hq, head_dim_v];  lse fp32 [total_q, Hq] or NULL
 *   workspace    >= PA_STATUS_BYTES device bytes (status word), zero-filled once.
 *                The status region also holds the work counters of the
 *                persistent kernel (int32 at bytes 64 and 128): one CTA per SM
 *                takes (256-row query block, head) items from them, and the
 *                last CTA to finish sets them back to zero, so they need no
 *                clearing between calls.  With pa_prefill_workspace_size(shapes)
 *                bytes the call also orders the items longest first (a small
 *                sorting kernel writes the order after the status region);
 *                with less it uses a fixed order.  Results are identical
 *                either way.  Calls that share a workspace must not overlap
 *                in time (one stream).
 */
pa_status pa_prefill(const pa_prefill_shapes* shapes, const void* q, const void* k, const void* v,
                     const void* k_rope, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                     const int32_t* block_table, const int32_t* qo_offset, int causal, float scale,
                     void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes with which pa_prefill also orders its work longest first:
 * PA_STATUS_BYTES + 4 * batch * ceil(max_seqlen_q / 256). */
size_t pa_prefill_workspace_size(const pa_prefill_shapes* shapes);

/*
 * pa_prefill_mla_fp8 -- the MLA prefill of pa_prefill with the per-head parts
 * of q and k in e4m3: Modular flare_mla_prefill's overload taking q_nope,
 * q_rope, q_scale and k_scales.  The page gives those arguments but not the
 * granularity of the scales; here there is one fp32 scale per head:
 *   score(i, j, h) = scale * (q_scale[h] * k_scale[g] * <q_nope[i, h], k_nope[j, g]>
 *                             + <q_rope[i, h], k_rope[j, 0]>),   g = h / (Hq / Hk)
 *   q_nope   e4m3 [total_q, Hq, 128]      q_rope  bf16 [total_q, Hq, 64]
 *   k_nope   e4m3 [total_k, Hk, 128]      k_rope  bf16 [total_k, 1, 64]
 *   v        bf16 [total_k, Hk, 128]      out     bf16 [total_q, Hq, 128]
 *   q_scale  fp32 [Hq], k_scale fp32 [Hk] (device), positive and finite
 * shapes: dtype PA_KV_FP8_E4M3, head_dim_qk 192, rope_dim 64, head_dim_v 128;
 * keys are ragged (no block table); cu_seqlens, qo_offset, causal, lse and the
 * workspace as for pa_prefill.  The q_nope . k_nope products run on the e4m3
 * tensor path, the rope part and P.V in bf16; to add both into one
 * accumulator the kernel divides the query's rope part by q_scale * k_scale
 * once and holds it as two bf16 levels (hi + lo, about 16 significant bits).
 * A scale that is not positive and finite is recorded as PA_ERR_INVALID_ARG
 * in the status word.
 */
pa_status pa_prefill_mla_fp8(const pa_prefill_shapes* shapes, const void* q_nope, const void* q_rope,
                             const float* q_scale, const void* k_nope, const float* k_scale, const void* v,
                             const void* k_rope, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             const int32_t* qo_offset, int causal, float scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pa_prefill_mla_rope_fp8 -- the MLA prefill of pa_prefill with the shared
 * rope key quantised: Modular flare_mla_prefill's overload taking k_rope and
 * k_rope_scales.  The page gives the argument but not its granularity; here
 * there is one fp32 scale per key token:
 *   score(i, j, h) = scale * (<q[i, h, 0:128], k_nope[j, g]>
 *                             + k_rope_scales[j] * <q[i, h, 128:192], k_rope[j]>)
 *   q        bf16 [total_q, Hq, 192]      k_nope  bf16 [total_k, Hk, 128]
 *   v        bf16 [total_k, Hk, 128]      out     bf16 [total_q, Hq, 128]
 *   k_rope   e4m3 [total_k, 1, 64]        k_rope_scales fp32 [total_k] (device)
 * shapes: dtype PA_KV_BF16, head_dim_qk 192, rope_dim 64, head_dim_v 128;
 * keys are ragged (no block table); cu_seqlens, qo_offset, causal and lse as
 * for pa_prefill.  The call first expands the rope key, once for all heads,
 * into two bf16 levels hi + lo of code * scale (about 16 significant bits)
 * inside the workspace, then runs the MLA prefill with both levels as
 * key chunks.  workspace: pa_prefill_mla_rope_fp8_workspace_size(shapes)
 * bytes, zero-filled once (the status region as for pa_prefill; the two
 * levels, 2 x 128 bytes per key token, follow the ordering region);
 * PA_ERR_WORKSPACE if smaller.
 */
pa_status pa_prefill_mla_rope_fp8(const pa_prefill_shapes* shapes, const void* q, const void* k_nope,
                                  const void* v, const void* k_rope, const float* k_rope_scales,
                                  const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                  const int32_t* qo_offset, int causal, float scale, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes pa_prefill_mla_rope_fp8 needs: pa_prefill_workspace_size
 * rounded up to 256, then two regions of total_k * 128 bytes (each rounded up
 * to 256). */
size_t pa_prefill_mla_rope_fp8_workspace_size(const pa_prefill_shapes* shapes);

/* ----------------------------------------------------------------- mixed batches */

typedef struct {
    int32_t batch;             /* B sequences, decode (one query token) first */
    int32_t num_q_heads, num_kv_heads, head_dim; /* D = 128 */
    int32_t page_size;         /* must be 64 */
    int32_t max_pages_per_seq, num_pool_pages;
    int32_t kv_dtype;          /* PA_KV_BF16 */
    int32_t num_sms, ctas_per_sm, forced_splits;  /* for the decode part, as in pa_decode_shapes */
} pa_mixed_shapes;

typedef struct {
    int32_t num_decode;     /* leading sequences with one query token: the decode part */
    int32_t total_q;        /* cu_seqlens_q[B] */
    int32_t max_seqlen_q;   /* longest query segment of the prefill part */
    int32_t reserved;
    pa_decode_plan decode;  /* plan of the decode part (metadata = the first decode.meta_ints ints) */
    size_t workspace_bytes; /* decode workspace followed by the prefill workspace */
} pa_mixed_plan;

/*
 * A batch mixing single-token decode and longer (prefill / multi-token)
 * segments over one paged cache, as MATE's planner splits a batch at the first
 * sequence whose query length passes a threshold and runs a decode plan and a
 * prefill plan.  Here the threshold is one token: the leading sequences with
 * q_len == 1 run through the decode kernel (split-KV, merged), every sequence
 * from the first q_len > 1 on runs through the prefill kernel (which also takes
 * q_len == 1 rows).  Queries, outputs and lse stay in one ragged layout.
 *
 * pa_get_mixed_plan (host): cu_seqlens_q_host int32 [B+1], kv_lens_host int32 [B]
 * (keys per sequence, new tokens included, already in the cache),
 * block_table_host int32 [B, max_pages] or NULL; fills plan and writes the decode
 * part's metadata to meta_host (NULL: size only; PA_ERR_WORKSPACE if
 * meta_capacity_ints < plan->decode.meta_ints).
 *
 * pa_mixed (device): q bf16 [total_q, Hq, D]; pools [P, Hk, 64, D];
 * block_table [B, max_pages]; cu_seqlens_q [B+1]; cu_seqlens_k [B+1] (running
 * offsets of kv_lens); kv_lens [B]; meta_dev = the uploaded metadata; causal
 * rows see keys j <= kv_len - q_len + i; out bf16 [total_q, Hq, D]; lse fp32
 * [total_q, Hq] or NULL; workspace >= plan->workspace_bytes, zero-filled once.
 */
pa_status pa_get_mixed_plan(const int32_t* cu_seqlens_q_host, const int32_t* kv_lens_host,
                        const int32_t* block_table_host, const pa_mixed_shapes* shapes, int32_t* meta_host,
                        size_t meta_capacity_ints, pa_mixed_plan* plan);

pa_status pa_mixed(const pa_mixed_shapes* shapes, const pa_mixed_plan* plan, const void* q, const void* k_pool,
                   const void* v_pool, const int32_t* block_table, const int32_t* cu_seqlens_q,
                   const int32_t* cu_seqlens_k, const int32_t* kv_lens, const int32_t* meta_dev, float scale,
                   void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ----------------------------------------------------------------- append */

typedef struct {
    int32_t batch;             /* B sequences */
    int32_t num_kv_heads;      /* Hk */
    int32_t head_dim;          /* D: 64 or 128 */
    int32_t page_size;         /* must be 64 */
    int32_t max_pages_per_seq; /* block_table row stride */
    int32_t num_pool_pages;
    int32_t total_new;         /* cu_seqlens_new[B] */
    int32_t kv_dtype;          /* pa_kv_dtype of the pools */
} pa_append_shapes;

/*
 * pa_append_kv -- write new tokens' keys and values into their pages, the
 * step before a chunked prefill ("prefill writes into paged cache", FlashMLA
 * "Tensor Shapes Reference" section 4).  New token i of sequence b goes to
 * logical position p = start_pos[b] + i: row p % 64 of page
 * block_table[b, p / 64] ("Prefill to Cache Mapping").
 *
 *   k_new, v_new    bf16 [total_new, Hk, D] (fp16 for fp16 pools), ragged by cu_seqlens_new
 *   cu_seqlens_new  int32 [B+1] running offsets of the new tokens
 *   start_pos       int32 [B] position of each sequence's first new token (the
 *                   number of tokens already cached)
 *   block_table     int32 [B, max_pages_per_seq]; must already list the pages
 *                   that the new positions fall in
 *   k_pool, v_pool  [num_pool_pages, Hk, 64, D]: bf16 or fp16 (values copied bit
 *                   for bit), or e4m3 with k_scale / v_scale fp32 [Hk]: the stored
 *                   code is e4m3(x / scale) in fp32, nearest even, saturating
 *   workspace       >= PA_STATUS_BYTES (status word)
 * A position outside the block table or a page id outside the pool is skipped
 * and recorded as PA_ERR_DEVICE_BOUNDS.  Rows of different calls or tokens
 * must not collide (two writers to one row race).
 */
pa_status pa_append_kv(const pa_append_shapes* shapes, const void* k_new, const void* v_new,
                       const int32_t* cu_seqlens_new, const int32_t* start_pos, const int32_t* block_table,
                       void* k_pool, void* v_pool, const float* k_scale, const float* v_scale, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/* ----------------------------------------------------------------- status */

/*
 * Synchronise `stream`, read the status word at the start of `workspace`
 * (device), clear it, and return what the kernels recorded (PA_OK if nothing).
 * The first fault recorded since the last check wins.
 */
pa_status pa_check_status(void* workspace, cudaStream_t stream);

/* Message describing the last non-OK status returned on this host thread. */
const char* pa_last_error(void);

/* Time limit, in nanoseconds, of every device-side wait in launches made after
 * this call (default 2e9).  Process-wide. */
pa_status pa_set_wait_limit_ns(uint64_t limit_ns);

/* Form of the bf16 / fp16 pa_prefill for calls made after this one
 * (process-wide): enable = 0, the default, runs one CTA per 256-row work item
 * on the tensor cores of its SM; enable != 0 runs CTA pairs (cta_group::2,
 * M = 256 over two SMs, 512-row work items).  Both compute the same result
 * within the stated tolerances; the pair form is slower on the measured
 * workloads and kept for comparison.  The e4m3 MLA entry points are not
 * affected.  Always returns PA_OK; falls back to the one-CTA form where no
 * cluster of two CTAs fits. */
pa_status pa_set_prefill_cta_pairs(int enable);

/*
 * Test hook for failure detection: launch one CTA that waits, with the time
 * limit given, on a barrier that nothing arrives on, then records
 * PA_ERR_TIMEOUT in the status word and returns.  The context stays usable.
 */
pa_status pa_debug_wait_timeout(void* workspace, uint64_t limit_ns, cudaStream_t stream);

/* Library version, e.g. 100 for 0.1.0. */
int32_t pa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
