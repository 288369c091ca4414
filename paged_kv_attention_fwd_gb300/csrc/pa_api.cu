// pa_api.cu -- host side of libpa: argument validation, the split-KV
// scheduler (pa_get_metadata), tensor-map construction and kernel launches.
// Nothing here allocates device memory or synchronises a stream, except
// pa_check_status, whose job is to synchronise and read the status word.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "pa_internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
// pa_prefill's bf16 / fp16 form: 0 one CTA per 256-row work item (default),
// 1 CTA pairs on 512-row items (prefill_pair.cu)
std::atomic<int> g_prefill_cta_pairs{0};

pa_status fail(pa_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ tensor maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tiled map over a bf16 tensor of `rank` dims (innermost first), box of 64
// elements (128 bytes) innermost, 128-byte swizzle.
pa_status make_map(CUtensorMapDataType dtype, CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box);

pa_status make_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                        const uint32_t* box) {
    return make_map(CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, rank, dims, strides_bytes, box);
}

// 16-bit elements: the swizzled layout does not depend on which 16-bit type
pa_status make_map_16(bool f16, CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
    return make_map(f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, map, base, rank, dims,
                    strides_bytes, box);
}

// Encoded tensor maps of recent calls.  A serving loop passes the same
// buffers with the same shapes call after call; a map is a pure function of
// (type, base address, dims, strides, box), so a hit skips the driver's
// encode.  Sixteen entries, replaced round-robin, under one mutex.
struct MapKey {
    CUtensorMapDataType dtype;
    const void* base;
    int rank;
    uint64_t dims[5], strides[4];
    uint32_t box[5];
    bool operator==(const MapKey& o) const {
        if (dtype != o.dtype || base != o.base || rank != o.rank) return false;
        for (int i = 0; i < rank; ++i) {
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
            if (i + 1 < rank && strides[i] != o.strides[i]) return false;
        }
        return true;
    }
};

struct MapCache {
    static constexpr int kEntries = 16;
    std::mutex mu;
    MapKey key[kEntries];
    CUtensorMap map[kEntries];
    bool used[kEntries] = {};
    int next = 0;
};

MapCache& map_cache() {
    static MapCache c;
    return c;
}

// Tiled map, 128-byte swizzle (the box's inner extent is 128 bytes).
pa_status make_map(CUtensorMapDataType dtype, CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box) {
    MapKey key;
    std::memset(&key, 0, sizeof key);
    key.dtype = dtype;
    key.base = base;
    key.rank = rank;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides_bytes[i];
    }
    MapCache& cache = map_cache();
    {
        std::lock_guard<std::mutex> lock(cache.mu);
        for (int i = 0; i < MapCache::kEntries; ++i)
            if (cache.used[i] && cache.key[i] == key) {
                *map = cache.map[i];
                return PA_OK;
            }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = enc(map, dtype, rank, const_cast<void*>(base), d, s, b, e,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    std::lock_guard<std::mutex> lock(cache.mu);
    const int slot = cache.next;
    cache.next = (slot + 1) % MapCache::kEntries;
    cache.key[slot] = key;
    cache.map[slot] = *map;
    cache.used[slot] = true;
    return PA_OK;
}

// ------------------------------------------------------------ scheduler

struct SchedItem {
    int cost, index, b, s, kvh;
};

}  // namespace

namespace pa {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace pa

extern "C" {

int32_t pa_version(void) { return 100; }

const char* pa_last_error(void) { return g_last_error.c_str(); }

pa_status pa_set_wait_limit_ns(uint64_t limit_ns) {
    if (limit_ns == 0) return fail(PA_ERR_INVALID_ARG, "wait limit must be positive");
    g_wait_limit_ns.store(limit_ns);
    return PA_OK;
}

pa_status pa_set_prefill_cta_pairs(int enable) {
    g_prefill_cta_pairs.store(enable != 0 ? 1 : 0);
    return PA_OK;
}

pa_status pa_get_metadata(const int32_t* seq_lens_host, const int32_t* block_table_host, const pa_decode_shapes* sh,
                          int32_t* meta_host, size_t meta_capacity_ints, pa_decode_plan* plan) {
    pa::NvtxRange nvtx_range("pa_get_metadata");
    if (!sh || !plan) return fail(PA_ERR_INVALID_ARG, "shapes and plan must not be NULL");
    const int B = sh->batch, Hk = sh->num_kv_heads;
    if (B < 0) return fail(PA_ERR_INVALID_ARG, "batch must be >= 0 (got %d)", B);
    if (B > 0 && !seq_lens_host) return fail(PA_ERR_INVALID_ARG, "seq_lens_host must not be NULL");
    if (Hk <= 0 || Hk > 65535) return fail(PA_ERR_INVALID_ARG, "num_kv_heads must be in [1, 65535] (got %d)", Hk);
    if (sh->page_size != pa::kPage) return fail(PA_ERR_INVALID_ARG, "page_size must be 64 (got %d)", sh->page_size);
    if (sh->max_pages_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_pages_per_seq must be positive");
    if (sh->num_sms <= 0) return fail(PA_ERR_INVALID_ARG, "num_sms must be positive (got %d)", sh->num_sms);
    if (sh->ctas_per_sm < 0) return fail(PA_ERR_INVALID_ARG, "ctas_per_sm must be >= 0");
    if (sh->forced_splits < 0) return fail(PA_ERR_INVALID_ARG, "forced_splits must be >= 0");
    const int cps = sh->ctas_per_sm == 0 ? 1 : sh->ctas_per_sm;

    std::vector<int> pages(B);
    int64_t units = 0;
    for (int b = 0; b < B; ++b) {
        const int len = seq_lens_host[b];
        if (len < 0) return fail(PA_ERR_INVALID_ARG, "seq_lens[%d] = %d is negative", b, len);
        if ((int64_t)len > (int64_t)sh->max_pages_per_seq * pa::kPage)
            return fail(PA_ERR_INVALID_ARG, "seq_lens[%d] = %d exceeds max_pages_per_seq * 64 = %lld", b, len,
                        (long long)sh->max_pages_per_seq * pa::kPage);
        pages[b] = (int)cdiv(len, pa::kPage);
        units += (int64_t)pages[b] * Hk;
        if (block_table_host) {
            for (int p = 0; p < pages[b]; ++p) {
                const int32_t id = block_table_host[(int64_t)b * sh->max_pages_per_seq + p];
                if (id < 0 || id >= sh->num_pool_pages)
                    return fail(PA_ERR_INVALID_ARG, "block_table[%d, %d] = %d is outside [0, %d)", b, p, id,
                                sh->num_pool_pages);
            }
        }
    }
    const int64_t cap = (int64_t)sh->num_sms * cps;
    const int64_t chunk = std::max<int64_t>(4, cdiv(units, 2 * cap));  // two items per CTA share
    std::vector<int32_t> nsplit(B), indptr(B + 1, 0);
    for (int b = 0; b < B; ++b) {
        int n;
        if (pages[b] <= 1) n = 1;
        else if (sh->forced_splits > 0) n = std::min({sh->forced_splits, pages[b], PA_MAX_SPLITS});
        else n = (int)std::min<int64_t>(cdiv(pages[b], chunk), PA_MAX_SPLITS);
        nsplit[b] = n;
        indptr[b + 1] = indptr[b] + n;
    }
    const int64_t total_splits = indptr[B];
    std::vector<SchedItem> items;
    items.reserve((size_t)total_splits * Hk);
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < nsplit[b]; ++s) {
            const int lo = (int)((int64_t)s * pages[b] / nsplit[b]);
            const int hi = (int)((int64_t)(s + 1) * pages[b] / nsplit[b]);
            for (int g = 0; g < Hk; ++g) items.push_back({hi - lo + 1, (int)items.size(), b, s, g});
        }
    const int64_t nitems = (int64_t)items.size();
    const int64_t grid = std::min<int64_t>(nitems, cap);
    const int64_t meta_ints = pa::kMetaHeader + 2 * (int64_t)B + 1 + grid + 1 + 2 * nitems;
    if (meta_ints > INT32_MAX) return fail(PA_ERR_UNSUPPORTED, "metadata would exceed 2^31 entries");

    plan->total_splits = (int32_t)total_splits;
    plan->num_items = (int32_t)nitems;
    plan->grid = (int32_t)grid;
    plan->meta_ints = (int32_t)meta_ints;
    plan->ctas_per_sm = cps;
    plan->reserved = 0;
    const int64_t hq = std::max(sh->num_q_heads, 0), d = std::max(sh->head_dim, 0);
    plan->workspace_bytes = (size_t)PA_STATUS_BYTES + (size_t)(total_splits * hq * d * 4) +
                            (size_t)(((total_splits * hq * 4) + 255) / 256 * 256) +
                            (size_t)((((int64_t)B * Hk * 4) + 255) / 256 * 256);
    if (!meta_host) return PA_OK;
    if (meta_capacity_ints < (size_t)meta_ints)
        return fail(PA_ERR_WORKSPACE, "metadata needs %lld int32 entries, capacity is %zu", (long long)meta_ints,
                    meta_capacity_ints);

    // longest first; each to the least-loaded CTA, ties to the lowest index
    std::vector<SchedItem> order(items);
    std::stable_sort(order.begin(), order.end(), [](const SchedItem& x, const SchedItem& y) {
        return x.cost != y.cost ? x.cost > y.cost : x.index < y.index;
    });
    typedef std::pair<int64_t, int32_t> Load;  // (load, cta)
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int32_t c = 0; c < grid; ++c) heap.push({0, c});
    std::vector<std::vector<int32_t>> per_cta(grid);
    for (const SchedItem& it : order) {
        Load l = heap.top();
        heap.pop();
        per_cta[l.second].push_back(it.index);
        heap.push({l.first + it.cost, l.second});
    }
    int32_t* m = meta_host;
    m[0] = pa::kMetaMagic;
    m[1] = B;
    m[2] = Hk;
    m[3] = (int32_t)total_splits;
    m[4] = (int32_t)nitems;
    m[5] = (int32_t)grid;
    m[6] = (int32_t)std::min<int64_t>(chunk, INT32_MAX);
    m[7] = cps;
    int64_t o = pa::kMetaHeader;
    for (int b = 0; b < B; ++b) m[o++] = nsplit[b];
    for (int b = 0; b <= B; ++b) m[o++] = indptr[b];
    int32_t acc = 0;
    m[o++] = 0;
    for (int64_t c = 0; c < grid; ++c) {
        acc += (int32_t)per_cta[c].size();
        m[o++] = acc;
    }
    for (int64_t c = 0; c < grid; ++c)
        for (int32_t idx : per_cta[c]) {
            const SchedItem& it = items[idx];
            m[o++] = it.b;
            m[o++] = (it.s << 16) | it.kvh;
        }
    return PA_OK;
}

namespace {

pa_status validate_decode_common(const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* out,
                                 const void* meta_dev, const void* workspace, size_t workspace_bytes) {
    if (!sh || !plan) return fail(PA_ERR_INVALID_ARG, "shapes and plan must not be NULL");
    const int B = sh->batch, Hq = sh->num_q_heads, Hk = sh->num_kv_heads, D = sh->head_dim;
    if (B < 0) return fail(PA_ERR_INVALID_ARG, "batch must be >= 0");
    if (B == 0) return PA_OK;
    if (Hq <= 0 || Hk <= 0 || Hq % Hk != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", Hq, Hk);
    if (Hq / Hk > PA_MAX_GROUP)
        return fail(PA_ERR_UNSUPPORTED, "Hq / Hk = %d exceeds the supported group size %d", Hq / Hk, PA_MAX_GROUP);
    if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", D);
    if (sh->page_size != pa::kPage) return fail(PA_ERR_INVALID_ARG, "page_size must be 64 (got %d)", sh->page_size);
    if (!out || !meta_dev || !workspace) return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(out) || !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARG, "q, pools, out and workspace must be 16-byte aligned");
    if (plan->grid <= 0 || plan->total_splits < B || plan->meta_ints <= 0)
        return fail(PA_ERR_INVALID_ARG, "plan does not come from pa_get_metadata for this batch");
    if (workspace_bytes < plan->workspace_bytes)
        return fail(PA_ERR_WORKSPACE, "workspace has %zu bytes, the plan needs %zu", workspace_bytes,
                    plan->workspace_bytes);
    return PA_OK;
}

float* partial_o(void* workspace) {
    return reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + PA_STATUS_BYTES);
}

}  // namespace

namespace {
pa_status decode_launch(bool fused, const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* q,
                        const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev, float scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);
}

pa_status pa_decode_attend(const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* q,
                           const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                           const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev,
                           float scale, void* out, float* lse, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_decode_attend");
    return decode_launch(false, sh, plan, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, meta_dev,
                         scale, out, lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace pa {
// Every host-side check of a decode call (shapes, plan, pointers, alignment,
// workspace size, scale), without launching anything.
pa_status check_decode_call(const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* q,
                            const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev,
                            float scale, const void* out, const void* workspace, size_t workspace_bytes) {
    pa_status st = validate_decode_common(sh, plan, out, meta_dev, workspace, workspace_bytes);
    if (st != PA_OK || sh->batch == 0) return st;
    const int Hk = sh->num_kv_heads;
    if (sh->kv_dtype != PA_KV_BF16 && sh->kv_dtype != PA_KV_FP8_E4M3 && sh->kv_dtype != PA_KV_FP16)
        return fail(PA_ERR_INVALID_ARG, "unknown kv_dtype %d", sh->kv_dtype);
    const bool fp8 = sh->kv_dtype == PA_KV_FP8_E4M3;
    if (sh->max_pages_per_seq <= 0 || sh->num_pool_pages <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_pages_per_seq and num_pool_pages must be positive");
    if ((int64_t)sh->num_pool_pages * Hk * pa::kPage >= ((int64_t)1 << 31))
        return fail(PA_ERR_UNSUPPORTED, "pool rows (pages * Hk * 64) must be below 2^31");
    if (!q || !k_pool || !v_pool || !block_table || !seq_lens)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (fp8 && (!k_scale || !v_scale)) return fail(PA_ERR_INVALID_ARG, "e4m3 KV needs k_scale and v_scale");
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return fail(PA_ERR_INVALID_ARG, "q, pools, out and workspace must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale must be finite");
    return PA_OK;
}
}  // namespace pa

extern "C" {

namespace {
pa_status decode_launch(bool fused, const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* q,
                        const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                        const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev, float scale,
                        void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    pa_status st = pa::check_decode_call(sh, plan, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens,
                                         meta_dev, scale, out, workspace, workspace_bytes);
    if (st != PA_OK || sh->batch == 0) return st;
    const int B = sh->batch, Hq = sh->num_q_heads, Hk = sh->num_kv_heads, D = sh->head_dim;
    const bool fp8 = sh->kv_dtype == PA_KV_FP8_E4M3;
    const bool f16 = sh->kv_dtype == PA_KV_FP16;

    pa::DecodeArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.k_pool = static_cast<const uint8_t*>(k_pool);
    a.v_pool = static_cast<const uint8_t*>(v_pool);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.meta = meta_dev;
    a.out = static_cast<uint16_t*>(out);
    a.lse = lse;
    a.status = static_cast<int*>(workspace);
    a.o_part = partial_o(workspace);
    a.lse_part = a.o_part + (size_t)plan->total_splits * Hq * D;
    {
        const size_t lse_bytes = ((size_t)plan->total_splits * Hq * 4 + 255) / 256 * 256;
        int* ctr = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(a.lse_part) + lse_bytes);
        const size_t need = PA_STATUS_BYTES + (size_t)plan->total_splits * Hq * D * 4 + lse_bytes + (size_t)B * Hk * 4;
        a.counters = (fused && plan->total_splits > B && workspace_bytes >= need) ? ctr : nullptr;
    }
    a.batch = B;
    a.num_q_heads = Hq;
    a.num_kv_heads = Hk;
    a.group = Hq / Hk;
    a.max_pages = sh->max_pages_per_seq;
    a.num_pool_pages = sh->num_pool_pages;
    a.f16 = f16;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.wait_ns = g_wait_limit_ns.load();

    CUtensorMap mk, mv, mq;
    std::memset(&mk, 0, sizeof mk);
    std::memset(&mv, 0, sizeof mv);
    std::memset(&mq, 0, sizeof mq);
    if (!fp8) {
        const uint64_t dims[2] = {(uint64_t)D, (uint64_t)sh->num_pool_pages * Hk * pa::kPage};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64, 64};
        st = make_map_16(f16, &mk, k_pool, 2, dims, strides, box);
        if (st != PA_OK) return st;
        st = make_map_16(f16, &mv, v_pool, 2, dims, strides, box);
        if (st != PA_OK) return st;
        // query rows [B * Hq, D]; one box = the G heads of one KV group
        const uint64_t qdims[2] = {(uint64_t)D, (uint64_t)B * Hq};
        const uint32_t qbox[2] = {64, (uint32_t)(Hq / Hk)};
        st = make_map_16(f16, &mq, q, 2, qdims, strides, qbox);
        if (st != PA_OK) return st;
    } else if (D == 128) {
        // e4m3 pages: one 128-byte row per key, one box per 64-row page slab
        const uint64_t dims[2] = {128, (uint64_t)sh->num_pool_pages * Hk * pa::kPage};
        const uint64_t strides[1] = {128};
        const uint32_t box[2] = {128, 64};
        st = make_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, &mk, k_pool, 2, dims, strides, box);
        if (st != PA_OK) return st;
        st = make_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, &mv, v_pool, 2, dims, strides, box);
        if (st != PA_OK) return st;
    }
    cudaError_t e = pa::launch_decode(D, fp8, a, &mk, &mv, &mq, plan->grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    if (fused && plan->total_splits > B && !a.counters) {
        // no room for the arrival counters: merge in a second kernel
        return pa_decode_combine(sh, plan, meta_dev, out, lse, workspace, workspace_bytes, stream);
    }
    return PA_OK;
}
}  // namespace

pa_status pa_decode_combine(const pa_decode_shapes* sh, const pa_decode_plan* plan, const int32_t* meta_dev,
                            void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_decode_combine");
    pa_status st = validate_decode_common(sh, plan, out, meta_dev, workspace, workspace_bytes);
    if (st != PA_OK || sh->batch == 0) return st;
    if (plan->total_splits == sh->batch) return PA_OK;
    pa::CombineArgs c;
    c.meta = meta_dev;
    c.o_part = partial_o(workspace);
    c.lse_part = c.o_part + (size_t)plan->total_splits * sh->num_q_heads * sh->head_dim;
    c.out = static_cast<uint16_t*>(out);
    c.lse = lse;
    c.batch = sh->batch;
    c.num_q_heads = sh->num_q_heads;
    c.head_dim = sh->head_dim;
    c.f16 = sh->kv_dtype == PA_KV_FP16;
    cudaError_t e = pa::launch_combine(c, stream);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return PA_OK;
}

pa_status pa_decode(const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* q, const void* k_pool,
                    const void* v_pool, const float* k_scale, const float* v_scale, const int32_t* block_table,
                    const int32_t* seq_lens, const int32_t* meta_dev, float scale, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_decode");
    return decode_launch(true, sh, plan, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, meta_dev,
                         scale, out, lse, workspace, workspace_bytes, stream);
}

namespace {
// The launch arguments common to pa_prefill and pa_prefill_mla_fp8.
pa_status fill_prefill_args(const pa_prefill_shapes* sh, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            const int32_t* block_table, const int32_t* qo_offset, int causal, float scale, void* out,
                            float* lse, void* workspace, size_t workspace_bytes, bool f16, pa::PrefillArgs* a) {
    const int B = sh->batch, Hq = sh->num_q_heads, Hk = sh->num_kv_heads;
    const bool paged = block_table != nullptr;
    const bool rope = sh->rope_dim != 0;
    a->cu_q = cu_seqlens_q;
    a->cu_k = cu_seqlens_k;
    a->block_table = block_table;
    a->qo_offset = qo_offset;
    a->out = static_cast<uint16_t*>(out);
    a->lse = lse;
    a->status = static_cast<int*>(workspace);
    a->batch = B;
    a->num_q_heads = Hq;
    a->num_kv_heads = Hk;
    a->group = Hq / Hk;
    a->max_pages = paged ? sh->max_pages_per_seq : 0;
    a->num_pool_pages = paged ? sh->num_pool_pages : 0;
    a->total_q = sh->total_q;
    a->q_block = 256;
    a->num_q_tiles = (int32_t)cdiv(sh->max_seqlen_q, 256);
    // the longest-first unit order lives after the status word when the
    // workspace has room for it (see pa_prefill_workspace_size)
    const int64_t units = (int64_t)a->num_q_tiles * B;
    if (units > 65535) return fail(PA_ERR_UNSUPPORTED, "batch * ceil(max_seqlen_q / 256) must be <= 65535");
    a->order = (units <= 4096 && workspace_bytes >= PA_STATUS_BYTES + (size_t)units * 4)
                  ? reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(workspace) + PA_STATUS_BYTES)
                  : nullptr;
    a->causal = causal != 0;
    a->paged = paged;
    a->rope = rope;
    a->f16 = f16;
    a->scale_log2 = scale * 1.4426950408889634f;
    a->wait_ns = g_wait_limit_ns.load();
    a->f8 = 0;
    a->r8 = 0;
    a->q_scale = nullptr;
    a->k_scale = nullptr;
    return PA_OK;
}
}  // namespace

pa_status pa_prefill(const pa_prefill_shapes* sh, const void* q, const void* k, const void* v, const void* k_rope,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* block_table,
                     const int32_t* qo_offset, int causal, float scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_prefill");
    if (!sh) return fail(PA_ERR_INVALID_ARG, "shapes must not be NULL");
    const int B = sh->batch, Hq = sh->num_q_heads, Hk = sh->num_kv_heads;
    if (B < 0 || sh->total_q < 0 || sh->total_k < 0 || sh->max_seqlen_q < 0)
        return fail(PA_ERR_INVALID_ARG, "batch, total_q, total_k and max_seqlen_q must be >= 0");
    if (B == 0 || sh->total_q == 0 || sh->max_seqlen_q == 0) return PA_OK;
    if (Hq <= 0 || Hk <= 0 || Hq % Hk != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", Hq, Hk);
    if (Hq > 65535) return fail(PA_ERR_UNSUPPORTED, "num_q_heads above 65535");
    if (sh->dtype != PA_KV_BF16 && sh->dtype != PA_KV_FP16)
        return fail(PA_ERR_UNSUPPORTED, "prefill dtype must be PA_KV_BF16 or PA_KV_FP16 (got %d)", sh->dtype);
    const bool f16 = sh->dtype == PA_KV_FP16;
    const bool paged = block_table != nullptr;
    const bool rope = sh->rope_dim != 0;
    if (sh->head_dim_v != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim_v must be 128 (got %d)", sh->head_dim_v);
    if (!((sh->head_dim_qk == 128 && sh->rope_dim == 0) || (sh->head_dim_qk == 192 && sh->rope_dim == 64)))
        return fail(PA_ERR_UNSUPPORTED, "head_dim_qk / rope_dim must be 128 / 0 or 192 / 64 (got %d / %d)",
                    sh->head_dim_qk, sh->rope_dim);
    if (rope && paged) return fail(PA_ERR_UNSUPPORTED, "a shared rope key is supported with ragged keys only");
    if (rope && !k_rope) return fail(PA_ERR_INVALID_ARG, "rope_dim 64 needs k_rope");
    if (!rope && k_rope) return fail(PA_ERR_INVALID_ARG, "k_rope given but rope_dim is 0");
    if (paged) {
        if (sh->page_size != pa::kPage) return fail(PA_ERR_INVALID_ARG, "page_size must be 64 (got %d)", sh->page_size);
        if (sh->max_pages_per_seq <= 0 || sh->num_pool_pages <= 0)
            return fail(PA_ERR_INVALID_ARG, "paged keys need max_pages_per_seq and num_pool_pages > 0");
        if ((int64_t)sh->num_pool_pages * Hk * pa::kPage >= ((int64_t)1 << 31))
            return fail(PA_ERR_UNSUPPORTED, "pool rows (pages * Hk * 64) must be below 2^31");
    } else if (sh->total_k <= 0) {
        return fail(PA_ERR_INVALID_ARG, "ragged keys need total_k > 0");
    }
    if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out || !workspace)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (k_rope && !aligned16(k_rope)) ||
        !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARG, "q, k, v, k_rope, out and workspace must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale must be finite");
    if (workspace_bytes < PA_STATUS_BYTES)
        return fail(PA_ERR_WORKSPACE, "workspace needs %d bytes, got %zu", PA_STATUS_BYTES, workspace_bytes);

    const int dqk = sh->head_dim_qk, dk = dqk - sh->rope_dim;
    pa_status st = PA_OK;
    CUtensorMap mq, mk, mv, mr;
    std::memset(&mr, 0, sizeof mr);
    {
        const uint64_t dims[3] = {(uint64_t)dqk, (uint64_t)Hq, (uint64_t)sh->total_q};
        const uint64_t strides[2] = {(uint64_t)dqk * 2, (uint64_t)Hq * dqk * 2};
        const uint32_t box[3] = {64, 1, 128};
        pa_status st = make_map_16(f16, &mq, q, 3, dims, strides, box);
        if (st != PA_OK) return st;
    }
    if (paged) {
        const uint64_t dims[2] = {128, (uint64_t)sh->num_pool_pages * Hk * pa::kPage};
        const uint64_t strides[1] = {256};
        const uint32_t box[2] = {64, 64};
        pa_status st = make_map_16(f16, &mk, k, 2, dims, strides, box);
        if (st == PA_OK) st = make_map_16(f16, &mv, v, 2, dims, strides, box);
        if (st != PA_OK) return st;
    } else {
        const uint64_t dk_dims[3] = {(uint64_t)dk, (uint64_t)Hk, (uint64_t)sh->total_k};
        const uint64_t dk_str[2] = {(uint64_t)dk * 2, (uint64_t)Hk * dk * 2};
        const uint64_t dv_dims[3] = {128, (uint64_t)Hk, (uint64_t)sh->total_k};
        const uint64_t dv_str[2] = {256, (uint64_t)Hk * 256};
        const uint32_t box[3] = {64, 1, 128};
        pa_status st = make_map_16(f16, &mk, k, 3, dk_dims, dk_str, box);
        if (st == PA_OK) st = make_map_16(f16, &mv, v, 3, dv_dims, dv_str, box);
        if (st == PA_OK && rope) {
            const uint64_t rd[2] = {64, (uint64_t)sh->total_k};
            const uint64_t rs[1] = {128};
            const uint32_t rb[2] = {64, 128};
            st = make_map_16(f16, &mr, k_rope, 2, rd, rs, rb);
        }
        if (st != PA_OK) return st;
    }
    pa::PrefillArgs a;
    st = fill_prefill_args(sh, cu_seqlens_q, cu_seqlens_k, block_table, qo_offset, causal, scale, out, lse, workspace,
                           workspace_bytes, f16, &a);
    if (st != PA_OK) return st;
    if (g_prefill_cta_pairs.load() != 0) {
        // CTA pairs (512-row work items); each CTA loads 64 keys of a K tile,
        // so the ragged K and rope maps take 64-row boxes
        pa::PrefillArgs ap = a;
        ap.q_block = 512;
        ap.num_q_tiles = (int32_t)cdiv(sh->max_seqlen_q, 512);
        CUtensorMap mk2 = mk, mr2 = mr;
        if (!paged) {
            const uint64_t dk_dims[3] = {(uint64_t)dk, (uint64_t)Hk, (uint64_t)sh->total_k};
            const uint64_t dk_str[2] = {(uint64_t)dk * 2, (uint64_t)Hk * dk * 2};
            const uint32_t box[3] = {64, 1, 64};
            st = make_map_16(f16, &mk2, k, 3, dk_dims, dk_str, box);
            if (st == PA_OK && rope) {
                const uint64_t rd[2] = {64, (uint64_t)sh->total_k};
                const uint64_t rs[1] = {128};
                const uint32_t rb[2] = {64, 64};
                st = make_map_16(f16, &mr2, k_rope, 2, rd, rs, rb);
            }
            if (st != PA_OK) return st;
        }
        cudaError_t e = pa::launch_prefill_pair(ap, dqk, &mq, &mk2, &mv, &mr2, stream);
        if (e == cudaSuccess) return PA_OK;
        if (e != cudaErrorNotSupported) return cuda_fail(e, "prefill launch");
        // no cluster of two CTAs fits on this device: one CTA per work item
    }
    CUtensorMap mqr;
    std::memset(&mqr, 0, sizeof mqr);
    cudaError_t e = pa::launch_prefill(a, dqk, &mq, &mk, &mv, &mr, &mqr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PA_OK;
}

pa_status pa_append_kv(const pa_append_shapes* sh, const void* k_new, const void* v_new,
                       const int32_t* cu_seqlens_new, const int32_t* start_pos, const int32_t* block_table,
                       void* k_pool, void* v_pool, const float* k_scale, const float* v_scale, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_append_kv");
    if (!sh) return fail(PA_ERR_INVALID_ARG, "shapes must not be NULL");
    if (sh->batch < 0 || sh->total_new < 0) return fail(PA_ERR_INVALID_ARG, "batch and total_new must be >= 0");
    if (sh->batch == 0 || sh->total_new == 0) return PA_OK;
    if (sh->num_kv_heads <= 0 || sh->num_kv_heads > 65535)
        return fail(PA_ERR_INVALID_ARG, "num_kv_heads must be in [1, 65535] (got %d)", sh->num_kv_heads);
    if (sh->head_dim != 64 && sh->head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64 or 128 (got %d)", sh->head_dim);
    if (sh->page_size != pa::kPage) return fail(PA_ERR_INVALID_ARG, "page_size must be 64 (got %d)", sh->page_size);
    if (sh->max_pages_per_seq <= 0 || sh->num_pool_pages <= 0)
        return fail(PA_ERR_INVALID_ARG, "max_pages_per_seq and num_pool_pages must be positive");
    if (sh->kv_dtype != PA_KV_BF16 && sh->kv_dtype != PA_KV_FP8_E4M3 && sh->kv_dtype != PA_KV_FP16)
        return fail(PA_ERR_INVALID_ARG, "unknown kv_dtype %d", sh->kv_dtype);
    const bool fp8 = sh->kv_dtype == PA_KV_FP8_E4M3;
    if (!k_new || !v_new || !cu_seqlens_new || !start_pos || !block_table || !k_pool || !v_pool || !workspace)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (fp8 && (!k_scale || !v_scale)) return fail(PA_ERR_INVALID_ARG, "e4m3 pools need k_scale and v_scale");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return fail(PA_ERR_INVALID_ARG, "k_new, v_new and the pools must be 16-byte aligned");
    if (workspace_bytes < PA_STATUS_BYTES)
        return fail(PA_ERR_WORKSPACE, "workspace needs %d bytes, got %zu", PA_STATUS_BYTES, workspace_bytes);
    pa::AppendArgs a;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.cu_new = cu_seqlens_new;
    a.start_pos = start_pos;
    a.block_table = block_table;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.status = static_cast<int*>(workspace);
    a.batch = sh->batch;
    a.num_kv_heads = sh->num_kv_heads;
    a.head_dim = sh->head_dim;
    a.max_pages = sh->max_pages_per_seq;
    a.num_pool_pages = sh->num_pool_pages;
    a.total_new = sh->total_new;
    a.fp8 = fp8;
    cudaError_t e = pa::launch_append(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return PA_OK;
}

namespace {
pa_decode_shapes mixed_decode_shapes(const pa_mixed_shapes* sh, int num_decode) {
    pa_decode_shapes d;
    d.batch = num_decode;
    d.num_q_heads = sh->num_q_heads;
    d.num_kv_heads = sh->num_kv_heads;
    d.head_dim = sh->head_dim;
    d.page_size = sh->page_size;
    d.max_pages_per_seq = sh->max_pages_per_seq;
    d.num_pool_pages = sh->num_pool_pages;
    d.kv_dtype = sh->kv_dtype;
    d.num_sms = sh->num_sms;
    d.ctas_per_sm = sh->ctas_per_sm;
    d.forced_splits = sh->forced_splits;
    return d;
}

pa_prefill_shapes mixed_prefill_shapes(const pa_mixed_shapes* sh, const pa_mixed_plan* plan) {
    pa_prefill_shapes p;
    p.batch = sh->batch - plan->num_decode;
    p.num_q_heads = sh->num_q_heads;
    p.num_kv_heads = sh->num_kv_heads;
    p.head_dim_qk = sh->head_dim;
    p.head_dim_v = sh->head_dim;
    p.rope_dim = 0;
    p.max_seqlen_q = plan->max_seqlen_q;
    p.total_q = plan->total_q;
    p.total_k = 0;
    p.page_size = sh->page_size;
    p.max_pages_per_seq = sh->max_pages_per_seq;
    p.num_pool_pages = sh->num_pool_pages;
    p.num_sms = sh->num_sms;
    p.dtype = sh->kv_dtype;
    return p;
}
}  // namespace

pa_status pa_get_mixed_plan(const int32_t* cu_q, const int32_t* kv_lens, const int32_t* block_table_host,
                        const pa_mixed_shapes* sh, int32_t* meta_host, size_t meta_capacity_ints,
                        pa_mixed_plan* plan) {
    pa::NvtxRange nvtx_range("pa_get_mixed_plan");
    if (!sh || !plan) return fail(PA_ERR_INVALID_ARG, "shapes and plan must not be NULL");
    const int B = sh->batch;
    if (B < 0) return fail(PA_ERR_INVALID_ARG, "batch must be >= 0");
    if (B > 0 && (!cu_q || !kv_lens)) return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q_host and kv_lens_host are needed");
    if (sh->head_dim != 128) return fail(PA_ERR_UNSUPPORTED, "mixed batches need head_dim 128 (got %d)", sh->head_dim);
    if (sh->kv_dtype != PA_KV_BF16 && sh->kv_dtype != PA_KV_FP16)
        return fail(PA_ERR_UNSUPPORTED, "mixed batches need bf16 or fp16 pools (kv_dtype %d)", sh->kv_dtype);
    std::memset(plan, 0, sizeof *plan);
    int nd = 0;
    while (nd < B && cu_q[nd + 1] - cu_q[nd] == 1) ++nd;
    int maxq = 0;
    for (int b = 0; b < B; ++b) {
        const int ql = cu_q[b + 1] - cu_q[b];
        if (ql < 0) return fail(PA_ERR_INVALID_ARG, "cu_seqlens_q must not decrease (at %d)", b);
        if (ql > kv_lens[b])
            return fail(PA_ERR_INVALID_ARG, "sequence %d has %d query tokens but only %d keys", b, ql, kv_lens[b]);
        if (b >= nd) maxq = std::max(maxq, ql);
    }
    plan->num_decode = nd;
    plan->total_q = B > 0 ? cu_q[B] : 0;
    plan->max_seqlen_q = maxq;
    size_t dec_ws = 0;
    if (nd > 0) {
        pa_decode_shapes d = mixed_decode_shapes(sh, nd);
        pa_status st = pa_get_metadata(kv_lens, block_table_host, &d, meta_host, meta_capacity_ints, &plan->decode);
        if (st != PA_OK && !(st == PA_ERR_WORKSPACE && !meta_host)) return st;
        dec_ws = (plan->decode.workspace_bytes + 255) / 256 * 256;
    }
    pa_prefill_shapes p = mixed_prefill_shapes(sh, plan);
    const size_t pre_ws = B - nd > 0 ? pa_prefill_workspace_size(&p) : PA_STATUS_BYTES;
    plan->workspace_bytes = dec_ws + pre_ws;
    if (block_table_host && B - nd > 0) {
        for (int b = nd; b < B; ++b) {
            if ((int64_t)kv_lens[b] > (int64_t)sh->max_pages_per_seq * pa::kPage)
                return fail(PA_ERR_INVALID_ARG, "kv_lens[%d] exceeds max_pages_per_seq * 64", b);
            for (int j = 0; j < (kv_lens[b] + pa::kPage - 1) / pa::kPage; ++j) {
                const int32_t id = block_table_host[(int64_t)b * sh->max_pages_per_seq + j];
                if (id < 0 || id >= sh->num_pool_pages)
                    return fail(PA_ERR_INVALID_ARG, "block_table[%d, %d] = %d is outside [0, %d)", b, j, id,
                                sh->num_pool_pages);
            }
        }
    }
    return PA_OK;
}

pa_status pa_mixed(const pa_mixed_shapes* sh, const pa_mixed_plan* plan, const void* q, const void* k_pool,
                   const void* v_pool, const int32_t* block_table, const int32_t* cu_seqlens_q,
                   const int32_t* cu_seqlens_k, const int32_t* kv_lens, const int32_t* meta_dev, float scale,
                   void* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_mixed");
    if (!sh || !plan) return fail(PA_ERR_INVALID_ARG, "shapes and plan must not be NULL");
    if (workspace_bytes < plan->workspace_bytes)
        return fail(PA_ERR_WORKSPACE, "workspace has %zu bytes, the plan needs %zu", workspace_bytes,
                    plan->workspace_bytes);
    if (!workspace || !block_table || !cu_seqlens_q || !cu_seqlens_k)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    const int nd = plan->num_decode;
    size_t dec_ws = 0;
    if (nd > 0) {
        pa_decode_shapes d = mixed_decode_shapes(sh, nd);
        dec_ws = (plan->decode.workspace_bytes + 255) / 256 * 256;
        pa_status st = pa_decode(&d, &plan->decode, q, k_pool, v_pool, nullptr, nullptr, block_table, kv_lens,
                                 meta_dev, scale, out, lse, workspace, plan->decode.workspace_bytes, stream);
        if (st != PA_OK) return st;
    }
    if (sh->batch - nd > 0) {
        pa_prefill_shapes p = mixed_prefill_shapes(sh, plan);
        return pa_prefill(&p, q, k_pool, v_pool, nullptr, cu_seqlens_q + nd, cu_seqlens_k + nd,
                          block_table + (size_t)nd * sh->max_pages_per_seq, nullptr, 1, scale, out, lse,
                          static_cast<uint8_t*>(workspace) + dec_ws, workspace_bytes - dec_ws, stream);
    }
    return PA_OK;
}

pa_status pa_prefill_mla_fp8(const pa_prefill_shapes* sh, const void* q_nope, const void* q_rope,
                             const float* q_scale, const void* k_nope, const float* k_scale, const void* v,
                             const void* k_rope, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             const int32_t* qo_offset, int causal, float scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_prefill_mla_fp8");
    if (!sh) return fail(PA_ERR_INVALID_ARG, "shapes must not be NULL");
    const int B = sh->batch, Hq = sh->num_q_heads, Hk = sh->num_kv_heads;
    if (B < 0 || sh->total_q < 0 || sh->total_k < 0 || sh->max_seqlen_q < 0)
        return fail(PA_ERR_INVALID_ARG, "batch, total_q, total_k and max_seqlen_q must be >= 0");
    if (B == 0 || sh->total_q == 0 || sh->max_seqlen_q == 0) return PA_OK;
    if (Hq <= 0 || Hk <= 0 || Hq % Hk != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", Hq, Hk);
    if (Hq > 65535) return fail(PA_ERR_UNSUPPORTED, "num_q_heads above 65535");
    if (sh->dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_INVALID_ARG, "pa_prefill_mla_fp8 needs dtype PA_KV_FP8_E4M3 (got %d)", sh->dtype);
    if (sh->head_dim_qk != 192 || sh->rope_dim != 64 || sh->head_dim_v != 128)
        return fail(PA_ERR_UNSUPPORTED, "pa_prefill_mla_fp8 needs head_dim_qk 192, rope_dim 64, head_dim_v 128");
    if (sh->total_k <= 0) return fail(PA_ERR_INVALID_ARG, "ragged keys need total_k > 0");
    if (!q_nope || !q_rope || !q_scale || !k_nope || !k_scale || !v || !k_rope || !cu_seqlens_q || !cu_seqlens_k ||
        !out || !workspace)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(k_nope) || !aligned16(v) || !aligned16(k_rope) ||
        !aligned16(out) || !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARG, "q_nope, q_rope, k_nope, v, k_rope, out and workspace must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale must be finite");
    if (workspace_bytes < PA_STATUS_BYTES)
        return fail(PA_ERR_WORKSPACE, "workspace needs %d bytes, got %zu", PA_STATUS_BYTES, workspace_bytes);

    CUtensorMap mq, mqr, mk, mv, mr;
    const uint64_t tq = (uint64_t)sh->total_q, tk = (uint64_t)sh->total_k;
    {   // per-head parts: one 128-byte e4m3 row per (token, head)
        const uint64_t qd[3] = {128, (uint64_t)Hq, tq}, qs[2] = {128, (uint64_t)Hq * 128};
        const uint64_t kd[3] = {128, (uint64_t)Hk, tk}, ks[2] = {128, (uint64_t)Hk * 128};
        const uint32_t box[3] = {128, 1, 128};
        pa_status st = make_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, &mq, q_nope, 3, qd, qs, box);
        if (st == PA_OK) st = make_map(CU_TENSOR_MAP_DATA_TYPE_UINT8, &mk, k_nope, 3, kd, ks, box);
        if (st != PA_OK) return st;
    }
    {   // bf16 parts: q_rope [Tq, Hq, 64], v [Tk, Hk, 128], k_rope [Tk, 64]
        const uint64_t rd[3] = {64, (uint64_t)Hq, tq}, rs[2] = {128, (uint64_t)Hq * 128};
        const uint64_t vd[3] = {128, (uint64_t)Hk, tk}, vs[2] = {256, (uint64_t)Hk * 256};
        const uint32_t box[3] = {64, 1, 128};
        const uint64_t krd[2] = {64, tk}, krs[1] = {128};
        const uint32_t krb[2] = {64, 128};
        pa_status st = make_map_bf16(&mqr, q_rope, 3, rd, rs, box);
        if (st == PA_OK) st = make_map_bf16(&mv, v, 3, vd, vs, box);
        if (st == PA_OK) st = make_map_bf16(&mr, k_rope, 2, krd, krs, krb);
        if (st != PA_OK) return st;
    }
    pa::PrefillArgs a;
    pa_status st = fill_prefill_args(sh, cu_seqlens_q, cu_seqlens_k, nullptr, qo_offset, causal, scale, out, lse,
                                     workspace, workspace_bytes, false, &a);
    if (st != PA_OK) return st;
    a.f8 = 1;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    cudaError_t e = pa::launch_prefill(a, 192, &mq, &mk, &mv, &mr, &mqr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PA_OK;
}

pa_status pa_page_table_from_flat(const int32_t* kv_indices, int64_t num_indices, const int32_t* kv_lens,
                                  int32_t batch, int32_t max_pages_per_seq, int32_t* block_table, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_page_table_from_flat");
    if (batch <= 0 || batch > pa::kMaxBatch)
        return fail(PA_ERR_UNSUPPORTED, "batch must be in [1, %d] (got %d)", pa::kMaxBatch, batch);
    if (max_pages_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_pages_per_seq must be positive");
    if ((int64_t)batch * max_pages_per_seq >= ((int64_t)1 << 40))
        return fail(PA_ERR_UNSUPPORTED, "batch * max_pages_per_seq is too large");
    if (num_indices < 0) return fail(PA_ERR_INVALID_ARG, "num_indices must be >= 0");
    if ((num_indices > 0 && !kv_indices) || !kv_lens || !block_table || !workspace)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (workspace_bytes < PA_STATUS_BYTES)
        return fail(PA_ERR_WORKSPACE, "workspace needs %d bytes, got %zu", PA_STATUS_BYTES, workspace_bytes);
    cudaError_t e = pa::launch_page_table(kv_indices, num_indices, kv_lens, batch, max_pages_per_seq, block_table,
                                          static_cast<int*>(workspace), stream);
    if (e != cudaSuccess) return cuda_fail(e, "page table launch");
    return PA_OK;
}

size_t pa_prefill_workspace_size(const pa_prefill_shapes* sh) {
    if (!sh || sh->batch <= 0 || sh->max_seqlen_q <= 0) return PA_STATUS_BYTES;
    return PA_STATUS_BYTES + (size_t)sh->batch * (size_t)cdiv(sh->max_seqlen_q, 256) * 4;
}

namespace {
// pa_prefill_mla_rope_fp8's workspace: pa_prefill's, then the rope key's two
// bf16 levels [total_k, 64] each, every region 256-byte aligned
size_t rope_levels_offset(const pa_prefill_shapes* sh) { return (pa_prefill_workspace_size(sh) + 255) / 256 * 256; }
size_t rope_level_bytes(const pa_prefill_shapes* sh) {
    return ((size_t)(sh->total_k > 0 ? sh->total_k : 0) * 128 + 255) / 256 * 256;
}
}  // namespace

size_t pa_prefill_mla_rope_fp8_workspace_size(const pa_prefill_shapes* sh) {
    if (!sh) return PA_STATUS_BYTES;
    return rope_levels_offset(sh) + 2 * rope_level_bytes(sh);
}

pa_status pa_prefill_mla_rope_fp8(const pa_prefill_shapes* sh, const void* q, const void* k_nope, const void* v,
                                  const void* k_rope, const float* k_rope_scales, const int32_t* cu_seqlens_q,
                                  const int32_t* cu_seqlens_k, const int32_t* qo_offset, int causal, float scale,
                                  void* out, float* lse, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_prefill_mla_rope_fp8");
    if (!sh) return fail(PA_ERR_INVALID_ARG, "shapes must not be NULL");
    const int B = sh->batch, Hq = sh->num_q_heads, Hk = sh->num_kv_heads;
    if (B < 0 || sh->total_q < 0 || sh->total_k < 0 || sh->max_seqlen_q < 0)
        return fail(PA_ERR_INVALID_ARG, "batch, total_q, total_k and max_seqlen_q must be >= 0");
    if (B == 0 || sh->total_q == 0 || sh->max_seqlen_q == 0) return PA_OK;
    if (Hq <= 0 || Hk <= 0 || Hq % Hk != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)", Hq, Hk);
    if (Hq > 65535) return fail(PA_ERR_UNSUPPORTED, "num_q_heads above 65535");
    if (sh->dtype != PA_KV_BF16)
        return fail(PA_ERR_UNSUPPORTED, "pa_prefill_mla_rope_fp8 needs dtype PA_KV_BF16 (got %d)", sh->dtype);
    if (sh->head_dim_qk != 192 || sh->rope_dim != 64 || sh->head_dim_v != 128)
        return fail(PA_ERR_UNSUPPORTED, "pa_prefill_mla_rope_fp8 needs head_dim_qk 192, rope_dim 64, head_dim_v 128");
    if (sh->total_k <= 0) return fail(PA_ERR_INVALID_ARG, "ragged keys need total_k > 0");
    if (!q || !k_nope || !v || !k_rope || !k_rope_scales || !cu_seqlens_q || !cu_seqlens_k || !out || !workspace)
        return fail(PA_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned16(q) || !aligned16(k_nope) || !aligned16(v) || !aligned16(k_rope) || !aligned16(out) ||
        !aligned16(workspace))
        return fail(PA_ERR_INVALID_ARG, "q, k_nope, v, k_rope, out and workspace must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(k_rope_scales) % 4 != 0)
        return fail(PA_ERR_INVALID_ARG, "k_rope_scales must be 4-byte aligned");
    if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale must be finite");
    const size_t need = pa_prefill_mla_rope_fp8_workspace_size(sh);
    if (workspace_bytes < need) return fail(PA_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* hi = reinterpret_cast<uint16_t*>(ws + rope_levels_offset(sh));
    uint16_t* lo = reinterpret_cast<uint16_t*>(ws + rope_levels_offset(sh) + rope_level_bytes(sh));
    CUtensorMap mq, mk, mv, mr, mrl;
    const uint64_t tq = (uint64_t)sh->total_q, tk = (uint64_t)sh->total_k;
    {
        const uint64_t qd[3] = {192, (uint64_t)Hq, tq}, qs[2] = {384, (uint64_t)Hq * 384};
        const uint64_t kd[3] = {128, (uint64_t)Hk, tk}, ks[2] = {256, (uint64_t)Hk * 256};
        const uint32_t box[3] = {64, 1, 128};
        const uint64_t rd[2] = {64, tk}, rs[1] = {128};
        const uint32_t rb[2] = {64, 128};
        pa_status st = make_map_bf16(&mq, q, 3, qd, qs, box);
        if (st == PA_OK) st = make_map_bf16(&mk, k_nope, 3, kd, ks, box);
        if (st == PA_OK) st = make_map_bf16(&mv, v, 3, kd, ks, box);
        if (st == PA_OK) st = make_map_bf16(&mr, hi, 2, rd, rs, rb);
        if (st == PA_OK) st = make_map_bf16(&mrl, lo, 2, rd, rs, rb);
        if (st != PA_OK) return st;
    }
    pa::PrefillArgs a;
    pa_status st = fill_prefill_args(sh, cu_seqlens_q, cu_seqlens_k, nullptr, qo_offset, causal, scale, out, lse,
                                     workspace, workspace_bytes, false, &a);
    if (st != PA_OK) return st;
    a.r8 = 1;
    cudaError_t e = pa::launch_rope_expand(static_cast<const uint8_t*>(k_rope), k_rope_scales, hi, lo, sh->total_k,
                                           stream);
    if (e != cudaSuccess) return cuda_fail(e, "rope key expansion launch");
    e = pa::launch_prefill(a, 192, &mq, &mk, &mv, &mr, &mrl, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return PA_OK;
}

pa_status pa_get_static_plan(const pa_decode_shapes* sh, pa_decode_plan* plan) {
    pa::NvtxRange nvtx_range("pa_get_static_plan");
    if (!sh || !plan) return fail(PA_ERR_INVALID_ARG, "shapes and plan must not be NULL");
    const int B = sh->batch, Hk = sh->num_kv_heads;
    if (B <= 0 || B > pa::kMaxBatch)
        return fail(PA_ERR_UNSUPPORTED, "device scheduling needs 1 <= batch <= %d (got %d)", pa::kMaxBatch, B);
    if (Hk <= 0 || Hk > 65535) return fail(PA_ERR_INVALID_ARG, "num_kv_heads must be in [1, 65535] (got %d)", Hk);
    if (sh->page_size != pa::kPage) return fail(PA_ERR_INVALID_ARG, "page_size must be 64 (got %d)", sh->page_size);
    if (sh->max_pages_per_seq <= 0) return fail(PA_ERR_INVALID_ARG, "max_pages_per_seq must be positive");
    if (sh->num_sms <= 0 || sh->ctas_per_sm < 0 || sh->forced_splits < 0)
        return fail(PA_ERR_INVALID_ARG, "num_sms must be positive, ctas_per_sm and forced_splits >= 0");
    const int cps = sh->ctas_per_sm == 0 ? 1 : sh->ctas_per_sm;
    const int64_t cap = (int64_t)sh->num_sms * cps;
    const int64_t splits = sh->forced_splits > 0 ? (int64_t)B * std::min(sh->forced_splits, PA_MAX_SPLITS)
                                                 : B + cdiv(2 * cap, Hk);
    const int64_t items = splits * Hk;
    if (items > 16384) return fail(PA_ERR_UNSUPPORTED, "device scheduling handles up to 16384 work items (%lld)",
                                   (long long)items);
    plan->total_splits = (int32_t)splits;
    plan->num_items = (int32_t)items;
    plan->grid = (int32_t)cap;
    plan->meta_ints = (int32_t)(pa::kMetaHeader + 2 * (int64_t)B + 1 + cap + 1 + 2 * items);
    plan->ctas_per_sm = cps;
    plan->reserved = 1;  // capacity plan
    const int64_t hq = std::max(sh->num_q_heads, 0), d = std::max(sh->head_dim, 0);
    plan->workspace_bytes = (size_t)PA_STATUS_BYTES + (size_t)(splits * hq * d * 4) +
                            (size_t)(((splits * hq * 4) + 255) / 256 * 256) +
                            (size_t)((((int64_t)B * Hk * 4) + 255) / 256 * 256);
    return PA_OK;
}

pa_status pa_get_metadata_device(const pa_decode_shapes* sh, const pa_decode_plan* plan, const int32_t* seq_lens_dev,
                                 int32_t* meta_dev, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_get_metadata_device");
    if (!sh || !plan) return fail(PA_ERR_INVALID_ARG, "shapes and plan must not be NULL");
    if (!seq_lens_dev || !meta_dev) return fail(PA_ERR_INVALID_ARG, "seq_lens_dev and meta_dev must not be NULL");
    pa_decode_plan check;
    pa_status st = pa_get_static_plan(sh, &check);
    if (st != PA_OK) return st;
    if (plan->reserved != 1 || plan->num_items != check.num_items || plan->grid != check.grid)
        return fail(PA_ERR_INVALID_ARG, "the plan must come from pa_get_static_plan for these shapes");
    int p2 = 1;  // sort keys: one per split
    while (p2 < plan->total_splits) p2 <<= 1;
    const size_t smem = pa::schedule_smem_bytes(sh->batch, p2);
    if (smem > 227 * 1024) return fail(PA_ERR_UNSUPPORTED, "schedule needs %zu bytes of shared memory", smem);
    cudaError_t e = pa::launch_schedule(seq_lens_dev, sh->batch, sh->num_kv_heads, sh->max_pages_per_seq,
                                        plan->ctas_per_sm, plan->grid, sh->forced_splits, p2, meta_dev, stream);
    if (e != cudaSuccess) return cuda_fail(e, "schedule launch");
    return PA_OK;
}

pa_status pa_check_status(void* workspace, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_check_status");
    if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace must not be NULL");
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    if (word == 0) return PA_OK;
    e = cudaMemsetAsync(workspace, 0, sizeof word, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    switch (word) {
        case PA_ERR_TIMEOUT:
            return fail(PA_ERR_TIMEOUT, "a device-side wait ran past its time limit");
        case PA_ERR_DEVICE_BOUNDS:
            return fail(PA_ERR_DEVICE_BOUNDS, "a kernel met a page id or length out of range");
        default:
            return fail((pa_status)word, "device status %d", word);
    }
}

pa_status pa_debug_wait_timeout(void* workspace, uint64_t limit_ns, cudaStream_t stream) {
    if (!workspace) return fail(PA_ERR_INVALID_ARG, "workspace must not be NULL");
    cudaError_t e = pa::launch_wait_timeout_probe(static_cast<int*>(workspace), limit_ns, stream);
    if (e != cudaSuccess) return cuda_fail(e, "wait-timeout probe launch");
    return PA_OK;
}

}  // extern "C"
