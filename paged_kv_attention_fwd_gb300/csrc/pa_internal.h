// pa_internal.h -- declarations shared by the host API and the kernel files.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pa.h"

// NVTX v3 is header-only: without a profiler attached each push/pop is a
// check of one function pointer.
#include <nvtx3/nvToolsExt.h>

namespace pa {

constexpr int kPage = 64;
constexpr int kMetaHeader = 8;
constexpr int32_t kMetaMagic = 0x50414D31;

// Arguments of the persistent decode kernel (passed by value as a grid constant).
struct DecodeArgs {
    const uint16_t* q;         // bf16 [B, Hq, D]
    const uint8_t* k_pool;     // raw pool bytes (used by the e4m3 kernel's bulk copies)
    const uint8_t* v_pool;
    const float* k_scale;      // [Hk] (e4m3) or nullptr
    const float* v_scale;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const int32_t* meta;
    uint16_t* out;             // bf16 [B, Hq, D]
    float* lse;                // [B, Hq] or nullptr
    float* o_part;             // fp32 [total_splits, Hq, D]
    float* lse_part;           // fp32 [total_splits, Hq]
    int* status;               // status word
    int* counters;             // [B * Hk] split arrivals (fused combine), or nullptr: leave partials
    int32_t batch, num_q_heads, num_kv_heads, group, max_pages, num_pool_pages;
    int32_t f16;               // 16-bit pages are fp16 (q and out fp16 too), else bf16
    float scale_log2;          // softmax scale * log2(e)
    uint64_t wait_ns;
};

struct CombineArgs {
    const int32_t* meta;
    const float* o_part;
    const float* lse_part;
    uint16_t* out;
    float* lse;
    int32_t batch, num_q_heads, head_dim;
    int32_t f16;  // out is fp16, else bf16
};

// Launchers (decode.cu).  Return the CUDA error of the launch.
cudaError_t launch_decode(int head_dim, bool fp8, const DecodeArgs& a, const CUtensorMap* map_k,
                          const CUtensorMap* map_v, const CUtensorMap* map_q, int grid, cudaStream_t stream);
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(int* status, uint64_t limit_ns, cudaStream_t stream);

// Prefill (prefill.cu)
struct PrefillArgs {
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* block_table;
    const int32_t* qo_offset;
    const int32_t* order;  // [batch * num_q_tiles] unit order in the workspace, or nullptr
    uint16_t* out;   // bf16 [total_q, Hq, Dv]
    float* lse;      // [total_q, Hq] or nullptr
    int* status;
    int32_t batch, num_q_heads, num_kv_heads, group, max_pages, num_pool_pages, total_q;
    int32_t num_q_tiles;  // query blocks per segment: ceil(max_seqlen_q / q_block)
    int32_t q_block;      // query rows of one work item: 256 (one CTA) or 512 (a CTA pair)
    int32_t causal, paged, rope;
    int32_t f16;  // q, k, v, k_rope and out are fp16, else bf16
    int32_t f8;   // MLA with e4m3 q_nope / k_nope and per-head scales
    int32_t r8;   // MLA whose rope key arrives as bf16 hi + lo levels (from e4m3 codes and scales)
    const float* q_scale;  // f8: fp32 [Hq]
    const float* k_scale;  // f8: fp32 [Hk]
    float scale_log2;
    uint64_t wait_ns;
};

// e4m3 rope key codes [tokens, 64] times one fp32 scale per token -> two bf16
// levels hi = bf16(x), lo = bf16(x - hi), each [tokens, 64]
cudaError_t launch_rope_expand(const uint8_t* codes, const float* scales, uint16_t* hi, uint16_t* lo,
                               int64_t tokens, cudaStream_t stream);

// The longest-first order of the work units, into a.order (nothing when it is null).
cudaError_t launch_prefill_order(const PrefillArgs& a, cudaStream_t stream);

// The bf16 / fp16 prefill on CTA pairs (prefill_pair.cu): a.q_block must be
// 512; map_k and map_r have 64-row boxes (each CTA loads 64 keys of a tile).
// Returns cudaErrorNotSupported when no 2-CTA cluster fits on the device.
cudaError_t launch_prefill_pair(const PrefillArgs& a, int head_dim_qk, const CUtensorMap* map_q,
                                const CUtensorMap* map_k, const CUtensorMap* map_v, const CUtensorMap* map_r,
                                cudaStream_t stream);

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim_qk, const CUtensorMap* map_q,
                           const CUtensorMap* map_k, const CUtensorMap* map_v, const CUtensorMap* map_r,
                           const CUtensorMap* map_qr, cudaStream_t stream);

struct AppendArgs {
    const uint16_t* k_new;  // bf16 [total_new, Hk, D]
    const uint16_t* v_new;
    const int32_t* cu_new;
    const int32_t* start_pos;
    const int32_t* block_table;
    void* k_pool;
    void* v_pool;
    const float* k_scale;
    const float* v_scale;
    int* status;
    int32_t batch, num_kv_heads, head_dim, max_pages, num_pool_pages, total_new, fp8;
};

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);

// Device-side scheduler (schedule.cu)
constexpr int kMaxBatch = 8192;  // sequences the device-side metadata handles
size_t schedule_smem_bytes(int B, int p2cap);
// block table rows from a flat list of page ids (pa_page_table_from_flat)
cudaError_t launch_page_table(const int32_t* kv_indices, int64_t num_indices, const int32_t* kv_lens, int B,
                              int max_pages, int32_t* block_table, int* status, cudaStream_t stream);
cudaError_t launch_schedule(const int32_t* seq_lens, int B, int Hk, int max_pages, int cps, int cap, int forced,
                            int p2cap, int32_t* meta, cudaStream_t stream);

// Record a message for pa_last_error() on this host thread (pa_api.cu).
void set_last_error(const char* msg);

// The host-side checks of a decode call, launching nothing (pa_api.cu).
pa_status check_decode_call(const pa_decode_shapes* sh, const pa_decode_plan* plan, const void* q,
                            const void* k_pool, const void* v_pool, const float* k_scale, const float* v_scale,
                            const int32_t* block_table, const int32_t* seq_lens, const int32_t* meta_dev,
                            float scale, const void* out, const void* workspace, size_t workspace_bytes);

// A named NVTX range over one library call (from construction to the end of
// the scope), so a timeline shows which pa_* call enqueued which kernels.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Allow `kernel` `bytes` of dynamic shared memory on the current device.  A
// function attribute belongs to one device's context, so it is set once per
// (kernel, device): `done` holds one bit per device id (ids >= 64 set it on
// every launch).  Concurrent first calls may both set it; that is harmless.
template <typename K>
cudaError_t ensure_dynamic_smem(K* kernel, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace pa
