// decode.cu -- single-token attention over a paged KV cache on sm_103a.
//
// One persistent CTA per SM walks the work list the host scheduler dealt it:
// items (sequence b, split s, KV head g), each a contiguous range of 64-row
// pages (FlashMLA "Tensor Shapes Reference": paged K/V blocks of section 1,
// logical token -> block_table column as in "Prefill to Cache Mapping").
// Within a CTA the pages stream through a multi-stage shared-memory ring:
//
//   warp 0      producer: block_table lookup, TMA (bf16, 128-byte swizzle) or
//               plain bulk copies (e4m3) of whole 64 x D page slabs; with
//               16-bit pages also each item's query rows (one TMA box of the
//               group's heads), so that no thread waits on a global load
//               between items
//   warp 1      MMA issuer: tcgen05.mma, f32 accumulators in TMEM
//                 S^T[128 keys, 16 heads] = K_tile[128, D] . Q_group[16, D]^T
//                 O^T[D, 16 heads]        = V_tile^T[D, 128] . P^T[128, 16]
//               (the query heads of one KV group -- contiguous groups, as in
//               the "Grouped-Query Attention" diagram -- padded to 16 form N)
//   warps 2-5   softmax: one TMEM lane (= key of the tile, = d of the output)
//               per thread; per-head running max by warp transpose-reduce,
//               exp2, partial sums, P written back to shared memory; the
//               output accumulates in registers with the usual rescale
//   warps 6-9   (e4m3 only) convert e4m3 pages to f16 operand tiles (exact)
//
// (e4m3 pages at D = 128 take decode_f8_kernel below: no conversion pass, QK
// and PV issued from two warps, separate K and V rings.)
//
// Items whose sequence has more than one split write fp32 partials (output
// normalised by its own sum, plus its log-sum-exp); the last warp merges a
// sequence's splits as soon as they are all written (pa_decode), or
// combine_kernel does afterwards.  Every wait is bounded; a timeout raises the CTA's abort flag,
// records PA_ERR_TIMEOUT, drains in-flight copies and MMAs, frees TMEM and
// returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdio>
#include <mutex>

#include "pa_internal.h"
#include "pa_launch.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kNPad = 16;  // MMA N: query heads of one KV group, padded
constexpr float kLn2 = 0.69314718055994531f;

// barrier slots
enum : int {
    B_FULL = 0,    // [4] stage filled (TMA bytes landed)
    B_EMPTY = 4,   // [4] stage free again
    B_QF = 8,      // [2] query tile written
    B_SF = 10,     // [2] S tile in TMEM
    B_PF = 12,     // [2] P written (and dead V rows zeroed)
    B_OF = 14,     // [2] O tile in TMEM
    B_DONE = 16,   // all MMAs retired (teardown)
    B_KHF = 17,    // e4m3: converted K tile ready
    B_KHE = 18,    // e4m3: converted K tile consumed
    B_VHF = 19,    // [2] e4m3: converted V tile ready
    B_VHE = 21,    // [2] e4m3: converted V tile consumed
    B_PW = 23,     // [2] an item's partials written (merge warp)
    B_HD = 25,     // [2] merge warp done with an item
    B_QE = 27,     // [2] query tile free again (16-bit pages: its last QK retired)
    B_COUNT = 29
};

constexpr uint32_t kTmemCols = 64;
__host__ __device__ constexpr uint32_t s_col(uint32_t b) { return b * 16u; }
__host__ __device__ constexpr uint32_t o_col(uint32_t b) { return 32u + b * 16u; }

template <int D, bool FP8>
struct DecodeLayout {
    static constexpr int kChunks = D / 64;             // 64-column (128-byte) chunks of a 16-bit row
    static constexpr int kTile16 = kChunks * 2 * 8192;  // 128-key tile of 16-bit K or V, swizzled
    static constexpr int kRawPage = 64 * D;             // one e4m3 page slab, row-major
    static constexpr int kRawTile = 2 * kRawPage;
    static constexpr int kStages = FP8 ? 3 : (D == 128 ? 3 : 4);
    static constexpr int kStageBytes = FP8 ? 2 * kRawTile : 2 * kTile16;
    static constexpr int kKhOff = kStages * kStageBytes;
    static constexpr int kVhOff = kKhOff + (FP8 ? kTile16 : 0);
    static constexpr int kQOff = kVhOff + (FP8 ? 2 * kTile16 : 0);
    static constexpr int kQBytes = kChunks * kNPad * 128;
    static constexpr int kPOff = kQOff + 2 * kQBytes;
    static constexpr int kPBytes = 2 * kNPad * 128;
    static constexpr int kRedOff = kPOff + 2 * kPBytes;
    static constexpr int kRedBytes = 4 * kNPad * 4 * 4;
    static constexpr int kEnd = kRedOff + kRedBytes;
    // With D = 64 the PV MMA (M = 128) also reads a second 64-row MN atom
    // 16 KB past each V tile; its rows are discarded, but the window must be
    // inside the allocation.
    static constexpr int kLastV = FP8 ? kVhOff + kTile16 : (kStages - 1) * kStageBytes + kTile16;
    static constexpr int kGuardEnd = D == 64 ? kLastV + 32768 : 0;
    static constexpr int kBytes = kEnd > kGuardEnd ? kEnd : kGuardEnd;
    static constexpr int kSmem = kBytes + 1024;
    static constexpr int kMergeWarp = FP8 ? 10 : 6;  // last warp: split merge (pa_decode)
    static constexpr int kThreads = (kMergeWarp + 1) * 32;
    static_assert(kStages <= 4, "barrier slots");
};

struct Item {
    int b, s, kvh, nsplit, split_base, p0, p1, seq_len;
};

__device__ __forceinline__ void record(int* status, int code) { atomicCAS(status, 0, code); }

__device__ __forceinline__ void fail(const DecodeArgs& a, volatile int* abort_flag, int code) {
    *abort_flag = 1;
    record(a.status, code);
}

__device__ __forceinline__ int items_offset(const int32_t* meta, int B) {
    return kMetaHeader + 2 * B + 1 + meta[5] + 1;
}

__device__ __forceinline__ Item load_item(const DecodeArgs& a, int idx, int items_off) {
    const int32_t* meta = a.meta;
    Item it;
    int b = __ldg(&meta[items_off + 2 * idx]);
    const int w = __ldg(&meta[items_off + 2 * idx + 1]);
    int s = w >> 16, kvh = w & 0xFFFF;
    bool ok = (unsigned)b < (unsigned)a.batch && kvh < a.num_kv_heads;
    if (!ok) b = 0;
    int nsplit = __ldg(&meta[kMetaHeader + b]);
    if (nsplit < 1 || s >= nsplit) ok = false;
    int len = __ldg(&a.seq_lens[b]);
    len = len < 0 ? 0 : len;
    int pages = (len + kPage - 1) / kPage;
    if (pages > a.max_pages) {
        record(a.status, PA_ERR_DEVICE_BOUNDS);
        pages = a.max_pages;
        len = pages * kPage;
    }
    if (!ok) {
        record(a.status, PA_ERR_DEVICE_BOUNDS);
        nsplit = 1; s = 0; kvh = 0; pages = 0; len = 0;
    }
    it.b = b; it.s = s; it.kvh = kvh; it.nsplit = nsplit;
    it.split_base = __ldg(&meta[kMetaHeader + a.batch + b]);
    it.p0 = (int)(((long long)s * pages) / nsplit);
    it.p1 = (int)(((long long)(s + 1) * pages) / nsplit);
    it.seq_len = len;
    return it;
}

__device__ __forceinline__ int item_tiles(const Item& it) { return (it.p1 - it.p0 + 1) >> 1; }

// The first kItemCache items of a CTA are decoded once, in the prologue, into
// shared memory: every role reads its next item there instead of repeating
// the chain of dependent global loads at each item boundary.
constexpr int kItemCache = 64;

__device__ __forceinline__ void fill_item_cache(Item* cache, const DecodeArgs& a, int it_lo, int it_hi,
                                                int items_off, int lane) {
    const int n = min(it_hi - it_lo, kItemCache);
    for (int i = lane; i < n; i += 32) cache[i] = load_item(a, it_lo + i, items_off);
}

__device__ __forceinline__ Item get_item(const Item* cache, const DecodeArgs& a, int j, int it_lo, int items_off) {
    const int i = j - it_lo;
    return i < kItemCache ? cache[i] : load_item(a, j, items_off);
}

// All-reduce NP per-thread values over a warp by transposition: each
// shuffle level exchanges half of the remaining values, so NP = 16 costs 16
// shuffles instead of 80.  Returns the reduction of value head_of_lane<NP>(lane).
template <int NP, bool kMax>
__device__ __forceinline__ float warp_xreduce(const float (&x)[NP], int lane) {
    float v[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) v[i] = x[i];
#pragma unroll
    for (int cnt = NP, off = 16; cnt > 1; cnt >>= 1, off >>= 1) {
        const bool up = lane & off;
#pragma unroll
        for (int i = 0; i < cnt / 2; ++i) {
            const float send = up ? v[i] : v[i + cnt / 2];
            const float keep = up ? v[i + cnt / 2] : v[i];
            const float got = __shfl_xor_sync(0xffffffffu, send, off);
            v[i] = kMax ? fmaxf(keep, got) : keep + got;
        }
    }
#pragma unroll
    for (int off = 16 / NP; off >= 1; off >>= 1) {
        const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
        v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
    }
    return v[0];
}

// Which of the NP values lane `lane` holds after warp_xreduce<NP>.
template <int NP>
__device__ __forceinline__ int head_of_lane(int lane) {
    int h = 0;
#pragma unroll
    for (int cnt = NP, off = 16; cnt > 1; cnt >>= 1, off >>= 1)
        if (lane & off) h += cnt / 2;
    return h;
}

// One lane per value writes it out: the lanes whose bits below the last
// transposition offset are zero.
template <int NP>
__device__ __forceinline__ bool lane_writes(int lane) {
    return (lane & ((32 / NP) - 1)) == 0;
}

// Barrier over the 128 softmax threads that also ORs a flag across them, so
// that every thread takes the same abort decision.
__device__ __forceinline__ bool softmax_bar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}


// Barrier `id` over `nthreads` threads that also ORs a flag across them.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// the 16-bit output element: fp16 when the inputs are fp16, else bf16
__device__ __forceinline__ uint16_t out16(float x, bool f16) {
    return f16 ? __half_as_ushort(__float2half_rn(x)) : __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Split merge inside the decode kernel (pa_decode).  The softmax threads
// write an item's partials, then arrive on a barrier; one extra warp -- the
// merge warp -- takes it from there, off the softmax's critical path: it
// counts the split's arrival in the workspace (device-scope acquire-release)
// and, if that arrival completes the sequence's splits, merges them
//   L = m + ln sum_s exp(lse_s - m),  out = sum_s exp(lse_s - L) o_s
// and resets the counter for the next call.  Two barrier pairs (written /
// merged) let the softmax run up to two partial items ahead.

// Softmax side: all 128 threads, after writing partial item number k.
__device__ __forceinline__ bool partials_written(uint64_t* pw, uint64_t* hd, uint32_t k, volatile int* abort_sh,
                                                 uint64_t wait_ns) {
    if (k >= 2 && !mbar_wait(&hd[k & 1], ((k - 2) >> 1) & 1, abort_sh, wait_ns)) return false;
    mbar_arrive(&pw[k & 1]);
    return true;
}

template <int D>
__device__ void merge_warp(const DecodeArgs& a, const Item* items, int it_lo, int it_hi, int items_off,
                           uint64_t* pw, uint64_t* hd,
                           volatile int* abort_sh, int lane) {
    uint32_t k = 0;
    const int G = a.group;
    for (int j = it_lo; j < it_hi; ++j) {
        const Item it = get_item(items, a, j, it_lo, items_off);
        if (it.nsplit <= 1) continue;
        bool ok = mbar_wait(&pw[k & 1], (k >> 1) & 1, abort_sh, a.wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
            if (lane == 0) fail(a, abort_sh, PA_ERR_TIMEOUT);
            return;
        }
        int last = 0;
        int* ctr = a.counters + (long long)it.b * a.num_kv_heads + it.kvh;
        if (lane == 0) {
            int prev;
            asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
            last = prev == it.nsplit - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last) {
            const long long base = (long long)it.split_base * a.num_q_heads + (long long)it.kvh * G;
            const long long orow = (long long)it.b * a.num_q_heads + (long long)it.kvh * G;
            for (int h = 0; h < G; ++h) {
                float mx = -INFINITY;
                for (int s = 0; s < it.nsplit; ++s)
                    mx = fmaxf(mx, __ldcg(&a.lse_part[base + (long long)s * a.num_q_heads + h]));
                float acc[D / 32];
#pragma unroll
                for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
                float wsum = 0.f;
                if (mx != -INFINITY) {
                    for (int s = 0; s < it.nsplit; ++s) {
                        const long long prow = base + (long long)s * a.num_q_heads + h;
                        const float w = __expf(__ldcg(&a.lse_part[prow]) - mx);
                        wsum += w;
#pragma unroll
                        for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, __ldcg(&a.o_part[prow * D + lane + 32 * i]), acc[i]);
                    }
                }
                const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
                for (int i = 0; i < D / 32; ++i)
                    a.out[(orow + h) * D + lane + 32 * i] = out16(acc[i] * inv, a.f16);
                if (lane == 0 && a.lse) a.lse[orow + h] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
            }
            if (lane == 0) *ctr = 0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd[k & 1]);
        ++k;
    }
}

__device__ __forceinline__ uint16_t f32_to_16(float x, bool f16) {
    if (f16) return __half_as_ushort(__float2half_rn(x));
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

template <int D, bool FP8, int NP>
__global__ void __launch_bounds__(DecodeLayout<D, FP8>::kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_q) {
    using L = DecodeLayout<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[B_COUNT];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_store;
    __shared__ __align__(16) Item items_sh[kItemCache];
    volatile int* abort_sh = &abort_store;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&bars[B_FULL + s], 1);
            mbar_init(&bars[B_EMPTY + s], FP8 ? 128 : 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_QF + i], FP8 ? 128 : 1);
            mbar_init(&bars[B_QE + i], 1);
            mbar_init(&bars[B_SF + i], 1);
            mbar_init(&bars[B_PF + i], 128);
            mbar_init(&bars[B_OF + i], 1);
            mbar_init(&bars[B_VHF + i], 128);
            mbar_init(&bars[B_VHE + i], 1);
        }
        mbar_init(&bars[B_DONE], 1);
        mbar_init(&bars[B_KHF], 128);
        mbar_init(&bars[B_KHE], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_PW + i], 128);
            mbar_init(&bars[B_HD + i], 1);
        }
        *abort_sh = 0;
        fence_barrier_init();
    }
    if (warp >= 2 && warp < 6) {
        // P rows of padding heads must read as zero in every PV product, and
        // so must the query rows past the group (the query TMA writes only
        // the group's rows)
        uint4* p = reinterpret_cast<uint4*>(sm + L::kPOff);
        for (int i = threadIdx.x - 64; i < 2 * L::kPBytes / 16; i += 128) p[i] = make_uint4(0, 0, 0, 0);
        if constexpr (!FP8) {
            uint4* qz = reinterpret_cast<uint4*>(sm + L::kQOff);
            for (int i = threadIdx.x - 64; i < 2 * L::kQBytes / 16; i += 128) qz[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    // shared memory only up to here: this part overlaps the previous kernel
    grid_dependency_wait();
    const int32_t* meta = a.meta;
    const int B = a.batch;
    const int items_off = items_offset(meta, B);
    int it_lo = 0, it_hi = 0;
    if ((int)blockIdx.x < __ldg(&meta[5])) {
        it_lo = __ldg(&meta[kMetaHeader + 2 * B + 1 + blockIdx.x]);
        it_hi = __ldg(&meta[kMetaHeader + 2 * B + 1 + blockIdx.x + 1]);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    if (warp == L::kMergeWarp) fill_item_cache(items_sh, a, it_lo, it_hi, items_off, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t g = 0, qn = 0;
            uint32_t last_par[4] = {0, 0, 0, 0}, q_par[2] = {0, 0};
            bool issued[4] = {false, false, false, false}, q_issued[2] = {false, false};
            bool ok = true;
            constexpr uint32_t page_bytes = FP8 ? 64u * D : 64u * D * 2u;
            for (int j = it_lo; j < it_hi && ok; ++j) {
                const Item it = get_item(items_sh, a, j, it_lo, items_off);
                const int ntiles = item_tiles(it);
                const long long bt_row = (long long)it.b * a.max_pages;
                if (!FP8 && ntiles > 0) {
                    // the group's query rows -> rows 0..G-1 of query buffer qn & 1
                    const uint32_t qs = qn & 1;
                    if (!mbar_wait(&bars[B_QE + qs], ((qn >> 1) & 1) ^ 1, abort_sh, a.wait_ns)) {
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    uint64_t* qf = &bars[B_QF + qs];
                    mbar_arrive_expect_tx(qf, (uint32_t)a.group * D * 2u);
                    const int qrow = it.b * a.num_q_heads + it.kvh * a.group;
#pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
                        tma_load_2d(sm + L::kQOff + qs * L::kQBytes + c * (kNPad * 128), &map_q, qf, c * 64, qrow);
                    q_par[qs] = (qn >> 1) & 1;
                    q_issued[qs] = true;
                    ++qn;
                }
                for (int t = 0; t < ntiles; ++t, ++g) {
                    const int stage = g % L::kStages;
                    const int pa0 = it.p0 + 2 * t;
                    const int npg = min(2, it.p1 - pa0);
                    int pid[2];
                    pid[0] = __ldg(&a.block_table[bt_row + pa0]);
                    pid[1] = npg > 1 ? __ldg(&a.block_table[bt_row + pa0 + 1]) : 0;
                    if (!mbar_wait(&bars[B_EMPTY + stage], ((g / L::kStages) & 1) ^ 1, abort_sh, a.wait_ns)) {
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    bool valid[2];
                    uint32_t nvalid = 0;
                    for (int i = 0; i < 2; ++i) {
                        valid[i] = i < npg && (unsigned)pid[i] < (unsigned)a.num_pool_pages;
                        if (i < npg && !valid[i]) record(a.status, PA_ERR_DEVICE_BOUNDS);
                        nvalid += valid[i];
                    }
                    uint64_t* full = &bars[B_FULL + stage];
                    mbar_arrive_expect_tx(full, nvalid * 2u * page_bytes);
                    uint8_t* st = sm + stage * L::kStageBytes;
                    for (int i = 0; i < 2; ++i) {
                        if (!valid[i]) continue;
                        const long long slab = (long long)pid[i] * a.num_kv_heads + it.kvh;
                        if constexpr (FP8) {
                            bulk_load(st + i * L::kRawPage, a.k_pool + slab * L::kRawPage, L::kRawPage, full);
                            bulk_load(st + L::kRawTile + i * L::kRawPage, a.v_pool + slab * L::kRawPage, L::kRawPage,
                                      full);
                        } else {
#pragma unroll
                            for (int c = 0; c < L::kChunks; ++c) {
                                tma_load_2d(st + c * 16384 + i * 8192, &map_k, full, c * 64, (int)(slab * 64));
                                tma_load_2d(st + L::kTile16 + c * 16384 + i * 8192, &map_v, full, c * 64,
                                            (int)(slab * 64));
                            }
                        }
                    }
                    last_par[stage] = (g / L::kStages) & 1;
                    issued[stage] = true;
                }
            }
            // every issued copy must land before the CTA may exit
            for (int s = 0; s < L::kStages; ++s)
                if (issued[s]) mbar_wait(&bars[B_FULL + s], last_par[s], nullptr, a.wait_ns);
            for (int s = 0; s < 2; ++s)
                if (q_issued[s]) mbar_wait(&bars[B_QF + s], q_par[s], nullptr, a.wait_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const bool as_f16 = FP8 || a.f16;  // operand format: fp16, else bf16
            const uint32_t idesc_qk = idesc_f16(128, kNPad, !as_f16, false, false);
            const uint32_t idesc_pv = idesc_f16(128, kNPad, !as_f16, true, false);
            uint32_t g = 0, qi = 0;
            bool pending = false, ok = true;
            auto issue_pv = [&](uint32_t k) -> bool {
                if (!mbar_wait(&bars[B_PF + (k & 1)], (k >> 1) & 1, abort_sh, a.wait_ns)) return false;
                if (FP8 && !mbar_wait(&bars[B_VHF + (k & 1)], (k >> 1) & 1, abort_sh, a.wait_ns)) return false;
                tc_fence_after();
                const uint32_t vbase = FP8 ? smem_u32(sm + L::kVhOff + (k & 1) * L::kTile16)
                                           : smem_u32(sm + (k % L::kStages) * L::kStageBytes + L::kTile16);
                const uint32_t pbase = smem_u32(sm + L::kPOff + (k & 1) * L::kPBytes);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int page = kk >> 2, grp = kk & 3;
                    const uint64_t adesc = sdesc_sw128(vbase + page * 8192 + grp * 2048, 16384, 1024);
                    const uint64_t bdesc = sdesc_sw128(pbase + page * 2048 + grp * 32, 16, 1024);
                    mma_ss(tbase + o_col(k & 1), adesc, bdesc, idesc_pv, kk > 0);
                }
                mma_commit(&bars[B_OF + (k & 1)]);
                if (FP8) mma_commit(&bars[B_VHE + (k & 1)]);
                else mma_commit(&bars[B_EMPTY + (k % L::kStages)]);
                return true;
            };
            for (int j = it_lo; j < it_hi && ok; ++j) {
                const Item it = get_item(items_sh, a, j, it_lo, items_off);
                const int ntiles = item_tiles(it);
                if (ntiles == 0) continue;
                if (!mbar_wait(&bars[B_QF + (qi & 1)], (qi >> 1) & 1, abort_sh, a.wait_ns)) {
                    fail(a, abort_sh, PA_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                const uint32_t qslot = qi & 1;
                const uint32_t qbase = smem_u32(sm + L::kQOff + qslot * L::kQBytes);
                ++qi;
                for (int t = 0; t < ntiles; ++t, ++g) {
                    const int stage = g % L::kStages;
                    const bool got = FP8 ? mbar_wait(&bars[B_KHF], g & 1, abort_sh, a.wait_ns)
                                         : mbar_wait(&bars[B_FULL + stage], (g / L::kStages) & 1, abort_sh, a.wait_ns);
                    if (!got) {
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kbase = FP8 ? smem_u32(sm + L::kKhOff) : smem_u32(sm + stage * L::kStageBytes);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int c = kk >> 2, off = (kk & 3) * 32;
                        const uint64_t adesc = sdesc_sw128(kbase + c * 16384 + off, 16, 1024);
                        const uint64_t bdesc = sdesc_sw128(qbase + c * 2048 + off, 16, 1024);
                        mma_ss(tbase + s_col(g & 1), adesc, bdesc, idesc_qk, kk > 0);
                    }
                    mma_commit(&bars[B_SF + (g & 1)]);
                    if (FP8) mma_commit(&bars[B_KHE]);
                    if (pending && !issue_pv(g - 1)) {
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    pending = true;
                }
                if (!FP8) mma_commit(&bars[B_QE + qslot]);  // the item's QKs are all issued
            }
            if (ok && pending && !issue_pv(g - 1)) fail(a, abort_sh, PA_ERR_TIMEOUT);
            // all MMAs must retire before TMEM is freed and shared memory released
            mma_commit(&bars[B_DONE]);
            mbar_wait(&bars[B_DONE], 0, nullptr, a.wait_ns);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax
        const int q4 = warp & 3;          // TMEM lane quarter this warp may access
        const int row = q4 * 32 + lane;   // key of the tile (S) / output column d (O)
        const int hl = head_of_lane<NP>(lane);
        const bool writer = lane_writes<NP>(lane);
        const int G = a.group;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        float* red = reinterpret_cast<float*>(sm + L::kRedOff);

        auto next_nonempty = [&](int j) {
            while (j < it_hi && item_tiles(get_item(items_sh, a, j, it_lo, items_off)) == 0) ++j;
            return j;
        };
        // query rows of the item's KV group -> swizzled K-major tile of 16 rows
        auto load_q = [&](int j, uint32_t qidx) {
            const Item it = get_item(items_sh, a, j, it_lo, items_off);
            uint8_t* qb = sm + L::kQOff + (qidx & 1) * L::kQBytes;
            constexpr int kRowChunks = D / 8;  // 16-byte chunks per row
            for (int c = row; c < kNPad * kRowChunks; c += 128) {
                const int h = c / kRowChunks, dc = c % kRowChunks;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (h < G) {
                    const long long qrow = (long long)it.b * a.num_q_heads + (long long)it.kvh * G + h;
                    v = __ldg(reinterpret_cast<const uint4*>(a.q + qrow * D) + dc);
                    if constexpr (FP8) {
                        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
                            w[i] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
                                   ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
                        }
                        v = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                *reinterpret_cast<uint4*>(qb + (dc >> 3) * (kNPad * 128) + h * 128 + (((dc & 7) ^ (h & 7)) << 4)) = v;
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars[B_QF + (qidx & 1)]);
        };

        int qload = next_nonempty(it_lo);
        uint32_t qload_idx = 0;
        if constexpr (FP8) {
            for (int k = 0; k < 2 && qload < it_hi; ++k) {
                load_q(qload, qload_idx++);
                qload = next_nonempty(qload + 1);
            }
        }

        uint32_t g = 0, qi = 0, npartial = 0;
        bool aborted = false;
        for (int j = it_lo; j < it_hi && !aborted; ++j) {
            const Item it = get_item(items_sh, a, j, it_lo, items_off);
            const int ntiles = item_tiles(it);
            const bool partial = it.nsplit > 1;
            const long long head0 = (long long)it.kvh * G;
            const long long orow = partial ? (long long)(it.split_base + it.s) * a.num_q_heads + head0
                                           : (long long)it.b * a.num_q_heads + head0;
            if (ntiles == 0) {
                // empty key range: out = 0, lse = -inf
                for (int h = 0; h < G; ++h) {
                    if (row < D) {
                        if (partial) a.o_part[(orow + h) * D + row] = 0.f;
                        else a.out[(orow + h) * D + row] = 0;
                    }
                }
                if (row < G) {
                    if (partial) a.lse_part[orow + row] = -INFINITY;
                    else if (a.lse) a.lse[orow + row] = -INFINITY;
                }
                if (partial && a.counters &&
                    !partials_written(&bars[B_PW], &bars[B_HD], npartial++, abort_sh, a.wait_ns))
                    fail(a, abort_sh, PA_ERR_TIMEOUT);  // the next barrier takes every thread out
                continue;
            }
            if (FP8 && qi >= 1 && qload < it_hi) {
                load_q(qload, qload_idx++);
                qload = next_nonempty(qload + 1);
            }
            ++qi;
            const float sl2 = a.scale_log2 * (FP8 ? __ldg(&a.k_scale[it.kvh]) : 1.f);
            const int key_end = min(it.seq_len, it.p1 * kPage);
            float m[NP], lp[NP], o[NP], alpha_prev[NP];
#pragma unroll
            for (int h = 0; h < NP; ++h) { m[h] = -INFINITY; lp[h] = 0.f; o[h] = 0.f; alpha_prev[h] = 1.f; }

            auto fold = [&](uint32_t k) {
                if (!mbar_wait(&bars[B_OF + (k & 1)], (k >> 1) & 1, abort_sh, a.wait_ns)) fail(a, abort_sh, PA_ERR_TIMEOUT);
                tc_fence_after();
                uint32_t r[NP];
                tmem_ld_cols<NP>(tbase + lane_addr + o_col(k & 1), r);
                tmem_ld_wait();
                reg_fence(r);
#pragma unroll
                for (int h = 0; h < NP; ++h) o[h] = fmaf(o[h], alpha_prev[h], __uint_as_float(r[h]));
            };

            for (int t = 0; t < ntiles; ++t, ++g) {
                const int pa0 = it.p0 + 2 * t;
                const int npg = min(2, it.p1 - pa0);
                const int key = pa0 * kPage + row;
                const bool valid = row < npg * kPage && key < key_end;
                if (!mbar_wait(&bars[B_SF + (g & 1)], (g >> 1) & 1, abort_sh, a.wait_ns))
                    fail(a, abort_sh, PA_ERR_TIMEOUT);
                tc_fence_after();
                uint32_t sr[NP];
                tmem_ld_cols<NP>(tbase + lane_addr + s_col(g & 1), sr);
                tmem_ld_wait();
                reg_fence(sr);
                float x[NP];
#pragma unroll
                for (int h = 0; h < NP; ++h) x[h] = valid ? __uint_as_float(sr[h]) * sl2 : -INFINITY;
                const float wmax = warp_xreduce<NP, true>(x, lane);
                float* rb = red + (g & 1) * 64;
                if (writer) rb[hl * 4 + q4] = wmax;
                if (softmax_bar_or(*abort_sh != 0)) { aborted = true; break; }
                float alpha[NP];
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    const float4 r4 = reinterpret_cast<const float4*>(rb)[h];
                    const float mt = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
                    const float mn = fmaxf(m[h], mt);
                    const bool none = mn == -INFINITY;
                    alpha[h] = none ? 1.f : exp2f(m[h] - mn);
                    x[h] = none ? 0.f : exp2f(x[h] - mn);  // x[h] = -inf -> 0
                    lp[h] = fmaf(lp[h], alpha[h], x[h]);
                    m[h] = mn;
                }
                // P^T tile (K-major: rows = heads, 128 keys in two 64-key chunks)
                uint8_t* pb = sm + L::kPOff + (g & 1) * L::kPBytes + (row >> 6) * (kNPad * 128);
#pragma unroll
                for (int h = 0; h < NP; ++h)
                    if (h < G)
                        *reinterpret_cast<uint16_t*>(pb + sw128_offset(h, row & 63)) = f32_to_16(x[h], FP8 || a.f16);
                if (!FP8 && !valid) {
                    // a dead key's V row may hold anything (NaN included); 0 * NaN
                    // would poison the PV product, so zero the row first
                    const int stage = g % L::kStages;
                    mbar_wait(&bars[B_FULL + stage], (g / L::kStages) & 1, abort_sh, a.wait_ns);
                    uint8_t* vr = sm + stage * L::kStageBytes + L::kTile16 + (row >> 6) * 8192 + (row & 63) * 128;
#pragma unroll
                    for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
                        for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(vr + c * 16384 + i * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars[B_PF + (g & 1)]);
                if (t > 0) fold(g - 1);
#pragma unroll
                for (int h = 0; h < NP; ++h) alpha_prev[h] = alpha[h];
            }
            if (aborted) break;
            fold(g - 1);
            tc_fence_before();

            // ---- epilogue: total sums, normalise, write
            const float wsum = warp_xreduce<NP, false>(lp, lane);
            float* rl = red + 128 + (qi & 1) * 64;
            if (writer) rl[hl * 4 + q4] = wsum;
            if (softmax_bar_or(*abort_sh != 0)) { aborted = true; break; }
            const float vs = FP8 ? __ldg(&a.v_scale[it.kvh]) : 1.f;
            float mine_m = 0.f, mine_l = 0.f;
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                const float4 r4 = reinterpret_cast<const float4*>(rl)[h];
                const float l = (r4.x + r4.y) + (r4.z + r4.w);
                if (h == row) { mine_m = m[h]; mine_l = l; }
                if (h < G && row < D) {
                    const float val = l > 0.f ? o[h] * (vs / l) : 0.f;
                    if (partial) a.o_part[(orow + h) * D + row] = val;
                    else a.out[(orow + h) * D + row] = out16(val, a.f16);
                }
            }
            if (row < G) {
                const float lse = mine_l > 0.f ? (mine_m + log2f(mine_l)) * kLn2 : -INFINITY;
                if (partial) a.lse_part[orow + row] = lse;
                else if (a.lse) a.lse[orow + row] = lse;
            }
            if (partial && a.counters &&
                !partials_written(&bars[B_PW], &bars[B_HD], npartial++, abort_sh, a.wait_ns))
                fail(a, abort_sh, PA_ERR_TIMEOUT);  // the next barrier takes every thread out
        }
        tc_fence_before();
    } else if (warp == L::kMergeWarp) {
        // ------------------------------------------------------------ split merge
        if (a.counters) merge_warp<D>(a, items_sh, it_lo, it_hi, items_off, &bars[B_PW], &bars[B_HD], abort_sh, lane);
    } else {
        // ------------------------------------------------------------ e4m3 -> f16 converters
        if constexpr (FP8) {
            const int ct = threadIdx.x - 192;  // tile row (key) this thread converts
            const int page = ct >> 6, r = ct & 63;
            uint32_t g = 0;
            bool ok = true;
            constexpr int kSrcChunks = D / 16;  // 16 e4m3 per 16-byte chunk
            auto convert_row = [&](const uint8_t* src, uint8_t* dst_tile, bool zero) {
#pragma unroll 4
                for (int i = 0; i < kSrcChunks; ++i) {
                    const int cc = (i + ct) % kSrcChunks;  // staggered: no bank conflicts
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
                    if (!zero) {
                        const uint4 raw = *reinterpret_cast<const uint4*>(src + cc * 16);
                        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                        uint32_t h2[8];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __half2_raw a0 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[k] & 0xFFFFu), __NV_E4M3);
                            const __half2_raw a1 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[k] >> 16), __NV_E4M3);
                            h2[2 * k] = (uint32_t)a0.x | ((uint32_t)a0.y << 16);
                            h2[2 * k + 1] = (uint32_t)a1.x | ((uint32_t)a1.y << 16);
                        }
                        lo = make_uint4(h2[0], h2[1], h2[2], h2[3]);
                        hi = make_uint4(h2[4], h2[5], h2[6], h2[7]);
                    }
                    const int d = cc * 16;  // first of the 16 elements
                    uint8_t* t = dst_tile + (d >> 6) * 16384 + page * 8192;
                    *reinterpret_cast<uint4*>(t + sw128_offset(r, d & 63)) = lo;
                    *reinterpret_cast<uint4*>(t + sw128_offset(r, (d & 63) + 8)) = hi;
                }
            };
            for (int j = it_lo; j < it_hi && ok; ++j) {
                const Item it = get_item(items_sh, a, j, it_lo, items_off);
                const int ntiles = item_tiles(it);
                const int key_end = min(it.seq_len, it.p1 * kPage);
                for (int t = 0; t < ntiles; ++t, ++g) {
                    const int stage = g % L::kStages;
                    const int pa0 = it.p0 + 2 * t;
                    const int npg = min(2, it.p1 - pa0);
                    const bool row_live = page < npg;
                    const bool key_live = row_live && pa0 * kPage + ct < key_end;
                    if (!mbar_wait(&bars[B_FULL + stage], (g / L::kStages) & 1, abort_sh, a.wait_ns) ||
                        (g > 0 && !mbar_wait(&bars[B_KHE], (g - 1) & 1, abort_sh, a.wait_ns))) {
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const uint8_t* raw = sm + stage * L::kStageBytes;
                    if (row_live) convert_row(raw + page * L::kRawPage + r * D, sm + L::kKhOff, false);
                    fence_proxy_async_smem();
                    mbar_arrive(&bars[B_KHF]);
                    if (g >= 2 && !mbar_wait(&bars[B_VHE + (g & 1)], ((g - 2) >> 1) & 1, abort_sh, a.wait_ns)) {
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    convert_row(raw + L::kRawTile + page * L::kRawPage + r * D, sm + L::kVhOff + (g & 1) * L::kTile16,
                                !key_live);
                    fence_proxy_async_smem();
                    mbar_arrive(&bars[B_VHF + (g & 1)]);
                    mbar_arrive(&bars[B_EMPTY + stage]);
                }
            }
        }
    }

    // the next programmatic launch may take this SM once every CTA is here
    // (issued after the prologue instead, its CTAs would wait on the SMs of
    // this launch's tail: 0.6% slower)
    allow_dependents_launch();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// e4m3 pages, D = 128: both products on the e4m3 tensor path (kind::f8f6f4),
// straight from the TMA-loaded pages -- no conversion pass, so shared memory
// holds only the page ring (5 stages of 2 pages of K and V).
//   S^T[128 keys, 48] = K_tile . Q3^T: the bf16 query of each head is scaled
//     by a power of two (max |q| -> [128, 256)) and split into three e4m3
//     levels hi + mid + lo (the split keeps 12 significant bits; bf16 has 8),
//     stacked as 48 rows of one MMA operand, so that one N = 48 product per
//     32 bytes of d gives the three level products side by side; the softmax
//     adds them.  Every tcgen05.mma costs the issuing thread about as much as
//     a whole tile's worth of the tensor pipe here, so the issue count, not
//     the math, is what this saves;
//   O^T[128 d, 32]    = V_tile^T . P2: P * 256 split into two e4m3 levels
//     (hi + lo, about bf16 precision) in columns 0-15 and 16-31, summed when
//     the output is folded.
// The per-tile softmax is one long dependent chain (max, exp2, the P split,
// the fold).  With groups of up to 8 heads two softmax warpgroups (WG = 2)
// take alternate tiles of an item, each with its own running max, sum and
// output, so that two chains share every SM sub-partition; at the end of the
// item the second warpgroup hands (m, l, o) to the first through shared
// memory, which merges the two and writes.  Larger groups keep one warpgroup
// (register budget).  Warps: 0 producer, 1 QK issuer, 2 .. 1 + 4 WG softmax,
// then the split merge warp and the PV issuer.
// K and V tiles (2 pages x 64 rows x 128 B each) have rings of their own: a
// K slot is free again once its QK retired, well before the tile's softmax
// and PV are done, so more of shared memory holds loads still in flight.
template <int WG>
struct F8Layout {
    static constexpr int kKSlots = 4;
    static constexpr int kVSlots = 7;
    static constexpr int kNB = 2 * WG;          // S, O and P buffers
    static constexpr int kSlotBytes = 16384;
    static constexpr int kVOff = kKSlots * kSlotBytes;
    static constexpr int kQ3Off = kVOff + kVSlots * kSlotBytes;
    static constexpr int kQ3Bytes = 48 * 128;   // rows = level * 16 + head
    static constexpr int kPOff = kQ3Off + 2 * kQ3Bytes;
    // P, MN-major with 128-byte swizzle: row = key; buffer b takes bytes
    // 32b .. 32b+31 of every row (hi heads, then lo heads), so that all
    // kNB <= 4 buffers share one region and the MMA descriptor of buffer b
    // starts 32b bytes in
    static constexpr int kPBytes = 128 * 128;
    static constexpr int kRedOff = kPOff + kPBytes;
    static constexpr int kRedBytes = 1024;      // per warpgroup: [2][64] maxima, [2][64] sums
    static constexpr int kQscOff = kRedOff + WG * kRedBytes;  // [2][16] floats
    static constexpr int kXOff = kQscOff + 128;  // hand-over, per item parity: o [8][128], m [8], l [8]
    static constexpr int kXFloats = 8 * 128 + 16;
    static constexpr int kXBytes = WG == 2 ? 2 * kXFloats * 4 : 0;
    static constexpr int kBytes = kXOff + kXBytes;
    static constexpr int kSmem = kBytes + 1024;
    static constexpr int kMergeWarp = 2 + 4 * WG;
    static constexpr int kPvWarp = kMergeWarp + 1;
    static constexpr int kThreads = (kPvWarp + 1) * 32;
    // TMEM: S buffers of 48 columns (three query levels x 16) in 64-column
    // slots, then O buffers of 32 columns (hi and lo P levels x 16)
    static constexpr uint32_t kTmemCols = WG == 2 ? 512 : 256;
    __host__ __device__ static constexpr uint32_t s_col(uint32_t b) { return b * 64u; }
    __host__ __device__ static constexpr uint32_t o_col(uint32_t b) { return kNB * 64u + b * 32u; }
    static_assert(kQ3Off % 1024 == 0 && kPOff % 1024 == 0, "swizzle atoms need 1024-byte alignment");
    static_assert(kSmem <= 232448 - 4096, "shared memory per CTA (dynamic + static)");
    static_assert(kKSlots <= 8 && kVSlots <= 8, "barrier slots");
    static_assert(o_col(kNB - 1) + 32 <= kTmemCols, "TMEM columns");
};

enum : int {
    F_KFULL = 0,    // [8] K slot filled
    F_KEMPTY = 8,   // [8] K slot free again (its QK retired)
    F_VFULL = 16,   // [8] V slot filled
    F_VEMPTY = 24,  // [8] V slot free again (its PV retired)
    F_QF = 32,      // [2] query levels written
    F_SF = 34,      // [4] S tile in TMEM
    F_PF = 38,      // [4] P written
    F_OF = 42,      // [4] O tile in TMEM
    F_DONE = 46,    // all QK MMAs retired (teardown)
    F_PW = 47,      // [2] an item's partials written (merge warp)
    F_HD = 49,      // [2] merge warp done with an item
    F_DONE2 = 51,   // all PV MMAs retired (teardown)
    F_COUNT = 52
};

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
    __half2 hh;
    hh = *reinterpret_cast<const __half2*>(&h);
    return __half22float2(hh);
}

template <int NP, int WG>
__global__ void __launch_bounds__(F8Layout<WG>::kThreads, 1)
    decode_f8_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v) {
    using L = F8Layout<WG>;
    static_assert(WG == 1 || NP <= 8, "the hand-over buffer holds 8 heads");
    constexpr int D = 128;
    constexpr int NB = L::kNB, NK = L::kKSlots, NV = L::kVSlots;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[F_COUNT];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_store;
    __shared__ __align__(16) Item items_sh[kItemCache];
    volatile int* abort_sh = &abort_store;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t* meta = a.meta;
    const int B = a.batch;
    const int items_off = items_offset(meta, B);
    int it_lo = 0, it_hi = 0;
    if ((int)blockIdx.x < __ldg(&meta[5])) {
        it_lo = __ldg(&meta[kMetaHeader + 2 * B + 1 + blockIdx.x]);
        it_hi = __ldg(&meta[kMetaHeader + 2 * B + 1 + blockIdx.x + 1]);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(&bars[F_KFULL + s], 1);
            mbar_init(&bars[F_KEMPTY + s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&bars[F_VFULL + s], 1);
            mbar_init(&bars[F_VEMPTY + s], 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&bars[F_SF + i], 1);
            mbar_init(&bars[F_PF + i], 128);
            mbar_init(&bars[F_OF + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[F_QF + i], 128);
            mbar_init(&bars[F_PW + i], 128);
            mbar_init(&bars[F_HD + i], 1);
        }
        mbar_init(&bars[F_DONE], 1);
        mbar_init(&bars[F_DONE2], 1);
        *abort_sh = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == L::kMergeWarp) fill_item_cache(items_sh, a, it_lo, it_hi, items_off, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t g = 0, issued[2] = {0u, 0u};  // tiles whose K / V copies were issued
            bool ok = true;
            for (int j = it_lo; j < it_hi && ok; ++j) {
                const Item it = get_item(items_sh, a, j, it_lo, items_off);
                const int ntiles = item_tiles(it);
                const long long bt_row = (long long)it.b * a.max_pages;
                for (int t = 0; t < ntiles; ++t, ++g) {
                    const int pa0 = it.p0 + 2 * t;
                    const int npg = min(2, it.p1 - pa0);
                    int pid[2];
                    pid[0] = __ldg(&a.block_table[bt_row + pa0]);
                    pid[1] = npg > 1 ? __ldg(&a.block_table[bt_row + pa0 + 1]) : 0;
                    bool valid[2];
                    uint32_t nvalid = 0;
                    for (int i = 0; i < 2; ++i) {
                        valid[i] = i < npg && (unsigned)pid[i] < (unsigned)a.num_pool_pages;
                        if (i < npg && !valid[i]) record(a.status, PA_ERR_DEVICE_BOUNDS);
                        nvalid += valid[i];
                    }
                    int row[2];
                    for (int i = 0; i < 2; ++i) row[i] = (int)(((long long)pid[i] * a.num_kv_heads + it.kvh) * 64);
                    // K, then V, each into the next slot of its ring
#pragma unroll
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        const int ns = kv == 0 ? NK : NV;
                        const int slot = g % ns;
                        uint64_t* empty = &bars[(kv == 0 ? F_KEMPTY : F_VEMPTY) + slot];
                        uint64_t* full = &bars[(kv == 0 ? F_KFULL : F_VFULL) + slot];
                        if (!mbar_wait(empty, ((g / ns) & 1) ^ 1, abort_sh, a.wait_ns)) {
                            fail(a, abort_sh, PA_ERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full, nvalid * 8192u);
                        uint8_t* dst = sm + (kv == 0 ? 0 : L::kVOff) + slot * L::kSlotBytes;
                        for (int i = 0; i < 2; ++i)
                            if (valid[i]) tma_load_2d(dst + i * 8192, kv == 0 ? &map_k : &map_v, full, 0, row[i]);
                        issued[kv] = g + 1;
                    }
                    if (!ok) break;
                }
            }
            // wait for the copies still in flight: with n tiles issued, slot
            // s last took tile n - 1 - ((n - 1 - s) mod slots), if s < n
            for (int kv = 0; kv < 2; ++kv) {
                const int ns = kv == 0 ? NK : NV;
                const uint32_t n = issued[kv];
                for (int s2 = 0; s2 < ns; ++s2) {
                    if ((uint32_t)s2 >= n) continue;
                    const uint32_t last = n - 1 - ((n - 1 - s2) % ns);
                    mbar_wait(&bars[(kv == 0 ? F_KFULL : F_VFULL) + s2], (last / ns) & 1, nullptr, a.wait_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ QK issuer
        // Tile g uses S/O/P buffer g % NB; its softmax is done by warpgroup
        // g % WG.  QK and PV are issued by two threads in two warps, each
        // blocking on its own barriers, so that neither product waits behind
        // the other and no thread spends its time polling (a tcgen05.commit
        // tracks the MMAs of the thread that issues it, so each thread
        // commits its own).  S buffer g % NB is free again once P(g - NB) is
        // written: the softmax read S(g - NB) before that.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_e4m3(128, 48, false, false);
            uint32_t g = 0, qi = 0;
            bool ok = true;
            for (int j = it_lo; j < it_hi && ok; ++j) {
                const int ntiles = item_tiles(get_item(items_sh, a, j, it_lo, items_off));
                if (ntiles == 0) continue;
                if (!mbar_wait(&bars[F_QF + (qi & 1)], (qi >> 1) & 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                const uint32_t qbase = smem_u32(sm + L::kQ3Off + (qi & 1) * L::kQ3Bytes);
                ++qi;
                for (int t = 0; t < ntiles; ++t, ++g) {
                    if (g >= (uint32_t)NB &&
                        !mbar_wait(&bars[F_PF + (g - NB) % NB], ((g - NB) / NB) & 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&bars[F_KFULL + g % NK], (g / NK) & 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kbase = smem_u32(sm + (g % NK) * L::kSlotBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // 32 bytes of d per step; N = 48 = hi, mid, lo levels
                        mma_f8_ss(tbase + L::s_col(g % NB), sdesc_sw128(kbase + kk * 32, 16, 1024),
                                  sdesc_sw128(qbase + kk * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                    mma_commit(&bars[F_SF + g % NB]);
                    mma_commit(&bars[F_KEMPTY + g % NK]);
                }
            }
            if (!ok) fail(a, abort_sh, PA_ERR_TIMEOUT);
            mma_commit(&bars[F_DONE]);
            mbar_wait(&bars[F_DONE], 0, nullptr, a.wait_ns);
        }
    } else if (warp == L::kPvWarp) {
        // ------------------------------------------------------------ PV issuer
        // PV(g) once P(g) is written; its completion hands O(g) to the fold
        // and releases V slot g % NV.
        if (lane == 0) {
            constexpr uint32_t idesc_pv = idesc_e4m3(128, 32, true, true);
            uint32_t total = 0;
            for (int j = it_lo; j < it_hi; ++j) total += (uint32_t)item_tiles(get_item(items_sh, a, j, it_lo, items_off));
            bool ok = true;
            for (uint32_t g = 0; g < total; ++g) {
                if (!mbar_wait(&bars[F_PF + g % NB], (g / NB) & 1, abort_sh, a.wait_ns) ||
                    !mbar_wait(&bars[F_VFULL + g % NV], (g / NV) & 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t vbase = smem_u32(sm + L::kVOff + (g % NV) * L::kSlotBytes);
                const uint32_t pbase = smem_u32(sm + L::kPOff) + (g % NB) * 32u;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)  // 32 keys per step
                    mma_f8_ss(tbase + L::o_col(g % NB), sdesc_sw128(vbase + kk * 4096, 1024, 1024),
                              sdesc_sw128(pbase + kk * 4096, 1024, 1024), idesc_pv, kk > 0);
                mma_commit(&bars[F_OF + g % NB]);
                mma_commit(&bars[F_VEMPTY + g % NV]);
            }
            if (!ok) fail(a, abort_sh, PA_ERR_TIMEOUT);
            mma_commit(&bars[F_DONE2]);
            mbar_wait(&bars[F_DONE2], 0, nullptr, a.wait_ns);
        }
    } else if (warp == L::kMergeWarp) {
        // ------------------------------------------------------------ split merge
        if (a.counters) merge_warp<D>(a, items_sh, it_lo, it_hi, items_off, &bars[F_PW], &bars[F_HD], abort_sh, lane);
    } else {
        // ------------------------------------------------------------ softmax
        const int wg = (warp - 2) >> 2;   // warpgroup: takes the tiles g with g % WG == wg
        const uint32_t wbar = 1 + wg;     // its named barrier (128 threads)
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const int hl = head_of_lane<NP>(lane);
        const bool writer = lane_writes<NP>(lane);
        const int G = a.group;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        float* red = reinterpret_cast<float*>(sm + L::kRedOff + wg * L::kRedBytes);
        float* qsc = reinterpret_cast<float*>(sm + L::kQscOff);

        auto next_nonempty = [&](int j) {
            while (j < it_hi && item_tiles(get_item(items_sh, a, j, it_lo, items_off)) == 0) ++j;
            return j;
        };
        // query of the item's KV group -> three e4m3 levels (rows level*16 + head),
        // by warpgroup 0.  fetch_q only issues the global loads (into pf0/pf1);
        // store_q, one item later, converts and writes, so the load latency is hidden.
        const int qh = row >> 3, qc = row & 7;  // head, 16-element chunk of d
        uint4 pf0 = make_uint4(0, 0, 0, 0), pf1 = make_uint4(0, 0, 0, 0);
        auto fetch_q = [&](int j) {
            const Item it = get_item(items_sh, a, j, it_lo, items_off);
            pf0 = pf1 = make_uint4(0, 0, 0, 0);
            if (qh < G) {
                const long long qrow = (long long)it.b * a.num_q_heads + (long long)it.kvh * G + qh;
                const uint4* src = reinterpret_cast<const uint4*>(a.q + qrow * D) + 2 * qc;
                pf0 = __ldg(src);
                pf1 = __ldg(src + 1);
            }
        };
        auto store_q = [&](uint32_t qidx) {
            uint8_t* qb = sm + L::kQ3Off + (qidx & 1) * L::kQ3Bytes;
            const int h = qh, c = qc;
            float v[16];
            {
                const uint32_t w[8] = {pf0.x, pf0.y, pf0.z, pf0.w, pf1.x, pf1.y, pf1.z, pf1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    v[2 * i] = __uint_as_float(w[i] << 16);
                    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(v[i]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            int e = 0;
            if (mx > 0.f) frexpf(mx, &e);              // mx in [2^(e-1), 2^e)
            const float up = ldexpf(1.f, 8 - e);       // scaled max in [128, 256)
            uint32_t lv[3][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float r0 = v[2 * i] * up, r1 = v[2 * i + 1] * up;  // exact (power of two)
#pragma unroll
                for (int l = 0; l < 3; ++l) {
                    const uint32_t b2 = e4m3x2(r0, r1);
                    const float2 back = e4m3x2_to_f2(b2);
                    r0 -= back.x;
                    r1 -= back.y;
                    if (i & 1) lv[l][i >> 1] |= b2 << 16;
                    else lv[l][i >> 1] = b2;
                }
            }
#pragma unroll
            for (int l = 0; l < 3; ++l) {
                const int qr = l * 16 + h;
                *reinterpret_cast<uint4*>(qb + qr * 128 + ((c ^ (qr & 7)) << 4)) =
                    make_uint4(lv[l][0], lv[l][1], lv[l][2], lv[l][3]);
            }
            if (c == 0) qsc[(qidx & 1) * 16 + h] = ldexpf(1.f, e - 8);
            fence_proxy_async_smem();
            mbar_arrive(&bars[F_QF + (qidx & 1)]);
        };

        int qload = next_nonempty(it_lo);
        uint32_t qload_idx = 0;
        if (wg == 0) {
            for (int k = 0; k < 2 && qload < it_hi; ++k) {
                fetch_q(qload);
                store_q(qload_idx++);
                qload = next_nonempty(qload + 1);
            }
            if (qload < it_hi) fetch_q(qload);
        }
        named_bar_sync(3, 128 * WG);  // query scales of the first items visible to every softmax thread

        // Only barrier results (uniform over the threads that take part) end
        // a loop: a failed wait records the error and raises the abort flag,
        // and the next barrier takes everyone out together.
        uint32_t g0 = 0, qi = 0, npartial = 0, lt = 0;
        bool aborted = false;
        for (int j = it_lo; j < it_hi && !aborted; ++j) {
            const Item it = get_item(items_sh, a, j, it_lo, items_off);
            const int ntiles = item_tiles(it);
            const bool partial = it.nsplit > 1;
            const long long head0 = (long long)it.kvh * G;
            const long long orow = partial ? (long long)(it.split_base + it.s) * a.num_q_heads + head0
                                           : (long long)it.b * a.num_q_heads + head0;
            if (ntiles == 0) {
                if (wg == 0) {
                    for (int h = 0; h < G; ++h) {
                        if (partial) a.o_part[(orow + h) * D + row] = 0.f;
                        else a.out[(orow + h) * D + row] = 0;
                    }
                    if (row < G) {
                        if (partial) a.lse_part[orow + row] = -INFINITY;
                        else if (a.lse) a.lse[orow + row] = -INFINITY;
                    }
                    if (partial && a.counters &&
                        !partials_written(&bars[F_PW], &bars[F_HD], npartial++, abort_sh, a.wait_ns))
                        fail(a, abort_sh, PA_ERR_TIMEOUT);
                }
                continue;
            }
            if (wg == 0 && qi >= 1 && qload < it_hi) {
                store_q(qload_idx++);
                qload = next_nonempty(qload + 1);
                if (qload < it_hi) fetch_q(qload);
            }
            const float base_l2 = a.scale_log2 * __ldg(&a.k_scale[it.kvh]);
            float sl2[NP];
#pragma unroll
            for (int h = 0; h < NP; ++h) sl2[h] = base_l2 * qsc[(qi & 1) * 16 + h];
            ++qi;
            const int key_end = min(it.seq_len, it.p1 * kPage);
            float m[NP], lp[NP], o[NP], alpha_prev[NP];
#pragma unroll
            for (int h = 0; h < NP; ++h) { m[h] = -INFINITY; lp[h] = 0.f; o[h] = 0.f; alpha_prev[h] = 1.f; }

            auto fold = [&](uint32_t k) {
                if (!mbar_wait(&bars[F_OF + k % NB], (k / NB) & 1, abort_sh, a.wait_ns)) fail(a, abort_sh, PA_ERR_TIMEOUT);
                tc_fence_after();
                uint32_t rh[NP], rl[NP];
                tmem_ld_cols<NP>(tbase + lane_addr + L::o_col(k % NB), rh);
                tmem_ld_cols<NP>(tbase + lane_addr + L::o_col(k % NB) + 16, rl);
                tmem_ld_wait();
                reg_fence(rh);
                reg_fence(rl);
#pragma unroll
                for (int h = 0; h < NP; ++h)
                    o[h] = fmaf(o[h], alpha_prev[h], (__uint_as_float(rh[h]) + __uint_as_float(rl[h])) * (1.f / 256.f));
            };

            bool have_prev = false;
            uint32_t gprev = 0;
            const int t0 = (int)((uint32_t)(wg - (int)g0) & (uint32_t)(WG - 1));
            for (int t = t0; t < ntiles; t += WG, ++lt) {
                const uint32_t g = g0 + t;
                const int pa0 = it.p0 + 2 * t;
                const int npg = min(2, it.p1 - pa0);
                const int key = pa0 * kPage + row;
                const bool valid = row < npg * kPage && key < key_end;
                if (!mbar_wait(&bars[F_SF + g % NB], (g / NB) & 1, abort_sh, a.wait_ns))
                    fail(a, abort_sh, PA_ERR_TIMEOUT);
                tc_fence_after();
                uint32_t sh[NP], sm_[NP], slo[NP];  // the three query-level products
                tmem_ld_cols<NP>(tbase + lane_addr + L::s_col(g % NB), sh);
                tmem_ld_cols<NP>(tbase + lane_addr + L::s_col(g % NB) + 16, sm_);
                tmem_ld_cols<NP>(tbase + lane_addr + L::s_col(g % NB) + 32, slo);
                tmem_ld_wait();
                reg_fence(sh);
                reg_fence(sm_);
                reg_fence(slo);
                float x[NP];
#pragma unroll
                for (int h = 0; h < NP; ++h)
                    x[h] = valid ? ((__uint_as_float(sh[h]) + __uint_as_float(sm_[h])) + __uint_as_float(slo[h])) * sl2[h]
                                 : -INFINITY;
                const float wmax = warp_xreduce<NP, true>(x, lane);
                float* rb = red + (lt & 1) * 64;
                if (writer) rb[hl * 4 + q4] = wmax;
                if (named_bar_or(wbar, 128, *abort_sh != 0)) { aborted = true; break; }
                float alpha[NP];
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    const float4 r4 = reinterpret_cast<const float4*>(rb)[h];
                    const float mt = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
                    const float mn = fmaxf(m[h], mt);
                    const bool none = mn == -INFINITY;
                    alpha[h] = none ? 1.f : exp2f(m[h] - mn);
                    x[h] = (none || h >= G) ? 0.f : exp2f(x[h] - mn);
                    lp[h] = fmaf(lp[h], alpha[h], x[h]);
                    m[h] = mn;
                }
                // P * 256 as two e4m3 levels; this key's row: bytes 0-15 hi, 16-31 lo
                uint32_t hw[4] = {0u, 0u, 0u, 0u}, lw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int h = 0; h < NP; h += 2) {
                    const float p0 = x[h] * 256.f, p1 = x[h + 1] * 256.f;
                    const uint32_t hb = e4m3x2(p0, p1);
                    const float2 back = e4m3x2_to_f2(hb);
                    const uint32_t lb = e4m3x2(p0 - back.x, p1 - back.y);
                    hw[h >> 2] |= hb << ((h & 2) * 8);
                    lw[h >> 2] |= lb << ((h & 2) * 8);
                }
                uint8_t* pb = sm + L::kPOff + row * 128;
                const int c0 = 2 * (int)(g % NB);  // this buffer's first 16-byte chunk of the row
                *reinterpret_cast<uint4*>(pb + ((c0 ^ (row & 7)) << 4)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4*>(pb + (((c0 + 1) ^ (row & 7)) << 4)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                if (!valid) {
                    // a dead key's V row may hold anything (NaN included): zero it
                    const int slot = g % NV;
                    mbar_wait(&bars[F_VFULL + slot], (g / NV) & 1, abort_sh, a.wait_ns);
                    uint8_t* vr = sm + L::kVOff + slot * L::kSlotBytes + (row >> 6) * 8192 + (row & 63) * 128;
#pragma unroll
                    for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4*>(vr + i * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&bars[F_PF + g % NB]);
                if (have_prev) fold(gprev);
#pragma unroll
                for (int h = 0; h < NP; ++h) alpha_prev[h] = alpha[h];
                have_prev = true;
                gprev = g;
            }
            g0 += ntiles;
            if (have_prev && !aborted) fold(gprev);
            tc_fence_before();

            // ---- end of item: this warpgroup's sums; with two warpgroups the
            // second hands (m, l, o) to the first, which merges and writes
            const float wsum = warp_xreduce<NP, false>(lp, lane);
            float* rl = red + 128 + (qi & 1) * 64;
            if (writer) rl[hl * 4 + q4] = wsum;
            bool ab = named_bar_or(wbar, 128, *abort_sh != 0);
            float* xo = reinterpret_cast<float*>(sm + L::kXOff) + (qi & 1) * L::kXFloats;
            float l_own[NP];
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                const float4 r4 = reinterpret_cast<const float4*>(rl)[h];
                l_own[h] = (r4.x + r4.y) + (r4.z + r4.w);
            }
            if constexpr (WG == 2) {
                if (wg == 1 && !ab) {
#pragma unroll
                    for (int h = 0; h < NP; ++h) {
                        xo[h * 128 + row] = o[h];
                        if (row == h) {
                            xo[1024 + h] = m[h];
                            xo[1032 + h] = l_own[h];
                        }
                    }
                }
                ab = named_bar_or(3, 256, ab || *abort_sh != 0);
            }
            if (ab) { aborted = true; break; }
            if (wg == 0) {
                const float vs = __ldg(&a.v_scale[it.kvh]);
                float mine_m = -INFINITY, mine_l = 0.f;
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    float mm = m[h], ll = l_own[h], oo = o[h];
                    if constexpr (WG == 2) {
                        const float m1 = xo[1024 + h], l1 = xo[1032 + h], o1 = xo[h * 128 + row];
                        const float mx = fmaxf(mm, m1);
                        const float a0 = mm == -INFINITY ? 0.f : exp2f(mm - mx);
                        const float a1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mx);
                        mm = mx;
                        ll = ll * a0 + l1 * a1;
                        oo = oo * a0 + o1 * a1;
                    }
                    if (h == row) { mine_m = mm; mine_l = ll; }
                    if (h < G) {
                        const float val = ll > 0.f ? oo * (vs / ll) : 0.f;
                        if (partial) a.o_part[(orow + h) * D + row] = val;
                        else a.out[(orow + h) * D + row] = __bfloat16_as_ushort(__float2bfloat16_rn(val));
                    }
                }
                if (row < G) {
                    const float lse = mine_l > 0.f ? (mine_m + log2f(mine_l)) * kLn2 : -INFINITY;
                    if (partial) a.lse_part[orow + row] = lse;
                    else if (a.lse) a.lse[orow + row] = lse;
                }
                if (partial && a.counters &&
                    !partials_written(&bars[F_PW], &bars[F_HD], npartial++, abort_sh, a.wait_ns))
                    fail(a, abort_sh, PA_ERR_TIMEOUT);
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, L::kTmemCols);
    }
}

template <int NP, int WG>
cudaError_t launch_f8_np(const DecodeArgs& a, const CUtensorMap* mk, const CUtensorMap* mv, int grid,
                         cudaStream_t stream) {
    using L = F8Layout<WG>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = ensure_dynamic_smem(decode_f8_kernel<NP, WG>, L::kSmem, configured);
    if (e != cudaSuccess) return e;
    decode_f8_kernel<NP, WG><<<grid, L::kThreads, L::kSmem, stream>>>(a, *mk, *mv);
    return cudaGetLastError();
}

// Merge split partials: L = m + ln sum_s exp(lse_s - m), out = sum_s exp(lse_s - L) o_s.
// One warp per (sequence, query head); sequences with one split were written
// directly by the decode kernel and are skipped.
__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= a.batch * a.num_q_heads) return;
    const int b = w / a.num_q_heads, h = w % a.num_q_heads;
    const int n = __ldg(&a.meta[kMetaHeader + b]);
    if (n <= 1) return;
    const int base = __ldg(&a.meta[kMetaHeader + a.batch + b]);
    float mx = -INFINITY;
    for (int s = 0; s < n; ++s) mx = fmaxf(mx, __ldg(&a.lse_part[(long long)(base + s) * a.num_q_heads + h]));
    const long long orow = (long long)b * a.num_q_heads + h;
    if (mx == -INFINITY) {
        for (int d = lane; d < a.head_dim; d += 32) a.out[orow * a.head_dim + d] = 0;
        if (lane == 0 && a.lse) a.lse[orow] = -INFINITY;
        return;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    for (int s = 0; s < n; ++s) {
        const long long prow = (long long)(base + s) * a.num_q_heads + h;
        const float wgt = __expf(__ldg(&a.lse_part[prow]) - mx);
        wsum += wgt;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int d = lane + 32 * i;
            if (d < a.head_dim) acc[i] = fmaf(wgt, __ldg(&a.o_part[prow * a.head_dim + d]), acc[i]);
        }
    }
    const float inv = 1.f / wsum;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int d = lane + 32 * i;
        if (d < a.head_dim) a.out[orow * a.head_dim + d] = out16(acc[i] * inv, a.f16);
    }
    if (lane == 0 && a.lse) a.lse[orow] = mx + __logf(wsum);
}

__global__ void wait_probe_kernel(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // nothing ever arrives on `bar`: the bounded wait must give up on its own
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, nullptr, limit_ns)) atomicCAS(status, 0, PA_ERR_TIMEOUT);
}

template <int D, bool FP8, int NP>
cudaError_t launch_decode_np(const DecodeArgs& a, const CUtensorMap* mk, const CUtensorMap* mv, const CUtensorMap* mq,
                             int grid, cudaStream_t stream) {
    using L = DecodeLayout<D, FP8>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = ensure_dynamic_smem(decode_kernel<D, FP8, NP>, L::kSmem, configured);
    if (e != cudaSuccess) return e;
    return launch_overlapped(decode_kernel<D, FP8, NP>, dim3(grid), dim3(L::kThreads), L::kSmem, stream, a, *mk, *mv,
                             *mq);
}

// The softmax works on the group's heads padded to 4, 8 or 16 (the MMA N stays 16).
template <int D, bool FP8>
cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap* mk, const CUtensorMap* mv, const CUtensorMap* mq,
                            int grid, cudaStream_t stream) {
    if (a.group <= 4) return launch_decode_np<D, FP8, 4>(a, mk, mv, mq, grid, stream);
    if (a.group <= 8) return launch_decode_np<D, FP8, 8>(a, mk, mv, mq, grid, stream);
    return launch_decode_np<D, FP8, 16>(a, mk, mv, mq, grid, stream);
}

}  // namespace

cudaError_t launch_decode(int head_dim, bool fp8, const DecodeArgs& a, const CUtensorMap* mk, const CUtensorMap* mv,
                          const CUtensorMap* mq, int grid, cudaStream_t stream) {
    if (head_dim == 128 && fp8) {
        if (a.group <= 4) return launch_f8_np<4, 2>(a, mk, mv, grid, stream);
        if (a.group <= 8) return launch_f8_np<8, 2>(a, mk, mv, grid, stream);
        return launch_f8_np<16, 1>(a, mk, mv, grid, stream);
    }
    if (head_dim == 128) return launch_decode_t<128, false>(a, mk, mv, mq, grid, stream);
    return fp8 ? launch_decode_t<64, true>(a, mk, mv, mq, grid, stream)
               : launch_decode_t<64, false>(a, mk, mv, mq, grid, stream);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
    const int warps = a.batch * a.num_q_heads;
    combine_kernel<<<(warps + 3) / 4, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(int* status, uint64_t limit_ns, cudaStream_t stream) {
    wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory.
//
// Some callers own no allocator of their own: a host framework may keep every
// byte of device memory in its own pool and forbid outside allocations, or a
// serving loop may not tolerate the device-wide synchronisation cudaMalloc
// can cause.  pa_decode needs a caller-provided workspace for its split-KV
// partials and status word; pa_decode_noalloc uses instead one scratch array
// that lives in this library's own device memory for as long as the library
// is loaded (every GPU that loads it holds kNoAllocScratchBytes).
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
struct NoAllocSlot {
    unsigned long long ctx_id;  // the context the address was looked up in (0: none yet)
    void* ptr;                  // device address of the scratch array in that context
};
NoAllocSlot g_noalloc_slot[128] = {};  // per device ordinal

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current context (0 if unknown).  A
// context created after cudaDeviceReset gets a new id, and with it a new copy
// of this library's module and of the scratch array.
unsigned long long current_ctx_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// In host code the array's name is only a host-side stand-in; its device
// address has to be asked for with the device current.  That is done once per
// device and context: the first call on a device (or the first after its
// context was reset) looks it up, later calls reuse it.
pa_status noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 128) return PA_ERR_CUDA;
    const unsigned long long id = current_ctx_id();
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocSlot& slot = g_noalloc_slot[dev];
    if (!slot.ptr || id == 0 || slot.ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return PA_ERR_CUDA;
        slot.ptr = p;
        slot.ctx_id = current_ctx_id();  // the lookup has made the device's context current
    }
    *out = slot.ptr;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_decode_shapes* shapes, const pa_decode_plan* plan, const void* q,
                                       const void* k_pool, const void* v_pool, const float* k_scale,
                                       const float* v_scale, const int32_t* block_table, const int32_t* seq_lens,
                                       const int32_t* meta_dev, float scale, void* out, float* lse,
                                       int32_t* status_host, cudaStream_t stream) {
    pa::NvtxRange nvtx_range("pa_decode_noalloc");
    if (!plan) {
        pa::set_last_error("plan must not be NULL");
        return PA_ERR_INVALID_ARG;
    }
    if (plan->workspace_bytes > kNoAllocScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "this plan needs %zu bytes of scratch; pa_decode_noalloc has a fixed %zu-byte scratch "
                 "(use pa_decode with a workspace, or fewer splits)",
                 plan->workspace_bytes, kNoAllocScratchBytes);
        pa::set_last_error(msg);
        return PA_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    pa_status st = noalloc_scratch(&scratch);
    if (st != PA_OK) {
        pa::set_last_error("could not look up the device address of the no-alloc scratch array");
        return st;
    }
    // every host-side check before anything is enqueued
    st = pa::check_decode_call(shapes, plan, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, meta_dev,
                               scale, out, scratch, kNoAllocScratchBytes);
    if (st != PA_OK) return st;
    // the status word must start at zero; the partials are written before read
    if (cudaMemsetAsync(scratch, 0, PA_STATUS_BYTES, stream) != cudaSuccess) {
        pa::set_last_error("clearing the no-alloc status word failed");
        return PA_ERR_CUDA;
    }
    st = pa_decode_attend(shapes, plan, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, meta_dev, scale,
                          out, lse, scratch, kNoAllocScratchBytes, stream);
    if (st != PA_OK) return st;
    st = pa_decode_combine(shapes, plan, meta_dev, out, lse, scratch, kNoAllocScratchBytes, stream);
    if (st != PA_OK || !status_host) return st;
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        pa::set_last_error("reading the no-alloc status word failed");
        return PA_ERR_CUDA;
    }
    *status_host = word;
    return PA_OK;
}
