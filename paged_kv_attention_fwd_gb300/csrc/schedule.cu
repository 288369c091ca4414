// schedule.cu -- the split-KV schedule computed on the device from device
// sequence lengths, so a decode step can be captured once in a CUDA graph and
// replayed with new lengths (MATE's static plans: capacities fixed at plan
// time, per-call lengths in device buffers, no host reads in the captured
// region).  Same split rule and packed layout as pa_get_metadata; the items,
// sorted longest first, are dealt to the CTAs in "snake" rounds (0..grid-1,
// then grid-1..0, ...) instead of least-loaded-first, which is sequential.
// One CTA of 128 to 1024 threads (a power of two the launcher sizes to the
// batch and the split capacity); shared memory holds the sort keys and the
// per-sequence page counts, split counts and split offsets.
#include <algorithm>

#include "pa_internal.h"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kMaxThreads = 1024;
constexpr int kMaxPer = 16;  // sort keys per thread: 16384 splits / 1024 threads

__device__ __forceinline__ long long block_sum(long long v, long long* tmp) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) tmp[w] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        long long t = threadIdx.x < (blockDim.x >> 5) ? tmp[threadIdx.x] : 0;
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) tmp[0] = t;
    }
    __syncthreads();
    const long long t = tmp[0];
    __syncthreads();
    return t;
}

// out[i] = in[0] + ... + in[i-1] for i in [0, n]
__device__ void block_exclusive_scan(const int* in, int* out, int n, int* tmp) {
    const int nw = blockDim.x >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += in[i];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    int x = local;  // inclusive scan within the warp
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += y;
    }
    if (l == 31) tmp[w] = x;
    __syncthreads();
    if (threadIdx.x < 32) {  // inclusive scan of the warp totals
        int t = threadIdx.x < nw ? tmp[threadIdx.x] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (threadIdx.x >= o) t += y;
        }
        tmp[threadIdx.x] = t;
    }
    __syncthreads();
    int run = (x - local) + (w > 0 ? tmp[w - 1] : 0);
    for (int i = lo; i < hi; ++i) {
        out[i] = run;
        run += in[i];
    }
    if (threadIdx.x == 0) out[n] = tmp[nw - 1];
    __syncthreads();
}

// T threads; below 1024 the launcher gives at most one sort key a thread
template <int T>
__global__ void __launch_bounds__(T, 1)
    schedule_kernel(const int32_t* seq_lens, int B, int Hk, int max_pages, int cps, int cap, int forced,
                    int p2cap, int32_t* meta) {
    constexpr int kPer = T == kMaxThreads ? kMaxPer : 4;
    allow_dependents_launch();  // the decode kernel's prologue overlaps this one
    extern __shared__ unsigned long long dyn[];
    unsigned long long* key = dyn;                              // [p2cap >= the split count]
    int* pages = reinterpret_cast<int*>(dyn + p2cap);           // [B]
    int* nsp = pages + B;                                       // [B]
    int* ind = nsp + B;                                         // [B + 1]
    __shared__ long long tmp64[32];
    __shared__ int tmp32[32];

    long long local = 0;
    for (int b = threadIdx.x; b < B; b += T) {
        const int len = max(seq_lens[b], 0);
        const int p = min((len + kPage - 1) / kPage, max_pages);
        pages[b] = p;
        local += p;
    }
    const long long units = block_sum(local, tmp64) * Hk;
    const long long shares = 2LL * cap;  // two items per CTA share
    const long long chunk = max(4LL, (units + shares - 1) / shares);
    for (int b = threadIdx.x; b < B; b += T) {
        const int p = pages[b];
        int n;
        if (p <= 1) n = 1;
        else if (forced > 0) n = min(min(forced, p), PA_MAX_SPLITS);
        else n = (int)min((long long)PA_MAX_SPLITS, (p + chunk - 1) / chunk);
        nsp[b] = n;
    }
    __syncthreads();
    block_exclusive_scan(nsp, ind, B, tmp32);
    const int total = ind[B];
    const int items = total * Hk;
    const int grid = min(items, cap);
    // The host rule orders work items by cost descending, then item index
    // ascending.  An item's cost depends only on its split, and the Hk items
    // of split g hold the consecutive indices g * Hk .. g * Hk + Hk - 1, so
    // that order is the splits' order (cost descending, split index
    // ascending) with each split expanded over its KV heads in order: sort the
    // splits, not the items.
    // keys: [63:32] 0x7FFFFFFF - cost, [31:14] b, [13:0] g (the host checks
    // give g < 16384 and b < 8192); b never decreases as g grows, so the low
    // word orders as g does and the final pass needs no search for b
    int p2 = 1;
    while (p2 < total) p2 <<= 1;
    for (int g = threadIdx.x; g < p2; g += T) {
        unsigned long long k = ~0ull;
        if (g < total) {
            int lo = 0, hi = B - 1;  // last b with ind[b] <= g
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (ind[mid] <= g) lo = mid;
                else hi = mid - 1;
            }
            const int b = lo, s = g - ind[b], n = nsp[b], p = pages[b];
            const int cost = (int)(((long long)(s + 1) * p) / n - ((long long)s * p) / n) + 1;
            k = ((unsigned long long)(unsigned)(0x7FFFFFFF - cost) << 32) | ((unsigned)b << 14) | (unsigned)g;
        }
        key[g] = k;
    }
    __syncthreads();
    // Bitonic sort.  The keys are unique, so the sorted order is too and any
    // sorting network reproduces the host rule's order.  Thread t holds the
    // keys at positions k * T + t in registers (T >= p2 / 16 by the
    // launcher); the stages whose partner (position ^ stride) lies in the same
    // warp run as shuffles with no barrier, in the warps that hold keys only,
    // the others through shared memory.
    const int per = p2 > T ? p2 / T : 1;
    const bool holds = (int)(threadIdx.x & ~31u) < p2;  // warp-uniform
    unsigned long long kr[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int pos = k * T + threadIdx.x;
        kr[k] = (k < per && pos < p2) ? key[pos] : ~0ull;
    }
    for (int size = 2; size <= p2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride < 32) {
                if (!holds) continue;
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    if (k >= per) break;
                    const int pos = k * T + threadIdx.x;
                    const unsigned long long other = __shfl_xor_sync(0xffffffffu, kr[k], stride);
                    const bool keep_min = ((pos & stride) == 0) == ((pos & size) == 0);
                    kr[k] = keep_min ? min(kr[k], other) : max(kr[k], other);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    if (k >= per) break;
                    const int pos = k * T + threadIdx.x;
                    if (pos < p2) key[pos] = kr[k];
                }
                __syncthreads();
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    if (k >= per) break;
                    const int pos = k * T + threadIdx.x;
                    if (pos < p2) {
                        const unsigned long long other = key[pos ^ stride];
                        const bool keep_min = ((pos & stride) == 0) == ((pos & size) == 0);
                        kr[k] = keep_min ? min(kr[k], other) : max(kr[k], other);
                    }
                }
                __syncthreads();
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        if (k >= per) break;
        const int pos = k * T + threadIdx.x;
        if (pos < p2) key[pos] = kr[k];
    }
    __syncthreads();
    // packed metadata: header, n_splits, split_indptr, cta_indptr, items
    if (threadIdx.x == 0) {
        meta[0] = kMetaMagic;
        meta[1] = B;
        meta[2] = Hk;
        meta[3] = total;
        meta[4] = items;
        meta[5] = grid;
        meta[6] = (int)min(chunk, (long long)0x7FFFFFFF);
        meta[7] = cps;
    }
    for (int b = threadIdx.x; b < B; b += T) meta[kMetaHeader + b] = nsp[b];
    for (int b = threadIdx.x; b <= B; b += T) meta[kMetaHeader + B + b] = ind[b];
    const int full = items / grid, rem = items % grid;
    const bool last_even = (full & 1) == 0;
    int32_t* cta_ptr = meta + kMetaHeader + 2 * B + 1;
    for (int c = threadIdx.x; c <= grid; c += T)
        cta_ptr[c] = c * full + (last_even ? min(c, rem) : max(0, c - (grid - rem)));
    int32_t* out_items = cta_ptr + grid + 1;
    for (int r = threadIdx.x; r < items; r += T) {
        const unsigned long long kk = key[r / Hk];
        const int g = (int)(kk & 0x3FFFu), b = (int)((kk >> 14) & 0x3FFFFu), kvh = r % Hk;
        const int rnd = r / grid, pos = r % grid;
        const int c = (rnd & 1) == 0 ? pos : grid - 1 - pos;
        const int slot = c * full + (last_even ? min(c, rem) : max(0, c - (grid - rem))) + rnd;
        out_items[2 * slot] = b;
        out_items[2 * slot + 1] = ((g - ind[b]) << 16) | kvh;
    }
}

// Block table rows from a flat list of page ids (MATE msa_interface,
// _build_page_table_from_flat_kv_indices, page counts as in _page_counts):
// sequence b owns the next ceil(kv_lens[b] / 64) ids of the list, in order, in
// the first columns of its row; every other entry is 0.  Every CTA scans the
// page counts into shared memory (int64 starts, one thread per contiguous run
// of sequences), then the grid fills the table with coalesced stores; CTA 0
// checks the list against the counts.
constexpr int kPtThreads = 1024;

__global__ void __launch_bounds__(kPtThreads) page_table_kernel(const int32_t* __restrict__ kv_indices,
                                                                int64_t num_indices, const int32_t* __restrict__ kv_lens,
                                                                int B, int max_pages, int32_t* __restrict__ bt,
                                                                int* status) {
    extern __shared__ long long start[];  // [B + 1]
    __shared__ long long warp_sum[kPtThreads / 32];
    allow_dependents_launch();  // an attention kernel after it may start its prologue
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int per = (B + kPtThreads - 1) / kPtThreads;
    const int b0 = min(B, t * per), b1 = min(B, b0 + per);
    bool bad = false;
    long long mine = 0;
    for (int b = b0; b < b1; ++b) {
        const int len = __ldg(&kv_lens[b]);
        bad |= len < 0;
        const long long c = len > 0 ? ((long long)len + kPage - 1) / kPage : 0;
        bad |= c > max_pages;
        mine += c;
    }
    // exclusive scan of the per-thread totals
    long long x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    long long run = x - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
    for (int b = b0; b < b1; ++b) {
        start[b] = run;
        const int len = __ldg(&kv_lens[b]);
        run += len > 0 ? ((long long)len + kPage - 1) / kPage : 0;
    }
    if (t == kPtThreads - 1) start[B] = warp_sum[31];
    __syncthreads();
    if (blockIdx.x == 0) {
        const bool any_bad = __syncthreads_or(bad) || start[B] != num_indices;
        if (t == 0 && any_bad) atomicCAS(status, 0, PA_ERR_DEVICE_BOUNDS);
    }
    const long long total = (long long)B * max_pages;
    for (long long e = (long long)blockIdx.x * kPtThreads + t; e < total; e += (long long)gridDim.x * kPtThreads) {
        const int b = (int)(e / max_pages), c = (int)(e - (long long)b * max_pages);
        const long long src = start[b] + c;
        const bool live = c < start[b + 1] - start[b] && src < num_indices;
        bt[e] = live ? __ldg(&kv_indices[src]) : 0;
    }
}

}  // namespace

size_t schedule_smem_bytes(int B, int p2cap) { return (size_t)p2cap * 8 + (size_t)(3 * B + 1) * 4; }

cudaError_t launch_schedule(const int32_t* seq_lens, int B, int Hk, int max_pages, int cps, int cap, int forced,
                            int p2cap, int32_t* meta, cudaStream_t stream) {
    const size_t smem = schedule_smem_bytes(B, p2cap);
    // a power of two with one sort key and at most 4 sequences a thread, up to
    // 1024 threads (then at most kMaxPer = 16 keys, p2cap <= 16384); the e4m3
    // decode workload's 166 splits ran 12.3 us on 128 threads, 10.3 on 256
    int threads = 128;
    while (threads < kMaxThreads && (threads < p2cap || threads * 4 < B)) threads <<= 1;
    if (threads * (threads == kMaxThreads ? kMaxPer : 4) < p2cap) return cudaErrorInvalidValue;
    // the attribute is per kernel and device: set it once per device, to the
    // largest size the host checks allow (16384 splits, 8192 sequences)
    static std::atomic<uint64_t> configured[4] = {};
    auto go = [&](auto kernel, std::atomic<uint64_t>& done) {
        cudaError_t e = ensure_dynamic_smem(kernel, (int)schedule_smem_bytes(kMaxBatch, 16384), done);
        if (e != cudaSuccess) return e;
        kernel<<<1, threads, smem, stream>>>(seq_lens, B, Hk, max_pages, cps, cap, forced, p2cap, meta);
        return cudaGetLastError();
    };
    switch (threads) {
        case 128: return go(schedule_kernel<128>, configured[0]);
        case 256: return go(schedule_kernel<256>, configured[1]);
        case 512: return go(schedule_kernel<512>, configured[2]);
        default: return go(schedule_kernel<1024>, configured[3]);
    }
}

cudaError_t launch_page_table(const int32_t* kv_indices, int64_t num_indices, const int32_t* kv_lens, int B,
                              int max_pages, int32_t* block_table, int* status, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = ensure_dynamic_smem(page_table_kernel, (int)((kMaxBatch + 1) * sizeof(long long)), configured);
    if (e != cudaSuccess) return e;
    const long long total = (long long)B * max_pages;
    const long long want = (total + 8 * kPtThreads - 1) / (8 * kPtThreads);
    const unsigned grid = (unsigned)std::max(1LL, std::min(want, 256LL));
    page_table_kernel<<<grid, kPtThreads, (size_t)(B + 1) * sizeof(long long), stream>>>(
        kv_indices, num_indices, kv_lens, B, max_pages, block_table, status);
    return cudaGetLastError();
}

}  // namespace pa
