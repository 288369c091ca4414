// prefill_common.cuh -- pieces shared by the two prefill kernels (one CTA per
// work item; a CTA pair per work item): element packing, the segment of a
// ragged batch, the causal tile count, and work index -> work item.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLn2f = 0.69314718055994531f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// work counters of the persistent prefill, int32 words of the status region
// (bytes 64 and 128 of the workspace): next work item, CTAs finished
constexpr int kPrefillNextWord = 16;
constexpr int kPrefillDoneWord = 32;

// two values as a packed 16-bit pair (low half first): fp16 or bf16
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi, bool f16) {
    if (f16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// the two values of a packed 16-bit pair (low half first): fp16 or bf16
__device__ __forceinline__ void unpack16x2(uint32_t w, bool f16, float& lo, float& hi) {
    if (f16) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        lo = f.x;
        hi = f.y;
    } else {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xFFFF0000u);
    }
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct Seg {
    int q0, q_len, k0, kv_len, off;
};

__device__ __forceinline__ Seg load_seg(const PrefillArgs& a, int b) {
    Seg s;
    s.q0 = __ldg(&a.cu_q[b]);
    s.q_len = __ldg(&a.cu_q[b + 1]) - s.q0;
    s.k0 = __ldg(&a.cu_k[b]);
    s.kv_len = __ldg(&a.cu_k[b + 1]) - s.k0;
    s.off = a.qo_offset ? __ldg(&a.qo_offset[b]) : s.kv_len - s.q_len;
    return s;
}

// KV tiles (of 128 keys) that query rows [r0, r1) of the segment can see.
__device__ __forceinline__ int kv_tiles_for(const Seg& s, int r0, int r1, bool causal) {
    if (r0 >= r1) return 0;
    long long lim = s.kv_len;
    if (causal) {
        const long long c = (long long)s.off + r1;  // keys 0 .. off + r1 - 1
        lim = c < lim ? c : lim;
    }
    if (lim <= 0) return 0;
    return (int)((lim + 127) / 128);
}

// One work item as the producer publishes it to the other roles: a query
// block (a.q_block rows: 256 for one CTA, 512 for a CTA pair) of one segment
// and one query head, split in two halves A and B (the two query tiles of the
// item, each 128 rows per CTA); valid == 0 ends the loop.
struct PItem {
    int valid, b, h, rA, nA, nB;
    Seg sg;
};

// Work index -> item.  Heads come in groups of hg (up to 32); within a group
// the unit rank is the slow index and the head the fast one.  With an order
// from prefill_order_kernel the units come sequence by sequence, longest
// first, so the items in flight together share one sequence's K/V tiles in L2
// across a group of heads.  Returns false for an idle unit (its rows lie past
// the segment).
__device__ __forceinline__ bool make_item(const PrefillArgs& a, int w, PItem& it) {
    const int units = a.num_q_tiles * a.batch;
    const int hg = a.num_q_heads < 32 ? a.num_q_heads : 32;
    const int group = w / (hg * units);
    const int in_group = w % (hg * units);
    const int hg_here = min(hg, a.num_q_heads - group * hg);  // the last group may be narrower
    const int rank = in_group / hg_here;
    const int unit = a.order ? __ldg(&a.order[rank]) : -1;
    const int b = unit >= 0 ? unit % a.batch : rank % a.batch;
    const int pair = unit >= 0 ? unit / a.batch : a.num_q_tiles - 1 - rank / a.batch;
    const Seg sg = load_seg(a, b);
    const int half = a.q_block / 2;
    const int rA = pair * a.q_block;  // first query row of tile A within the segment
    if (rA >= sg.q_len) return false;
    const bool causal = a.causal != 0;
    it.valid = 1;
    it.b = b;
    it.h = group * hg + in_group % hg_here;
    it.rA = rA;
    it.sg = sg;
    it.nA = kv_tiles_for(sg, rA, min(rA + half, sg.q_len), causal);
    it.nB = rA + half < sg.q_len ? kv_tiles_for(sg, rA + half, min(rA + a.q_block, sg.q_len), causal) : 0;
    return true;
}

}  // namespace
}  // namespace pa
