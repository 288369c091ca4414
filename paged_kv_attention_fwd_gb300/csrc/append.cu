// append.cu -- write new tokens' K and V into their pages (FlashMLA "Tensor
// Shapes Reference", section 4: prefill writes into the paged cache; token p
// of a sequence is row p % 64 of page block_table[b, p / 64], "Prefill to
// Cache Mapping").  A copy, so HBM-bound: one warp per (new token, group of up
// to 4 KV heads).  The warp finds the token's sequence, position and page
// once, then every lane issues all of its 16-byte loads (key and value rows of
// the group's heads, 8 elements each) before any store, so several loads per
// lane are in flight.  For e4m3 pools each piece of 8 elements is divided by
// the head's scale and rounded to e4m3, nearest even, saturating.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pa_internal.h"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr int kHeadsPerWarp = 4;
constexpr int kPiecesPerLane = kHeadsPerWarp * 2 * (128 / 8) / 32;  // D = 128: 4

// grid: x = tokens / 8 (one warp each), y = group of kHeadsPerWarp KV heads
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
    allow_dependents_launch();  // an attention kernel after it may start its prologue
    const int hk = a.num_kv_heads;
    const int tok = (int)(blockIdx.x * 8u + (threadIdx.x >> 5));
    const int lane = threadIdx.x & 31;
    if (tok >= a.total_new) return;
    const int h0 = (int)blockIdx.y * kHeadsPerWarp;
    const int nh = min(kHeadsPerWarp, hk - h0);
    // segment holding this token: last b with cu[b] <= tok
    int lo = 0, hi = a.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(&a.cu_new[mid]) <= tok) lo = mid;
        else hi = mid - 1;
    }
    const int b = lo;
    const long long pos = (long long)__ldg(&a.start_pos[b]) + (tok - __ldg(&a.cu_new[b]));
    if (pos < 0 || pos / kPage >= a.max_pages) {
        if (lane == 0) atomicCAS(a.status, 0, PA_ERR_DEVICE_BOUNDS);
        return;
    }
    const int page = __ldg(&a.block_table[(long long)b * a.max_pages + pos / kPage]);
    if ((unsigned)page >= (unsigned)a.num_pool_pages) {
        if (lane == 0) atomicCAS(a.status, 0, PA_ERR_DEVICE_BOUNDS);
        return;
    }
    const int lg = a.head_dim == 128 ? 4 : 3;  // log2 of the pieces of 8 elements (16 source bytes) in a row
    const int pieces = 1 << lg;
    const int total = nh * 2 * pieces;         // key and value rows of the group's heads
    // all loads first: piece idx = lane + 32 i -> head h0 + idx / (2 pieces), row (key, value), piece
    uint4 v[kPiecesPerLane];
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
        const int idx = lane + 32 * i;
        if (idx < total) {
            const int hl = idx >> (lg + 1), rem = idx & (2 * pieces - 1);
            const uint16_t* src = (rem >= pieces ? a.v_new : a.k_new) + ((long long)tok * hk + h0 + hl) * a.head_dim;
            v[i] = __ldg(reinterpret_cast<const uint4*>(src) + (rem & (pieces - 1)));
        }
    }
#pragma unroll
    for (int i = 0; i < kPiecesPerLane; ++i) {
        const int idx = lane + 32 * i;
        if (idx >= total) continue;
        const int hl = idx >> (lg + 1), rem = idx & (2 * pieces - 1), piece = rem & (pieces - 1);
        const bool is_v = rem >= pieces;
        const int h = h0 + hl;
        const long long dst_row = ((long long)page * hk + h) * kPage + pos % kPage;
        if (!a.fp8) {
            uint16_t* dst = static_cast<uint16_t*>(is_v ? a.v_pool : a.k_pool) + dst_row * a.head_dim;
            reinterpret_cast<uint4*>(dst)[piece] = v[i];
        } else {
            uint8_t* dst = static_cast<uint8_t*>(is_v ? a.v_pool : a.k_pool) + dst_row * a.head_dim;
            const float scale = __ldg(&(is_v ? a.v_scale : a.k_scale)[h]);
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t out[2] = {0u, 0u};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float x0 = __fdiv_rn(__uint_as_float(w4[k] << 16), scale);
                const float x1 = __fdiv_rn(__uint_as_float(w4[k] & 0xFFFF0000u), scale);
                const uint32_t b2 =
                    (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
                out[k >> 1] |= b2 << ((k & 1) * 16);
            }
            reinterpret_cast<uint2*>(dst)[piece] = make_uint2(out[0], out[1]);
        }
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    const unsigned groups = (unsigned)((a.num_kv_heads + kHeadsPerWarp - 1) / kHeadsPerWarp);
    append_kernel<<<dim3((unsigned)((a.total_new + 7) / 8), groups), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
