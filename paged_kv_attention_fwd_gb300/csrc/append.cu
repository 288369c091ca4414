// append.cu -- write new tokens' K and V into their pages (FlashMLA "Tensor
// Shapes Reference", section 4: prefill writes into the paged cache; token p
// of a sequence is row p % 64 of page block_table[b, p / 64], "Prefill to
// Cache Mapping").  A copy, so HBM-bound: one warp per (new token, KV head);
// lanes 0-15 move the key row and lanes 16-31 the value row in 16-byte pieces
// (for e4m3 pools each piece of 8 elements is divided by the head's scale and
// rounded to e4m3, nearest even, saturating).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
    const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= (long long)a.total_new * a.num_kv_heads) return;
    const int tok = (int)(w / a.num_kv_heads), h = (int)(w % a.num_kv_heads);
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
    const long long dst_row = ((long long)page * a.num_kv_heads + h) * kPage + pos % kPage;
    const long long src_row = (long long)tok * a.num_kv_heads + h;
    const bool is_v = lane >= 16;
    const uint16_t* src = (is_v ? a.v_new : a.k_new) + src_row * a.head_dim;
    const int pieces = a.head_dim / 8;  // 8 elements (16 source bytes) per piece
    if (!a.fp8) {
        uint16_t* dst = static_cast<uint16_t*>(is_v ? a.v_pool : a.k_pool) + dst_row * a.head_dim;
        for (int i = lane & 15; i < pieces; i += 16)
            reinterpret_cast<uint4*>(dst)[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
    } else {
        uint8_t* dst = static_cast<uint8_t*>(is_v ? a.v_pool : a.k_pool) + dst_row * a.head_dim;
        const float scale = __ldg(&(is_v ? a.v_scale : a.k_scale)[h]);
        for (int i = lane & 15; i < pieces; i += 16) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[2] = {0u, 0u};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float x0 = __fdiv_rn(__uint_as_float(w4[k] << 16), scale);
                const float x1 = __fdiv_rn(__uint_as_float(w4[k] & 0xFFFF0000u), scale);
                const uint32_t b2 =
                    (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
                out[k >> 1] |= b2 << ((k & 1) * 16);
            }
            reinterpret_cast<uint2*>(dst)[i] = make_uint2(out[0], out[1]);
        }
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    const long long warps = (long long)a.total_new * a.num_kv_heads;
    append_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
