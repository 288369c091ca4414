// prefill.cu -- causal (or full) attention for ragged query segments on sm_103a:
// chunked prefill against the paged cache (FlashMLA "Tensor Shapes Reference",
// section 4 mha_fwd_kvcache: K/V gathered through block_table, "Prefill to
// Cache Mapping"), ragged prefill (MATE dense mode, flash_attn_varlen_func)
// and the MLA shape whose 64-wide rope key is shared by all heads (Modular
// flare_mla_prefill: q depth 192 = 128 per-head + 64 shared, output depth 128),
// also with the per-head parts of q and k in e4m3 (its overload with q_nope,
// q_rope, q_scale and k_scales; one fp32 scale per head) or with the rope key
// in e4m3 (its overload with k_rope_scales; one fp32 scale per key token,
// expanded beforehand into two bf16 levels).
//
// Work item: (segment b, 256-row query block, query head h), two 128-row
// query tiles A and B that share every K/V tile.  Persistent: one CTA per SM
// takes items from a counter until none is left.
//
//   warp 0     producer: takes the items and publishes them to the other
//              warps, TMA of each item's two query tiles, then 128-key K and
//              V tiles into separate rings (paged: two 64-row page slabs per
//              tile through block_table; ragged: 3-D boxes over [T, H, D])
//   warp 1     MMA issuer (tcgen05, fp32 accumulators in TMEM, 512 columns):
//                S_X[128 q, 128 keys] = Q_X . K^T          (both from smem)
//                O_X[128 q, 128 dv]  += P_X . V            (P_X from TMEM)
//              issue order QK_A(j+1) right after PV_A(j), so the softmax of
//              one tile overlaps the other tile's MMAs
//   warps 2-5  softmax of tile A, warps 6-9 softmax of tile B: one query row
//              per thread (its TMEM lane), row max and sum without any
//              cross-thread exchange; P (bf16 or fp16) is stored over the S
//              columns it replaces (keys 0..63 -> columns 0..31, keys 64..127
//              -> columns 64..95);
//              O is rescaled in TMEM only when the running max grows by more
//              than 2^8 (otherwise the stale max stays exact and cheaper);
//              the query tile that takes an item's last K/V tile first zeroes
//              that tile's dead V rows
//
// Query row i of segment b sees key j iff j < kv_len and (not causal or
// j <= qo_offset + i), qo_offset defaulting to kv_len - q_len (MATE
// _normalize_qo_offset / _resolve_seqused_k).  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_internal.h"
#include "pa_launch.h"
#include "pa_ptx.cuh"
#include "prefill_common.cuh"

namespace pa {
namespace {

enum : int {
    P_QF = 0,   // the item's query tiles landed
    P_KF = 1,   // [2]
    P_KE = 3,   // [2]
    P_VF = 5,   // [2]
    P_VE = 7,   // [2]
    P_QE = 9,   // query buffers free again (the item's last QK retired)
    P_SF = 10,  // [2] S_A, S_B ready
    P_PF = 12,  // [2] P_A, P_B written
    P_OD = 14,  // [2] PV_A, PV_B retired
    P_DONE = 16,
    P_QS = 17,  // [2] e4m3 MLA: query tile A / B rope part rescaled
    P_IF = 19,  // [2] item slot published
    P_IE = 21,  // [2] item slot read by every consumer
    P_COUNT = 23
};

// F8 (MLA only): a key row is 128 e4m3 bytes (the per-head part) then 64 bf16
// (the rope part); a query row the same plus a third chunk: its rope part,
// divided by the head's scale, is held as two bf16 levels hi + lo (chunks 1
// and 2), so the division costs no precision.
// R8 (MLA only): the rope key arrives as two bf16 levels, hi and lo, expanded
// from e4m3 codes and per-token scales before the launch; a key row is the
// two per-head chunks, then hi, then lo, and the query's rope chunk meets both.
template <bool ROPE, bool F8, bool R8 = false>
struct PrefillLayout {
    static constexpr int kDqk = ROPE ? 192 : 128;
    static constexpr int kQChunks = F8 ? 3 : kDqk / 64;
    static constexpr int kKChunks = F8 ? 2 : kDqk / 64 + (R8 ? 1 : 0);
    static constexpr int kTile = 16384;                 // 128 rows x 128 bytes
    static constexpr int kQBytes = kQChunks * kTile;    // one 128-row query tile
    static constexpr int kKBytes = kKChunks * kTile;    // one 128-key K tile
    static constexpr int kVBytes = 2 * kTile;           // one 128-key V tile (dv 128)
    static constexpr int kNK = (ROPE && !F8) ? 1 : 2;
    static constexpr int kNV = 2;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + kNK * kKBytes;
    static constexpr int kBytes = kVOff + kNV * kVBytes;
    static constexpr int kSmem = kBytes + 1024;
    static_assert(kSmem + 512 <= 232448, "shared memory per CTA (dynamic + static)");
    static constexpr int kThreads = 320;
};

// Persistent: one CTA per SM takes work items from a counter in the status
// region until none is left.  Every barrier's phase runs on across items,
// so the producer loads the next item's query and first K/V tiles while the
// current item's last tiles and output are still in progress.
template <bool ROPE, bool PAGED, bool F8, bool R8, bool F16>
__global__ void __launch_bounds__(320, 1)
    prefill_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_r, const __grid_constant__ CUtensorMap map_qr) {
    static_assert(!F8 || (ROPE && !PAGED), "e4m3 query/key parts: MLA with ragged keys only");
    static_assert(!R8 || (ROPE && !PAGED && !F8), "two-level rope key: bf16 MLA with ragged keys only");
    static_assert(!F16 || (!F8 && !R8), "the e4m3 variants take bf16 parts");
    using L = PrefillLayout<ROPE, F8, R8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[P_COUNT];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_store;
    __shared__ PItem item_q[2];
    volatile int* abort_sh = &abort_store;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = a.num_q_tiles * a.batch * a.num_q_heads;  // work items
    int* next_item = a.status + kPrefillNextWord;
    int* ctas_done = a.status + kPrefillDoneWord;

    if (threadIdx.x == 0) {
        mbar_init(&bars[P_QF], 1);
        mbar_init(&bars[P_QE], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[P_KF + i], 1);
            mbar_init(&bars[P_KE + i], 1);
            mbar_init(&bars[P_VF + i], 1);
            mbar_init(&bars[P_VE + i], 1);
            mbar_init(&bars[P_SF + i], 1);
            mbar_init(&bars[P_PF + i], 128);
            mbar_init(&bars[P_OD + i], 1);
            mbar_init(&bars[P_QS + i], 128);
            mbar_init(&bars[P_IF + i], 1);
            mbar_init(&bars[P_IE + i], 9);  // the MMA thread and one lane of each softmax warp
        }
        mbar_init(&bars[P_DONE], 1);
        *abort_sh = 0;
        fence_barrier_init();
    }
    // launched as a programmatic dependent (of the unit-order kernel, or of
    // whatever the stream ran before): nothing global and no TMEM before this
    grid_dependency_wait();
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;
    // TMEM columns: S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512)
    auto s_col = [](int x) { return (uint32_t)(x * 128); };
    auto o_col = [](int x) { return (uint32_t)(256 + x * 128); };

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            bool ok = true;
            uint32_t k = 0;                          // items published
            uint32_t gt = 0;                         // K/V tiles of the items before this one
            uint32_t q_loads = 0, k_loads = 0, v_loads = 0;  // copies issued, for the drain
            for (;;) {
                PItem it;
                it.valid = 0;
                for (;;) {  // the next item that has rows
                    const int w = atomicAdd(next_item, 1);
                    if (w >= W) break;
                    if (make_item(a, w, it)) break;
                }
                // slot k & 1 is free once every consumer has read item k - 2
                if (!mbar_wait(&bars[P_IE + (k & 1)], ((k >> 1) & 1) ^ 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                item_q[k & 1] = it;
                mbar_arrive(&bars[P_IF + (k & 1)]);  // release: the consumers' wait sees the item
                if (!it.valid) break;
                const Seg& sg = it.sg;
                const int h = it.h, kvh = h / a.group;
                const int nkv = max(it.nA, it.nB);
                const int ntq = it.rA + 128 < sg.q_len ? 2 : 1;
                // query tiles, once the previous item's last QK retired
                if (k > 0 && !mbar_wait(&bars[P_QE], (k - 1) & 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bars[P_QF], ntq * (F8 ? 2 * L::kTile : L::kQBytes));
                for (int x = 0; x < ntq; ++x) {
                    uint8_t* qt = sm + L::kQOff + x * L::kQBytes;
                    if constexpr (F8) {
                        tma_load_3d(qt, &map_q, &bars[P_QF], 0, h, sg.q0 + it.rA + x * 128);             // q_nope e4m3
                        tma_load_3d(qt + L::kTile, &map_qr, &bars[P_QF], 0, h, sg.q0 + it.rA + x * 128);  // q_rope bf16
                    } else {
                        for (int c = 0; c < L::kQChunks; ++c)
                            tma_load_3d(qt + c * L::kTile, &map_q, &bars[P_QF], c * 64, h, sg.q0 + it.rA + x * 128);
                    }
                }
                q_loads = k + 1;
                const int kv_pages = (sg.kv_len + kPage - 1) / kPage;
                for (int j = 0; j < nkv && ok; ++j) {
                    const uint32_t g = gt + j;
                    // page ids of this tile (paged keys)
                    int pid[2] = {-1, -1};
                    if (PAGED) {
                        for (int i = 0; i < 2; ++i) {
                            const int p = 2 * j + i;
                            if (p < kv_pages && p < a.max_pages) {
                                const int id = __ldg(&a.block_table[(long long)it.b * a.max_pages + p]);
                                if ((unsigned)id < (unsigned)a.num_pool_pages) pid[i] = id;
                                else atomicCAS(a.status, 0, PA_ERR_DEVICE_BOUNDS);
                            } else if (p < kv_pages) {
                                atomicCAS(a.status, 0, PA_ERR_DEVICE_BOUNDS);
                            }
                        }
                    }
                    const int npid = (pid[0] >= 0) + (pid[1] >= 0);
                    // K tile
                    const int ks = g % L::kNK;
                    if (!mbar_wait(&bars[P_KE + ks], ((g / L::kNK) & 1) ^ 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    uint64_t* kf = &bars[P_KF + ks];
                    uint8_t* kt = sm + L::kKOff + ks * L::kKBytes;
                    if (PAGED) {
                        mbar_arrive_expect_tx(kf, npid * 2 * 8192);
                        for (int i = 0; i < 2; ++i)
                            if (pid[i] >= 0)
                                for (int c = 0; c < 2; ++c)
                                    tma_load_2d(kt + c * L::kTile + i * 8192, &map_k, kf, c * 64,
                                                (int)(((long long)pid[i] * a.num_kv_heads + kvh) * 64));
                    } else if constexpr (F8) {
                        mbar_arrive_expect_tx(kf, L::kKBytes);
                        tma_load_3d(kt, &map_k, kf, 0, kvh, sg.k0 + j * 128);           // k_nope e4m3
                        tma_load_2d(kt + L::kTile, &map_r, kf, 0, sg.k0 + j * 128);    // k_rope bf16
                    } else {
                        mbar_arrive_expect_tx(kf, L::kKBytes);
                        for (int c = 0; c < 2; ++c)
                            tma_load_3d(kt + c * L::kTile, &map_k, kf, c * 64, kvh, sg.k0 + j * 128);
                        if (ROPE) tma_load_2d(kt + 2 * L::kTile, &map_r, kf, 0, sg.k0 + j * 128);
                        if (R8) tma_load_2d(kt + 3 * L::kTile, &map_qr, kf, 0, sg.k0 + j * 128);  // rope lo level
                    }
                    k_loads = g + 1;
                    // V tile
                    const int vs = g % L::kNV;
                    if (!mbar_wait(&bars[P_VE + vs], ((g / L::kNV) & 1) ^ 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    uint64_t* vf = &bars[P_VF + vs];
                    uint8_t* vt = sm + L::kVOff + vs * L::kVBytes;
                    if (PAGED) {
                        mbar_arrive_expect_tx(vf, npid * 2 * 8192);
                        for (int i = 0; i < 2; ++i)
                            if (pid[i] >= 0)
                                for (int c = 0; c < 2; ++c)
                                    tma_load_2d(vt + c * L::kTile + i * 8192, &map_v, vf, c * 64,
                                                (int)(((long long)pid[i] * a.num_kv_heads + kvh) * 64));
                    } else {
                        mbar_arrive_expect_tx(vf, L::kVBytes);
                        for (int c = 0; c < 2; ++c)
                            tma_load_3d(vt + c * L::kTile, &map_v, vf, c * 64, kvh, sg.k0 + j * 128);
                    }
                    v_loads = g + 1;
                }
                if (!ok) break;
                gt += nkv;
                ++k;
            }
            if (!ok) {
                *abort_sh = 1;
                atomicCAS(a.status, 0, PA_ERR_TIMEOUT);
            }
            // every issued copy must land before the CTA may exit: with n
            // tiles issued, ring slot s last took tile n - 1 - ((n - 1 - s) mod slots)
            if (q_loads > 0) mbar_wait(&bars[P_QF], (q_loads - 1) & 1, nullptr, a.wait_ns);
            for (uint32_t s = 0; s < (uint32_t)L::kNK && s < k_loads; ++s) {
                const uint32_t last = k_loads - 1 - ((k_loads - 1 - s) % L::kNK);
                mbar_wait(&bars[P_KF + s], (last / L::kNK) & 1, nullptr, a.wait_ns);
            }
            for (uint32_t s = 0; s < (uint32_t)L::kNV && s < v_loads; ++s) {
                const uint32_t last = v_loads - 1 - ((v_loads - 1 - s) % L::kNV);
                mbar_wait(&bars[P_VF + s], (last / L::kNV) & 1, nullptr, a.wait_ns);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_f16(128, 128, !F16, false, false);
            constexpr uint32_t idesc_pv = idesc_f16(128, 128, !F16, false, true);
            constexpr uint32_t idesc_qk8 = idesc_e4m3(128, 128, false, false);
            const uint32_t qa = smem_u32(sm + L::kQOff);
            // Descriptors are built once: an MMA's operands differ from the first by
            // constant offsets, added to the start-address word (14 bits of 16-byte
            // units; shared memory stays below 256 KB, so it never carries).  The
            // issuing thread shares its SMSP with softmax warps, so every
            // instruction it saves between MMAs keeps the tensor pipe fed.
            const uint64_t qdesc = sdesc_sw128(qa, 16, 1024);
            const uint64_t kdesc = sdesc_sw128(smem_u32(sm + L::kKOff), 16, 1024);
            const uint64_t vdesc = sdesc_sw128(smem_u32(sm + L::kVOff), 16384, 1024);
            const uint32_t q_lo = (uint32_t)qdesc, q_hi = (uint32_t)(qdesc >> 32);
            const uint32_t k_lo = (uint32_t)kdesc, k_hi = (uint32_t)(kdesc >> 32);
            const uint32_t v_lo = (uint32_t)vdesc, v_hi = (uint32_t)(vdesc >> 32);
            auto qk = [&](int x, int kslot) {
                const uint32_t qw = q_lo + (uint32_t)((x * L::kQBytes) >> 4);
                const uint32_t kw = k_lo + (uint32_t)((kslot * L::kKBytes) >> 4);
                const uint32_t dt = tbase + s_col(x);
                if constexpr (F8) {
                    // per-head part on the e4m3 path (32 bytes of depth per MMA), then
                    // the rope part in bf16, hi and lo query levels against the same
                    // k_rope chunk, all into one accumulator
                    mma_f8_ss_w<0>(dt, qw, q_hi, kw, k_hi, idesc_qk8);
#pragma unroll
                    for (int kk = 1; kk < 4; ++kk)
                        mma_f8_ss_w<1>(dt, qw + (uint32_t)(kk * 2), q_hi, kw + (uint32_t)(kk * 2), k_hi, idesc_qk8);
#pragma unroll
                    for (int lvl = 1; lvl <= 2; ++lvl)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss_w<1>(dt, qw + (uint32_t)((lvl * L::kTile + kk * 32) >> 4), q_hi,
                                        kw + (uint32_t)((L::kTile + kk * 32) >> 4), k_hi, idesc_qk);
                } else {
                    mma_ss_w<0>(dt, qw, q_hi, kw, k_hi, idesc_qk);
#pragma unroll
                    for (int kk = 1; kk < L::kDqk / 16; ++kk) {
                        const uint32_t off = (uint32_t)(((kk >> 2) * L::kTile + (kk & 3) * 32) >> 4);
                        mma_ss_w<1>(dt, qw + off, q_hi, kw + off, k_hi, idesc_qk);
                    }
                    if constexpr (R8) {
                        // the query's rope chunk against the rope key's lo level
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss_w<1>(dt, qw + (uint32_t)((2 * L::kTile + kk * 32) >> 4), q_hi,
                                        kw + (uint32_t)((3 * L::kTile + kk * 32) >> 4), k_hi, idesc_qk);
                    }
                }
                mma_commit(&bars[P_SF + x]);
            };
            auto pv = [&](int x, int vslot, bool first) {
                const uint32_t vw = v_lo + (uint32_t)((vslot * L::kVBytes) >> 4);
                const uint32_t dt = tbase + o_col(x), at = tbase + s_col(x);
                if (first) mma_ts_w<0>(dt, at, vw, v_hi, idesc_pv);
                else mma_ts_w<1>(dt, at, vw, v_hi, idesc_pv);
#pragma unroll
                for (int kk = 1; kk < 8; ++kk)  // P of keys 64..127 sits 32 columns further on
                    mma_ts_w<1>(dt, at + kk * 8 + (kk >= 4 ? 32 : 0), vw + (uint32_t)((kk * 2048) >> 4), v_hi, idesc_pv);
                mma_commit(&bars[P_OD + x]);
            };
            bool ok = true;
            uint32_t k = 0, gt = 0, npv[2] = {0u, 0u}, nqs[2] = {0u, 0u};
            for (;;) {
                if (!mbar_wait(&bars[P_IF + (k & 1)], (k >> 1) & 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                const PItem it = item_q[k & 1];
                mbar_arrive(&bars[P_IE + (k & 1)]);
                if (!it.valid) break;
                const bool has_b = it.rA + 128 < it.sg.q_len;
                const int n[2] = {it.nA, it.nB};
                const int nkv = max(n[0], n[1]);
                ok = mbar_wait(&bars[P_QF], k & 1, abort_sh, a.wait_ns);
                if constexpr (F8) {
                    // the softmax threads divide the query's rope part by the head's scale first
                    for (int x = 0; x < 2 && ok; ++x)
                        if (x == 0 || has_b) ok = mbar_wait(&bars[P_QS + x], nqs[x]++ & 1, abort_sh, a.wait_ns);
                }
                if (!ok) break;
                // S for tile 0 of both query tiles
                if (nkv > 0) {
                    ok = mbar_wait(&bars[P_KF + gt % L::kNK], (gt / L::kNK) & 1, abort_sh, a.wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    for (int x = 0; x < 2; ++x)
                        if (n[x] > 0) qk(x, gt % L::kNK);
                    mma_commit(&bars[P_KE + gt % L::kNK]);
                }
                if (nkv <= 1) mma_commit(&bars[P_QE]);  // the item's last QK is issued
                for (int j = 0; j < nkv && ok; ++j) {
                    const uint32_t g = gt + j;
                    const int vs = g % L::kNV;
                    ok = mbar_wait(&bars[P_VF + vs], (g / L::kNV) & 1, abort_sh, a.wait_ns);
                    bool k_waited = false;
                    for (int x = 0; x < 2 && ok; ++x) {
                        if (j >= n[x]) continue;
                        ok = mbar_wait(&bars[P_PF + x], npv[x] & 1, abort_sh, a.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        pv(x, vs, j == 0);
                        ++npv[x];
                        if (j + 1 < n[x]) {
                            // P_x lives in S_x's columns.  MMAs issued by this thread
                            // execute in issue order, so the next S_x written here
                            // cannot overtake PV_x's read of P_x.
                            if (!k_waited) {
                                ok = mbar_wait(&bars[P_KF + (g + 1) % L::kNK], ((g + 1) / L::kNK) & 1, abort_sh,
                                               a.wait_ns);
                                k_waited = true;
                                if (!ok) break;
                                tc_fence_after();
                            }
                            qk(x, (g + 1) % L::kNK);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&bars[P_VE + vs]);
                    if (j + 1 < nkv) mma_commit(&bars[P_KE + (g + 1) % L::kNK]);
                    if (j + 2 == nkv) mma_commit(&bars[P_QE]);  // the item's last QK is issued
                }
                if (!ok) break;
                gt += nkv;
                ++k;
            }
            if (!ok) {
                *abort_sh = 1;
                atomicCAS(a.status, 0, PA_ERR_TIMEOUT);
            }
            mma_commit(&bars[P_DONE]);
            mbar_wait(&bars[P_DONE], 0, nullptr, a.wait_ns);
        }
    } else {
        // ---------------------------------------------------------------- softmax (A: warps 2-5, B: 6-9)
        const int x = warp >= 6 ? 1 : 0;
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;           // query row within the tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        // a compile-time element type: the P conversions in the exponential loop
        // carry no per-pair branch
        constexpr bool f16 = F16;
        bool ok = true;
        uint32_t kit = 0, gt = 0, ns = 0;  // items, K/V tiles before this item, S tiles of this query tile
        for (;;) {
            ok = mbar_wait(&bars[P_IF + (kit & 1)], (kit >> 1) & 1, abort_sh, a.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const PItem it = item_q[kit & 1];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[P_IE + (kit & 1)]);
            if (!it.valid) break;
            const Seg& sg = it.sg;
            const int h = it.h;
            const int i = it.rA + x * 128 + row;  // query row within the segment
            const int nx = x ? it.nB : it.nA;
            const int nkv = max(it.nA, it.nB);
            const bool active = x == 0 || it.rA + 128 < sg.q_len;
            // the query tile that takes the item's last K/V tile first zeroes its dead
            // V rows (they may hold anything, and 0 * NaN would poison the PV product)
            const bool zeroer = active && nkv > 0 && nkv * 128 > sg.kv_len && x == (it.nA == nkv ? 0 : 1);
            float sl2 = a.scale_log2;
            if constexpr (F8) {
                // score = scale * (s * <q_nope, k_nope> + <q_rope, k_rope>), s = q_scale[h] * k_scale[kvh]:
                // the rope part of this thread's query row is divided by s and held as
                // hi + lo bf16 levels (about 16 significant bits) so that both products
                // add in one accumulator, and s joins the softmax scale
                const float s = __ldg(&a.q_scale[h]) * __ldg(&a.k_scale[h / a.group]);
                const float inv = 1.f / s;
                if (!(s > 0.f) || !isfinite(s) || !isfinite(inv)) atomicCAS(a.status, 0, PA_ERR_INVALID_ARG);
                sl2 *= s;
                if (active) {
                    ok = mbar_wait(&bars[P_QF], kit & 1, abort_sh, a.wait_ns);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    // chunk 1 holds the row's 64 bf16 (TMA); chunks 1 and 2 share the
                    // swizzle pattern, so the lo level goes to the same offset in chunk 2
                    uint4* qh = reinterpret_cast<uint4*>(sm + L::kQOff + x * L::kQBytes + L::kTile + row * 128);
                    uint4* ql = qh + L::kTile / 16;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint4 w = qh[u];
                        const uint32_t e[4] = {w.x, w.y, w.z, w.w};
                        uint32_t eh[4], el[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float a0 = __uint_as_float(e[t] << 16) * inv;
                            const float a1 = __uint_as_float(e[t] & 0xFFFF0000u) * inv;
                            eh[t] = pack16x2(a0, a1, false);
                            const float h0 = __uint_as_float(eh[t] << 16), h1 = __uint_as_float(eh[t] & 0xFFFF0000u);
                            el[t] = pack16x2(a0 - h0, a1 - h1, false);
                        }
                        qh[u] = make_uint4(eh[0], eh[1], eh[2], eh[3]);
                        ql[u] = make_uint4(el[0], el[1], el[2], el[3]);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&bars[P_QS + x]);
                }
            }
            // keys this row may see: [0, lim)
            long long lim = sg.kv_len;
            if (a.causal) lim = min(lim, (long long)sg.off + i + 1);
            if (lim < 0) lim = 0;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; active && ok && j < nx; ++j) {
                ok = mbar_wait(&bars[P_SF + x], ns & 1, abort_sh, a.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const int vis = (int)min(128LL, max(0LL, lim - (long long)j * 128));  // visible keys of this tile
                // every key of the tile visible to every row of the warp, positive scale:
                // no per-element masking, and the max can be taken on the raw scores
                const bool full = __all_sync(0xffffffffu, vis >= 128) && sl2 > 0.f;
                // pass 1: row max of the scaled, masked scores (S read from TMEM, 64 columns
                // per wait); the second half stays in registers for pass 2
                float mt;
                uint32_t r[64];
                {
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        tmem_ld_x32(tbase + lane_addr + s_col(x) + hh * 64, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                        tmem_ld_x32(tbase + lane_addr + s_col(x) + hh * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                        tmem_ld_wait();
                        reg_fence(r);
                        if (full) {
#pragma unroll
                            for (int k = 0; k < 64; k += 2)
                                m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], __uint_as_float(r[k]), __uint_as_float(r[k + 1]));
                        } else {
#pragma unroll
                            for (int k = 0; k < 64; ++k)
                                if (hh * 64 + k < vis) m4[k & 3] = fmaxf(m4[k & 3], __uint_as_float(r[k]) * sl2);
                        }
                    }
                    mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    if (full) mt *= sl2;
                }
                // conditional rescale: keep the stale max unless the new one is 2^8 larger
                const bool grow = mt > m_run + kRescaleThreshold;
                float m_new = grow ? mt : m_run;
                const bool need_o = __any_sync(0xffffffffu, grow && j > 0 && m_run != -INFINITY);
                if (need_o) {
                    ok = mbar_wait(&bars[P_OD + x], (ns - 1) & 1, abort_sh, a.wait_ns);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    const float alpha = (grow && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld_x32(tbase + lane_addr + o_col(x) + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st_x32(tbase + lane_addr + o_col(x) + c * 32, o);
                    }
                    tmem_st_wait();
                }
                if (grow) {
                    if (m_run != -INFINITY) l_run *= ex2(m_run - m_new);
                    m_run = m_new;
                }
                const bool none = m_run == -INFINITY;
                const bool fast = __all_sync(0xffffffffu, full && !none);
                const float neg_m = -m_run;
                float rs0 = 0.f, rs1 = 0.f;
                // pass 2: P = exp2(x - m) in 16 bits, written over S columns already read:
                // keys 64..127 first, from the registers, to P columns 64..95, then keys
                // 0..63, read again, to P columns 0..31
#pragma unroll 1
                for (int t = 0; t < 2; ++t) {
                    const int hh = 1 - t;
                    uint32_t pw[32];
                    if (t == 1) {
                        tmem_ld_x32(tbase + lane_addr + s_col(x), *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
                        tmem_ld_x32(tbase + lane_addr + s_col(x) + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
                        tmem_ld_wait();
                        reg_fence(r);
                    }
                    if (fast) {
                        const uint64_t sc2 = f2_pack(__float_as_uint(sl2), __float_as_uint(sl2));
                        const uint64_t nm2 = f2_pack(__float_as_uint(neg_m), __float_as_uint(neg_m));
                        // two running sums, alternate pairs: half the add chain's length
                        uint64_t acc2 = f2_pack(0u, 0u), acc2b = f2_pack(0u, 0u);
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(r[2 * k], r[2 * k + 1]), sc2, nm2), x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            if (k & 1) acc2b = f2_add(acc2b, f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
                            else acc2 = f2_add(acc2, f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
                            pw[k] = pack16x2(p0, p1, f16);
                        }
                        float a0, a1;
                        f2_unpack(f2_add(acc2, acc2b), a0, a1);
                        rs0 += a0;
                        rs1 += a1;
                    } else {
#pragma unroll
                        for (int k = 0; k < 32; ++k) {
                            const int key = hh * 64 + 2 * k;
                            const float p0 = (none || key >= vis) ? 0.f : ex2(__uint_as_float(r[2 * k]) * sl2 - m_run);
                            const float p1 = (none || key + 1 >= vis) ? 0.f : ex2(__uint_as_float(r[2 * k + 1]) * sl2 - m_run);
                            rs0 += p0;
                            rs1 += p1;
                            pw[k] = pack16x2(p0, p1, f16);
                        }
                    }
                    tmem_st_x32(tbase + lane_addr + s_col(x) + hh * 64, pw);
                }
                const float rs = rs0 + rs1;
                l_run += rs;
                if (zeroer && j == nkv - 1) {
                    const uint32_t g = gt + j;
                    const int vs = g % L::kNV;
                    ok = mbar_wait(&bars[P_VF + vs], (g / L::kNV) & 1, abort_sh, a.wait_ns);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (row >= sg.kv_len - j * 128) {  // this thread's row of the V tile is a dead key
                        uint8_t* vr = sm + L::kVOff + vs * L::kVBytes + row * 128;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                *reinterpret_cast<uint4*>(vr + c * L::kTile + u * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&bars[P_PF + x]);
                ++ns;
            }
            // ---- epilogue
            if (active && ok) {
                const bool write = i < sg.q_len;
                const long long orow = ((long long)(sg.q0 + i) * a.num_q_heads + h);
                if (nx > 0) {
                    ok = mbar_wait(&bars[P_OD + x], (ns - 1) & 1, abort_sh, a.wait_ns);
                    ok = __all_sync(0xffffffffu, ok);
                }
                if (ok) {
                    tc_fence_after();
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                    uint16_t* dst = a.out + orow * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        if (nx > 0) {
                            tmem_ld_x32(tbase + lane_addr + o_col(x) + c * 32, o);
                            tmem_ld_wait();
                            reg_fence(o);
                        } else {
#pragma unroll
                            for (int kk = 0; kk < 32; ++kk) o[kk] = 0u;
                        }
                        if (write) {
                            uint32_t w[16];
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk)
                                w[kk] = pack16x2(__uint_as_float(o[2 * kk]) * inv, __uint_as_float(o[2 * kk + 1]) * inv, f16);
                            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                d4[kk] = make_uint4(w[4 * kk], w[4 * kk + 1], w[4 * kk + 2], w[4 * kk + 3]);
                        }
                    }
                    if (write && a.lse)
                        a.lse[orow] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2f : -INFINITY;
                }
            }
            if (!ok) break;
            // the next item's PV into O_x starts from P_x, which this thread
            // writes only after the reads above: no extra barrier
            tc_fence_before();
            gt += nkv;
            ++kit;
        }
        if (!ok) {
            *abort_sh = 1;
            atomicCAS(a.status, 0, PA_ERR_TIMEOUT);
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tbase, 512);
    }
    if (threadIdx.x == 0) {
        // the last CTA to finish leaves the work counters at zero for the next call
        __threadfence();
        if (atomicAdd(ctas_done, 1) == (int)gridDim.x - 1) {
            atomicExch(next_item, 0);
            atomicExch(ctas_done, 0);
        }
    }
}

// Order the (segment, 256-row query block) units sequence by sequence, the
// longest key range first, and within a sequence its last query block first
// (the most KV tiles under causal masking).  CTAs that run together then work
// on one sequence (across a group of heads), so its K/V tiles are shared in L2,
// and the costliest work still starts first.  One CTA; bitonic sort of up to
// 4096 64-bit keys in shared memory:
//   [63:40] 0xFFFFFF - kv_len   [39:20] b   [19:0] 0xFFFFF - query block
// with kv_len forced to 0 for idle units (their rows lie past q_len).
__global__ void __launch_bounds__(512) prefill_order_kernel(const PrefillArgs a, int32_t* order) {
    // the prefill kernel may be scheduled now: it runs its barrier set-up and
    // then waits for this kernel's completion before reading the order
    allow_dependents_launch();
    __shared__ unsigned long long key[4096];
    const int n = a.batch * a.num_q_tiles;
    int p2 = 1;
    while (p2 < n) p2 <<= 1;
    for (int u = threadIdx.x; u < p2; u += blockDim.x) {
        unsigned long long k = ~0ull;
        if (u < n) {
            const int b = u % a.batch, pair = u / a.batch;
            const Seg sg = load_seg(a, b);
            const long long kv = pair * a.q_block < sg.q_len ? min(max(sg.kv_len, 0), 0xFFFFFF - 1) : -1;
            k = ((unsigned long long)(0xFFFFFF - 1 - kv) << 40) | ((unsigned long long)b << 20) |
                (unsigned long long)(0xFFFFF - pair);
        }
        key[u] = k;
    }
    __syncthreads();
    for (int size = 2; size <= p2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = threadIdx.x; t < p2 / 2; t += blockDim.x) {
                const int lo = 2 * stride * (t / stride) + (t % stride);
                const int hi = lo + stride;
                const bool up = (lo & size) == 0;
                const unsigned long long x = key[lo], y = key[hi];
                if ((x > y) == up) {
                    key[lo] = y;
                    key[hi] = x;
                }
            }
            __syncthreads();
        }
    }
    for (int u = threadIdx.x; u < n; u += blockDim.x) {
        const unsigned long long kk = key[u];
        const int b = (int)((kk >> 20) & 0xFFFFF), pair = 0xFFFFF - (int)(kk & 0xFFFFF);
        order[u] = pair * a.batch + b;
    }
}

template <bool ROPE, bool PAGED, bool F8, bool R8 = false, bool F16 = false>
cudaError_t launch_t(const PrefillArgs& a, const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                     const CUtensorMap* mr, const CUtensorMap* mqr, cudaStream_t stream) {
    using L = PrefillLayout<ROPE, F8, R8>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = ensure_dynamic_smem(prefill_kernel<ROPE, PAGED, F8, R8, F16>, L::kSmem, configured);
    if (e != cudaSuccess) return e;
    if (a.order) {
        prefill_order_kernel<<<1, 512, 0, stream>>>(a, const_cast<int32_t*>(a.order));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // persistent: one CTA per SM, or one per work item when there are fewer
    const long long items = (long long)a.num_q_tiles * a.batch * a.num_q_heads;
    if (items <= 0) return cudaSuccess;
    if (items > 0x7FFFFFFFLL - 65536) return cudaErrorInvalidValue;  // the work counter is an int32
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(items < sms ? items : sms);
    return launch_overlapped(prefill_kernel<ROPE, PAGED, F8, R8, F16>, dim3(grid), dim3(L::kThreads), L::kSmem, stream,
                             a, *mq, *mk, *mv, *mr, *mqr);
}

// The e4m3 rope key times its token's scale as two bf16 levels, hi = bf16(x)
// and lo = bf16(x - hi): about 16 significant bits together, against the 4 of
// the code and the 24 of the scale (x itself is their fp32 product).  One
// thread per 8 codes; a token's 64 codes are 8 such groups.
__global__ void __launch_bounds__(256) rope_expand_kernel(const uint8_t* __restrict__ codes,
                                                          const float* __restrict__ scales,
                                                          uint16_t* __restrict__ hi, uint16_t* __restrict__ lo,
                                                          int64_t groups) {
    const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= groups) return;
    const float s = __ldg(&scales[gi >> 3]);
    const uint2 c = __ldg(reinterpret_cast<const uint2*>(codes) + gi);
    const uint32_t w[2] = {c.x, c.y};
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // codes 2i, 2i + 1
        const __half2_raw hr =
            __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)((w[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu), __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
        const float x0 = f.x * s, x1 = f.y * s;
        const uint32_t hb = pack16x2(x0, x1, false);
        float h0, h1;
        unpack16x2(hb, false, h0, h1);
        h[i] = hb;
        l[i] = pack16x2(x0 - h0, x1 - h1, false);
    }
    reinterpret_cast<uint4*>(hi)[gi] = make_uint4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<uint4*>(lo)[gi] = make_uint4(l[0], l[1], l[2], l[3]);
}

}  // namespace

cudaError_t launch_prefill_order(const PrefillArgs& a, cudaStream_t stream) {
    if (!a.order) return cudaSuccess;
    prefill_order_kernel<<<1, 512, 0, stream>>>(a, const_cast<int32_t*>(a.order));
    return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim_qk, const CUtensorMap* mq, const CUtensorMap* mk,
                           const CUtensorMap* mv, const CUtensorMap* mr, const CUtensorMap* mqr,
                           cudaStream_t stream) {
    if (a.f8) return launch_t<true, false, true>(a, mq, mk, mv, mr, mqr, stream);
    if (a.r8) return launch_t<true, false, false, true>(a, mq, mk, mv, mr, mqr, stream);
    if (head_dim_qk == 192)
        return a.f16 ? launch_t<true, false, false, false, true>(a, mq, mk, mv, mr, mqr, stream)
                     : launch_t<true, false, false, false, false>(a, mq, mk, mv, mr, mqr, stream);
    if (a.paged)
        return a.f16 ? launch_t<false, true, false, false, true>(a, mq, mk, mv, mr, mqr, stream)
                     : launch_t<false, true, false, false, false>(a, mq, mk, mv, mr, mqr, stream);
    return a.f16 ? launch_t<false, false, false, false, true>(a, mq, mk, mv, mr, mqr, stream)
                 : launch_t<false, false, false, false, false>(a, mq, mk, mv, mr, mqr, stream);
}

cudaError_t launch_rope_expand(const uint8_t* codes, const float* scales, uint16_t* hi, uint16_t* lo,
                               int64_t tokens, cudaStream_t stream) {
    const int64_t groups = tokens * 8;
    if (groups <= 0) return cudaSuccess;
    const int64_t blocks = (groups + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    rope_expand_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, hi, lo, groups);
    return cudaGetLastError();
}

}  // namespace pa
