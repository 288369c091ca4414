// prefill_pair.cu -- causal (or full) attention for ragged query segments with
// every tensor-core product shared by a pair of CTAs (tcgen05 cta_group::2,
// M = 256): chunked prefill against the paged cache (FlashMLA "Tensor Shapes
// Reference", section 4 mha_fwd_kvcache: K/V gathered through block_table),
// ragged prefill (MATE dense mode, flash_attn_varlen_func) and the MLA shape
// whose 64-wide rope key is shared by all heads (Modular flare_mla_prefill:
// q depth 192 = 128 per-head + 64 shared, output depth 128); bf16 or fp16.
//
// Why a pair: one CTA's M = 128 MMAs with both operands in shared memory need
// 8 KB of operand reads per 64-cycle instruction, the whole of the SM's
// shared-memory bandwidth, before the TMA writes of the K/V tiles.  Over a
// pair each CTA reads its own 128 query rows but only half of every K or V
// tile, and loads only that half from memory, so each SM moves about 40% fewer
// shared-memory bytes per FLOP.
//
// Work item: (segment b, 512-row query block, query head h), two MMA tiles A
// (rows 0-255) and B (rows 256-511).  CTA rank r of the pair holds rows
// r*128 .. r*128+127 of each: its own S and O accumulators in TMEM (S_A, S_B,
// O_A, O_B, 128 columns each), its own query rows in shared memory, keys
// r*64 .. r*64+63 of each 128-key K tile and columns r*64 .. r*64+63 of each
// V tile.  Persistent: each pair takes items from a counter until none is left.
//
//   warp 0     producer (both CTAs): rank 0 takes the items and publishes them
//              to both CTAs; each CTA loads its halves of the query, K and V
//              tiles by TMA, every copy completing on rank 0's barriers
//   warp 1     rank 0: MMA issuer (one thread) for the pair --
//                S_X[256 q, 128 keys] = Q_X . K^T        (both from smem)
//                O_X[256 q, 128 dv]  += P_X . V          (P_X from TMEM)
//              in the one-CTA kernel's order (QK_A(j+1) right after PV_A(j));
//              rank 1: idle after the TMEM allocation
//   warps 2-5  softmax of tile A, warps 6-9 of tile B, in both CTAs: one
//              query row per thread (its TMEM lane), S read in 32-column
//              chunks with the next chunk's load in flight; P (16-bit) over
//              the S columns; O rescaled in TMEM only when the running max
//              grows by more than 2^8.  Rank 0's warps of the tile that takes
//              an item's last K/V tile zero that tile's dead V rows in both
//              CTAs.
//
// Query row i of segment b sees key j iff j < kv_len and (not causal or
// j <= qo_offset + i), qo_offset defaulting to kv_len - q_len (MATE
// _normalize_qo_offset / _resolve_seqused_k).  Every wait is bounded; the
// only unbounded barriers are the two cluster-wide ones every thread reaches.
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "prefill_common.cuh"

namespace pa {
namespace {

constexpr int kMaxStages = 4;
// consumers of an item slot: rank 0's MMA thread and 8 softmax warps, rank 1's
// producer and 8 softmax warps
constexpr int kItemReaders = 18;

enum : int {
    B_QF = 0,                      // rank 0: the item's query tiles of both CTAs landed
    B_QE = 1,                      // both: query buffers free again (the item's last QK retired)
    B_SF = 2,                      // [2] both: S_A / S_B ready
    B_PF = 4,                      // [2] rank 0: P_A / P_B written in both CTAs (one arrival per warp)
    B_OD = 6,                      // [2] both: an item's last PV_A / PV_B retired
    B_IF = 8,                      // [2] both: item slot published
    B_IE = 10,                     // [2] rank 0: item slot read by every consumer
    B_DONE = 12,                   // rank 0: every MMA retired
    B_KF = 13,                     // [kMaxStages] rank 0: K tile landed in both CTAs
    B_VF = B_KF + kMaxStages,      // [kMaxStages] rank 0: V tile landed in both CTAs
    B_SE = B_VF + kMaxStages,      // [kMaxStages] both: ring stage (K and V tile) free
    B_COUNT = B_SE + kMaxStages
};

template <bool ROPE>
struct PairLayout {
    static constexpr int kDqk = ROPE ? 192 : 128;
    static constexpr int kChunks = kDqk / 64;          // 64-element (128-byte) chunks of a q or k row
    static constexpr int kQTile = 16384;               // 128 query rows x 128 bytes
    static constexpr int kKTile = 8192;                // 64 keys x 128 bytes
    static constexpr int kQBytes = kChunks * kQTile;   // this CTA's rows of one query tile
    static constexpr int kKBytes = kChunks * kKTile;   // this CTA's 64 keys of a 128-key K tile
    static constexpr int kVBytes = 16384;              // this CTA's 64 columns of a 128-key V tile
    static constexpr int kNS = ROPE ? 3 : 4;  // ring stages, each one K tile and one V tile
    static constexpr int kQOff = 0;
    static constexpr int kKOff = 2 * kQBytes;
    static constexpr int kVOff = kKOff + kNS * kKBytes;
    static constexpr int kBytes = kVOff + kNS * kVBytes;
    static constexpr int kSmem = kBytes + 1024;
    static constexpr int kThreads = 320;  // producer, MMA issuer, 8 softmax warps
    static_assert(kNS <= kMaxStages, "ring depth");
    static_assert(kSmem + 1024 <= 232448, "shared memory per CTA (dynamic + static)");
};

template <bool ROPE, bool PAGED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(320, 1)
    prefill_pair_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_r) {
    static_assert(!(ROPE && PAGED), "the shared rope key is defined for ragged keys");
    using L = PairLayout<ROPE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[B_COUNT];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_store;
    __shared__ int item_w[2];
    volatile int* abort_sh = &abort_store;

    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = a.num_q_tiles * a.batch * a.num_q_heads;  // work items
    int* next_item = a.status + kPrefillNextWord;
    int* ctas_done = a.status + kPrefillDoneWord;
    // shared::cluster address of barrier i in rank 0, and of a variable in rank 1
    auto lead = [&](int i) { return mapa_shared(smem_u32(&bars[i]), 0); };
    auto peer1 = [&](const void* p) { return mapa_shared(smem_u32(p), 1); };

    if (threadIdx.x == 0) {
        mbar_init(&bars[B_QF], 2);
        mbar_init(&bars[B_QE], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[B_SF + i], 1);
            mbar_init(&bars[B_PF + i], 8);
            mbar_init(&bars[B_OD + i], 1);
            mbar_init(&bars[B_IF + i], 1);
            mbar_init(&bars[B_IE + i], kItemReaders);
        }
        mbar_init(&bars[B_DONE], 1);
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&bars[B_KF + s], 2);
            mbar_init(&bars[B_VF + s], 2);
            mbar_init(&bars[B_SE + s], 1);
        }
        *abort_sh = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&tmem_base_sh, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;
    // TMEM columns: S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512)
    auto s_col = [](int x) { return (uint32_t)(x * 128); };
    auto o_col = [](int x) { return (uint32_t)(256 + x * 128); };

    if (warp == 0) {
        // ---------------------------------------------------------------- producer (both CTAs)
        if (lane == 0) {
            bool ok = true;
            uint32_t k = 0;   // items taken
            uint32_t gt = 0;  // K/V tiles of the items before this one
            uint32_t q_loads = 0, k_loads = 0, v_loads = 0;
            for (;;) {
                int w = -1;
                if (leader) {
                    PItem probe;
                    for (;;) {  // the next item that has rows
                        const int cand = atomicAdd(next_item, 1);
                        if (cand >= W) break;
                        if (make_item(a, cand, probe)) {
                            w = cand;
                            break;
                        }
                    }
                    // slot k & 1 is free once every consumer of both CTAs has read item k - 2
                    if (!mbar_wait_cl(&bars[B_IE + (k & 1)], ((k >> 1) & 1) ^ 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    item_w[k & 1] = w;
                    st_cl_u32(peer1(&item_w[k & 1]), (uint32_t)w);
                    mbar_arrive_cl(lead(B_IF + (k & 1)));
                    mbar_arrive_cl(peer1(&bars[B_IF + (k & 1)]));
                } else {
                    if (!mbar_wait_cl(&bars[B_IF + (k & 1)], (k >> 1) & 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    w = item_w[k & 1];
                    mbar_signal_cl(lead(B_IE + (k & 1)));
                }
                if (w < 0) break;
                PItem it;
                make_item(a, w, it);
                const Seg& sg = it.sg;
                const int h = it.h, kvh = h / a.group;
                const int n[2] = {it.nA, it.nB};
                const int nkv = max(n[0], n[1]);
                // this CTA's query rows of tiles A and B, loaded when the tile runs and has rows here
                bool qload[2];
                uint32_t qbytes = 0;
                for (int x = 0; x < 2; ++x) {
                    qload[x] = n[x] > 0 && it.rA + x * 256 + (int)rank * 128 < sg.q_len;
                    qbytes += qload[x] ? L::kQBytes : 0;
                }
                if (k > 0 && !mbar_wait(&bars[B_QE], (k - 1) & 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx_cl(lead(B_QF), qbytes);
                for (int x = 0; x < 2; ++x)
                    if (qload[x])
                        for (int c = 0; c < L::kChunks; ++c)
                            tma_load_3d_pair(sm + L::kQOff + x * L::kQBytes + c * L::kQTile, &map_q, lead(B_QF),
                                             c * 64, h, sg.q0 + it.rA + x * 256 + (int)rank * 128);
                q_loads = k + 1;
                const int kv_pages = (sg.kv_len + kPage - 1) / kPage;
                for (int j = 0; j < nkv && ok; ++j) {
                    const uint32_t g = gt + j;
                    int pid[2] = {-1, -1};  // page ids of this tile (paged keys)
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
                    // the ring stage is free once both tiles' PV of the tile that last used it retired
                    const int ks = g % L::kNS;
                    if (!mbar_wait(&bars[B_SE + ks], ((g / L::kNS) & 1) ^ 1, abort_sh, a.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // K: this CTA's 64 keys of the tile
                    uint8_t* kt = sm + L::kKOff + ks * L::kKBytes;
                    const uint32_t kf = lead(B_KF + ks);
                    if (PAGED) {
                        const int p = pid[rank];
                        mbar_arrive_expect_tx_cl(kf, p >= 0 ? (uint32_t)L::kKBytes : 0u);
                        if (p >= 0)
                            for (int c = 0; c < L::kChunks; ++c)
                                tma_load_2d_pair(kt + c * L::kKTile, &map_k, kf, c * 64,
                                                 (int)(((long long)p * a.num_kv_heads + kvh) * 64));
                    } else {
                        const int row = sg.k0 + j * 128 + (int)rank * 64;
                        mbar_arrive_expect_tx_cl(kf, L::kKBytes);
                        for (int c = 0; c < 2; ++c) tma_load_3d_pair(kt + c * L::kKTile, &map_k, kf, c * 64, kvh, row);
                        if (ROPE) tma_load_2d_pair(kt + 2 * L::kKTile, &map_r, kf, 0, row);
                    }
                    k_loads = g + 1;
                    // V: this CTA's 64 columns of the tile's 128 keys
                    const int vs = ks;
                    uint8_t* vt = sm + L::kVOff + vs * L::kVBytes;
                    const uint32_t vf = lead(B_VF + vs);
                    if (PAGED) {
                        const uint32_t npid = (pid[0] >= 0) + (pid[1] >= 0);
                        mbar_arrive_expect_tx_cl(vf, npid * 8192u);
                        for (int i = 0; i < 2; ++i)
                            if (pid[i] >= 0)
                                tma_load_2d_pair(vt + i * 8192, &map_v, vf, (int)rank * 64,
                                                 (int)(((long long)pid[i] * a.num_kv_heads + kvh) * 64));
                    } else {
                        mbar_arrive_expect_tx_cl(vf, L::kVBytes);
                        tma_load_3d_pair(vt, &map_v, vf, (int)rank * 64, kvh, sg.k0 + j * 128);
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
            // every issued copy must land before the pair may exit; the full
            // barriers (rank 0) count both CTAs' copies.  With n tiles issued,
            // ring slot s last took tile n - 1 - ((n - 1 - s) mod slots).
            if (leader) {
                if (q_loads > 0) mbar_wait(&bars[B_QF], (q_loads - 1) & 1, nullptr, a.wait_ns);
                for (uint32_t s = 0; s < (uint32_t)L::kNS && s < k_loads; ++s) {
                    const uint32_t last = k_loads - 1 - ((k_loads - 1 - s) % L::kNS);
                    mbar_wait(&bars[B_KF + s], (last / L::kNS) & 1, nullptr, a.wait_ns);
                }
                for (uint32_t s = 0; s < (uint32_t)L::kNS && s < v_loads; ++s) {
                    const uint32_t last = v_loads - 1 - ((v_loads - 1 - s) % L::kNS);
                    mbar_wait(&bars[B_VF + s], (last / L::kNS) & 1, nullptr, a.wait_ns);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer (rank 0)
        if (leader && lane == 0) {
            const uint32_t idesc_qk = idesc_f16(256, 128, !a.f16, false, false);
            const uint32_t idesc_pv = idesc_f16(256, 128, !a.f16, false, true);
            const uint32_t qa = smem_u32(sm + L::kQOff);
            // Descriptors are built once: an MMA's operands differ from the first by
            // constant offsets, added to the start-address word (14 bits of 16-byte
            // units; shared memory stays below 256 KB, so it never carries).
            const uint64_t qdesc = sdesc_sw128(qa, 16, 1024);
            const uint64_t kdesc = sdesc_sw128(smem_u32(sm + L::kKOff), 16, 1024);
            const uint64_t vdesc = sdesc_sw128(smem_u32(sm + L::kVOff), 8192, 1024);
            const uint32_t q_lo = (uint32_t)qdesc, q_hi = (uint32_t)(qdesc >> 32);
            const uint32_t k_lo = (uint32_t)kdesc, k_hi = (uint32_t)(kdesc >> 32);
            const uint32_t v_lo = (uint32_t)vdesc, v_hi = (uint32_t)(vdesc >> 32);
            auto qk = [&](int x, int kslot) {
                const uint32_t qw = q_lo + (uint32_t)((x * L::kQBytes) >> 4);
                const uint32_t kw = k_lo + (uint32_t)((kslot * L::kKBytes) >> 4);
                const uint32_t dt = tbase + s_col(x);
                mma_pair_ss_w<0>(dt, qw, q_hi, kw, k_hi, idesc_qk);
#pragma unroll
                for (int kk = 1; kk < L::kDqk / 16; ++kk)
                    mma_pair_ss_w<1>(dt, qw + (uint32_t)(((kk >> 2) * L::kQTile + (kk & 3) * 32) >> 4), q_hi,
                                     kw + (uint32_t)(((kk >> 2) * L::kKTile + (kk & 3) * 32) >> 4), k_hi, idesc_qk);
                mma_commit_pair_mc(&bars[B_SF + x], 3);
            };
            // O_x is read by the softmax only after the item's last PV_x (the epilogue,
            // which waits on O_D) and, for a rescale, after S_x of the next tile has
            // landed -- whose commit follows PV_x of this tile in issue order.  Keys
            // 16kk..16kk+15: P at TMEM columns 8kk..8kk+7 of S_x.
            auto pv = [&](int x, int vslot, bool first, bool last) {
                const uint32_t vw = v_lo + (uint32_t)((vslot * L::kVBytes) >> 4);
                const uint32_t dt = tbase + o_col(x), at = tbase + s_col(x);
                if (first) mma_pair_ts_w<0>(dt, at, vw, v_hi, idesc_pv);
                else mma_pair_ts_w<1>(dt, at, vw, v_hi, idesc_pv);
#pragma unroll
                for (int kk = 1; kk < 8; ++kk)
                    mma_pair_ts_w<1>(dt, at + kk * 8, vw + (uint32_t)((kk * 2048) >> 4), v_hi, idesc_pv);
                if (last) mma_commit_pair_mc(&bars[B_OD + x], 3);
            };
            bool ok = true;
            uint32_t k = 0, gt = 0, npv[2] = {0u, 0u};
            for (;;) {
                if (!mbar_wait_cl(&bars[B_IF + (k & 1)], (k >> 1) & 1, abort_sh, a.wait_ns)) {
                    ok = false;
                    break;
                }
                const int w = item_w[k & 1];
                mbar_signal_cl(lead(B_IE + (k & 1)));
                if (w < 0) break;
                PItem it;
                make_item(a, w, it);
                const int n[2] = {it.nA, it.nB};
                const int nkv = max(n[0], n[1]);
                ok = mbar_wait(&bars[B_QF], k & 1, abort_sh, a.wait_ns);
                if (!ok) break;
                // S for tile 0 of both query tiles
                if (nkv > 0) {
                    ok = mbar_wait(&bars[B_KF + gt % L::kNS], (gt / L::kNS) & 1, abort_sh, a.wait_ns);
                    if (!ok) break;
                    tc_fence_after();
                    for (int x = 0; x < 2; ++x)
                        if (n[x] > 0) qk(x, gt % L::kNS);
                }
                if (nkv <= 1) mma_commit_pair_mc(&bars[B_QE], 3);  // the item's last QK is issued
                for (int j = 0; j < nkv && ok; ++j) {
                    const uint32_t g = gt + j;
                    const int vs = g % L::kNS;
                    ok = mbar_wait(&bars[B_VF + vs], (g / L::kNS) & 1, abort_sh, a.wait_ns);
                    bool k_waited = false;
                    for (int x = 0; x < 2 && ok; ++x) {
                        if (j >= n[x]) continue;
                        ok = mbar_wait(&bars[B_PF + x], npv[x] & 1, abort_sh, a.wait_ns);
                        if (!ok) break;
                        tc_fence_after();
                        pv(x, vs, j == 0, j + 1 == n[x]);
                        ++npv[x];
                        if (j + 1 < n[x]) {
                            // P_x lives in S_x's columns; MMAs issued by this thread
                            // execute in order, so the next S_x cannot overtake PV_x
                            if (!k_waited) {
                                ok = mbar_wait(&bars[B_KF + (g + 1) % L::kNS], ((g + 1) / L::kNS) & 1, abort_sh, a.wait_ns);
                                k_waited = true;
                                if (!ok) break;
                                tc_fence_after();
                            }
                            qk(x, (g + 1) % L::kNS);
                        }
                    }
                    if (!ok) break;
                    // stage vs (K tile g, used by QK one step back, and V tile g) is consumed
                    mma_commit_pair_mc(&bars[B_SE + vs], 3);
                    if (j + 2 == nkv) mma_commit_pair_mc(&bars[B_QE], 3);  // the item's last QK is issued
                }
                if (!ok) break;
                gt += nkv;
                ++k;
            }
            if (!ok) {
                *abort_sh = 1;
                atomicCAS(a.status, 0, PA_ERR_TIMEOUT);
            }
            mma_commit_pair_mc(&bars[B_DONE], 1);
            mbar_wait(&bars[B_DONE], 0, nullptr, a.wait_ns);
        }
    } else {
        // ---------------------------------------------------------------- softmax (A: warps 2-5, B: 6-9)
        // One query row per thread (its TMEM lane).  S is read in 32-column
        // chunks with the next chunk's load in flight while the current chunk
        // is reduced (pass 1: the row max) or exponentiated (pass 2: P, 16-bit,
        // written over S columns already read: keys 32c..32c+31 -> P columns
        // 16c..16c+15), so the load latency is paid once per pass.
        const int x = warp >= 6 ? 1 : 0;
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;  // query row within this CTA's half of the tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        const uint32_t s_addr = tbase + lane_addr + s_col(x);
        const uint32_t o_addr = tbase + lane_addr + o_col(x);
        const bool f16 = a.f16 != 0;
        bool ok = true;
        uint32_t kit = 0, gt = 0, ns = 0;  // items, K/V tiles before this item, S tiles of this query tile
        uint32_t nod = 0;                   // items whose tile x ran (phases of O_D[x])
        for (;;) {
            ok = mbar_wait_cl(&bars[B_IF + (kit & 1)], (kit >> 1) & 1, abort_sh, a.wait_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const int w = item_w[kit & 1];
            __syncwarp();
            if (lane == 0) mbar_signal_cl(lead(B_IE + (kit & 1)));
            if (w < 0) break;
            PItem it;
            make_item(a, w, it);
            const Seg& sg = it.sg;
            const int h = it.h;
            const int r0 = it.rA + x * 256 + (int)rank * 128;  // this CTA's first row of the tile
            const int i = r0 + row;                            // query row within the segment
            const int nx = x ? it.nB : it.nA;
            const int nkv = max(it.nA, it.nB);
            const bool mine = nx > 0 && r0 < sg.q_len;  // this CTA's half of the tile has rows
            // rank 0's warps of the tile that takes the item's last K/V tile first zero
            // that tile's dead V rows in both CTAs (0 * NaN would poison the PV product)
            const bool zeroer = leader && nx > 0 && nkv * 128 > sg.kv_len && x == (it.nA == nkv ? 0 : 1);
            const float sl2 = a.scale_log2;
            long long lim = sg.kv_len;  // keys this row may see: [0, lim)
            if (a.causal) lim = min(lim, (long long)sg.off + i + 1);
            if (lim < 0) lim = 0;
            float m_run = -INFINITY, l_run = 0.f;
            for (int j = 0; ok && j < nx; ++j) {
                ok = mbar_wait(&bars[B_SF + x], ns & 1, abort_sh, a.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                if (mine) {
                    const int vis = (int)min(128LL, max(0LL, lim - (long long)j * 128));  // visible keys of this tile
                    // every key of the tile visible to every row of the warp, positive scale:
                    // no per-element masking, and the max can be taken on the raw scores
                    const bool full = __all_sync(0xffffffffu, vis >= 128) && sl2 > 0.f;
                    // pass 1: row max of the scaled, masked scores
                    float mt;
                    {
                        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                        uint32_t ra[32], rb[32];
                        auto reduce = [&](const uint32_t (&r)[32], int c) {
                            if (full) {
#pragma unroll
                                for (int kk = 0; kk < 32; kk += 2)
                                    m4[(kk >> 1) & 3] =
                                        fmax3(m4[(kk >> 1) & 3], __uint_as_float(r[kk]), __uint_as_float(r[kk + 1]));
                            } else {
#pragma unroll
                                for (int kk = 0; kk < 32; ++kk)
                                    if (c * 32 + kk < vis) m4[kk & 3] = fmaxf(m4[kk & 3], __uint_as_float(r[kk]) * sl2);
                            }
                        };
                        tmem_ld_x32(s_addr, ra);
                        tmem_ld_wait();
                        reg_fence(ra);
                        tmem_ld_x32(s_addr + 32, rb);
                        reduce(ra, 0);
                        tmem_ld_wait();
                        reg_fence(rb);
                        tmem_ld_x32(s_addr + 64, ra);
                        reduce(rb, 1);
                        tmem_ld_wait();
                        reg_fence(ra);
                        tmem_ld_x32(s_addr + 96, rb);
                        reduce(ra, 2);
                        tmem_ld_wait();
                        reg_fence(rb);
                        reduce(rb, 3);
                        mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                        if (full) mt *= sl2;
                    }
                    // conditional rescale: keep the stale max unless the new one is 2^8 larger
                    const bool grow = mt > m_run + kRescaleThreshold;
                    const float m_new = grow ? mt : m_run;
                    if (__any_sync(0xffffffffu, grow && j > 0 && m_run != -INFINITY)) {
                        // PV_x of the previous tile retired before this S_x landed (one commit covers both)
                        const float alpha = (grow && m_run != -INFINITY) ? ex2(m_run - m_new) : 1.f;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[32];
                            tmem_ld_x32(o_addr + c * 32, o);
                            tmem_ld_wait();
                            reg_fence(o);
#pragma unroll
                            for (int kk = 0; kk < 32; ++kk) o[kk] = __float_as_uint(__uint_as_float(o[kk]) * alpha);
                            tmem_st_x32(o_addr + c * 32, o);
                        }
                    }
                    if (grow) {
                        if (m_run != -INFINITY) l_run *= ex2(m_run - m_new);
                        m_run = m_new;
                    }
                    const bool none = m_run == -INFINITY;
                    const bool fast = __all_sync(0xffffffffu, full && !none);
                    const float neg_m = -m_run;
                    // pass 2: P = exp2(x - m); two packed partial sums keep the adds off one chain
                    uint64_t acc[2] = {f2_pack(0u, 0u), f2_pack(0u, 0u)};
                    float rsm = 0.f;
                    {
                        uint32_t ra[32], rb[32];
                        auto expo = [&](const uint32_t (&r)[32], int c) {
                            uint32_t pw[16];
                            if (fast) {
                                const uint64_t sc2 = f2_pack(__float_as_uint(sl2), __float_as_uint(sl2));
                                const uint64_t nm2 = f2_pack(__float_as_uint(neg_m), __float_as_uint(neg_m));
#pragma unroll
                                for (int kk = 0; kk < 16; ++kk) {
                                    float x0, x1;
                                    f2_unpack(f2_fma(f2_pack(r[2 * kk], r[2 * kk + 1]), sc2, nm2), x0, x1);
                                    const float p0 = ex2(x0), p1 = ex2(x1);
                                    acc[kk & 1] = f2_add(acc[kk & 1], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
                                    pw[kk] = pack16x2(p0, p1, f16);
                                }
                            } else {
#pragma unroll
                                for (int kk = 0; kk < 16; ++kk) {
                                    const int key = c * 32 + 2 * kk;
                                    const float p0 =
                                        (none || key >= vis) ? 0.f : ex2(__uint_as_float(r[2 * kk]) * sl2 - m_run);
                                    const float p1 =
                                        (none || key + 1 >= vis) ? 0.f : ex2(__uint_as_float(r[2 * kk + 1]) * sl2 - m_run);
                                    rsm += p0 + p1;
                                    pw[kk] = pack16x2(p0, p1, f16);
                                }
                            }
                            tmem_st_x16(s_addr + c * 16, pw);
                        };
                        tmem_ld_x32(s_addr, ra);
                        tmem_ld_wait();
                        reg_fence(ra);
                        tmem_ld_x32(s_addr + 32, rb);
                        expo(ra, 0);
                        tmem_ld_wait();
                        reg_fence(rb);
                        tmem_ld_x32(s_addr + 64, ra);
                        expo(rb, 1);
                        tmem_ld_wait();
                        reg_fence(ra);
                        tmem_ld_x32(s_addr + 96, rb);
                        expo(ra, 2);
                        tmem_ld_wait();
                        reg_fence(rb);
                        expo(rb, 3);
                    }
                    float a0, a1, b0, b1;
                    f2_unpack(acc[0], a0, a1);
                    f2_unpack(acc[1], b0, b1);
                    l_run += (a0 + a1) + (b0 + b1) + rsm;
                }
                if (zeroer && j == nkv - 1) {
                    // the V tile's halves of both CTAs landed once rank 0's full barrier completed
                    const uint32_t g = gt + j;
                    const int vs = g % L::kNS;
                    ok = mbar_wait(&bars[B_VF + vs], (g / L::kNS) & 1, abort_sh, a.wait_ns);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    if (row >= sg.kv_len - j * 128) {  // this thread's row of the V tile is a dead key
                        uint8_t* vr = sm + L::kVOff + vs * L::kVBytes + row * 128;
                        const uint32_t vr1 = peer1(vr);
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            *reinterpret_cast<uint4*>(vr + u * 16) = make_uint4(0, 0, 0, 0);
                            st_cl_v4(vr1 + u * 16, make_uint4(0, 0, 0, 0));
                        }
                    }
                    fence_proxy_async_cluster();
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                // a warp that wrote the peer's V rows releases them at cluster scope
                if (lane == 0) {
                    if (zeroer && j == nkv - 1) mbar_arrive_cl(lead(B_PF + x));
                    else mbar_signal_cl(lead(B_PF + x));
                }
                ++ns;
            }
            // ---- epilogue
            if (ok && mine) {
                const bool write = i < sg.q_len;
                const long long orow = ((long long)(sg.q0 + i) * a.num_q_heads + h);
                ok = mbar_wait(&bars[B_OD + x], nod & 1, abort_sh, a.wait_ns);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                    uint16_t* dst = a.out + orow * 128;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld_x32(o_addr + c * 32, o);
                        tmem_ld_wait();
                        reg_fence(o);
                        if (write) {
                            uint32_t wv[16];
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk)
                                wv[kk] = pack16x2(__uint_as_float(o[2 * kk]) * inv, __uint_as_float(o[2 * kk + 1]) * inv,
                                                  f16);
                            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                d4[kk] = make_uint4(wv[4 * kk], wv[4 * kk + 1], wv[4 * kk + 2], wv[4 * kk + 3]);
                        }
                    }
                    if (write && a.lse) a.lse[orow] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2f : -INFINITY;
                }
            } else if (ok && nx == 0 && r0 < sg.q_len) {
                // rows with no visible key: out = 0, lse = -inf
                if (i < sg.q_len) {
                    const long long orow = ((long long)(sg.q0 + i) * a.num_q_heads + h);
                    uint4* d4 = reinterpret_cast<uint4*>(a.out + orow * 128);
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk) d4[kk] = make_uint4(0, 0, 0, 0);
                    if (a.lse) a.lse[orow] = -INFINITY;
                }
            }
            if (nx > 0) ++nod;
            if (!ok) break;
            // the next item's PV into O_x starts from P_x, which this warp
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
    cluster_sync_all();  // the pair's MMAs, copies and peer accesses are over
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tbase, 512);
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

// Clusters of two CTAs of this kernel that fit on the device at once (per device, cached).
template <typename K>
int pair_capacity(K* kernel, int smem) {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_acquire);
        if (c > 0) return c;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(320);
    cfg.dynamicSmemBytes = (size_t)smem;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < 64 && clusters > 0) cached[dev].store(clusters, std::memory_order_release);
    return clusters;
}

template <bool ROPE, bool PAGED>
cudaError_t launch_pair_t(const PrefillArgs& a, const CUtensorMap* mq, const CUtensorMap* mk, const CUtensorMap* mv,
                          const CUtensorMap* mr, cudaStream_t stream) {
    using L = PairLayout<ROPE>;
    auto kernel = prefill_pair_kernel<ROPE, PAGED>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t e = ensure_dynamic_smem(kernel, L::kSmem, configured);
    if (e != cudaSuccess) return e;
    const int pairs_max = pair_capacity(kernel, L::kSmem);
    if (pairs_max <= 0) return cudaErrorNotSupported;
    const long long items = (long long)a.num_q_tiles * a.batch * a.num_q_heads;
    if (items <= 0) return cudaSuccess;
    if (items > 0x7FFFFFFFLL - 65536) return cudaErrorInvalidValue;  // the work counter is an int32
    e = launch_prefill_order(a, stream);
    if (e != cudaSuccess) return e;
    const unsigned pairs = (unsigned)(items < pairs_max ? items : pairs_max);
    kernel<<<2 * pairs, L::kThreads, L::kSmem, stream>>>(a, *mq, *mk, *mv, *mr);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillArgs& a, int head_dim_qk, const CUtensorMap* mq, const CUtensorMap* mk,
                                const CUtensorMap* mv, const CUtensorMap* mr, cudaStream_t stream) {
    if (a.f8 || a.r8 || a.q_block != 512) return cudaErrorInvalidValue;
    if (head_dim_qk == 192) return a.paged ? cudaErrorInvalidValue : launch_pair_t<true, false>(a, mq, mk, mv, mr, stream);
    return a.paged ? launch_pair_t<false, true>(a, mq, mk, mv, mr, stream)
                   : launch_pair_t<false, false>(a, mq, mk, mv, mr, stream);
}

}  // namespace pa
