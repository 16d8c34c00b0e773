// Split-KV paged tree attention on the 5th-generation tensor cores (bf16, head_dim 128).
//
// Same partial state as the CUDA-core kernel (m, l, acc per query row of one split),
// computed with tcgen05.  One kernel template, two shapes of work:
//
//   attn_tc_kernel<false> -- one CTA = 128 query rows (row r = node i * G + g of one kv
//     head; padded rows are zero) x one split of the sequence's logical tokens, in
//     128-token tiles.  Warp 0 streams the split's K pages (four-stage ring) and warp 6
//     its V pages (three stages) with TMA (one 16-token page x 64 head-dim columns per
//     copy, 128-byte swizzle; lanes 0-7 issue one page each).  The row blocks of one kv
//     head are adjacent in the grid, so they run together and the later readers of a
//     K/V tile find it in L2.
//
//   attn_tc_kernel<true> -- a cluster of two CTAs (along the grid's x) holds two adjacent
//     128-row blocks of one kv head (rank 0 the even block) and computes both with
//     256-row MMAs that span the pair (cta_group::2): S = Q K^T and O += P V are
//     256 x 128 x 16 instructions
//     issued by rank 0, each CTA's 128 rows in its own tensor memory.  The B operand is
//     split between the pair's shared memories, so each CTA copies only half of every
//     tile: of K the 64 tokens of pages 4*rank .. 4*rank+3 (both head-dim halves), of V
//     head dims 64*rank .. 64*rank+63 of all eight pages.  Half the L2 reads and half
//     the shared-memory operand traffic per SM of the one-CTA shape, with every copy a
//     plain TMA load into the CTA's own memory.  Rank 1's warp 1 forwards the landing
//     of each of its stages to rank 0 (a remote mbarrier arrive, in the order rank 0's
//     MMAs consume them); rank 0 commits every MMA group to the barriers of both CTAs.
//
// In both shapes:
//   * the partly filled last page of a sequence and pages past the split are written by
//     the producer warp itself, zero-filled, so nothing outside the sequence reaches
//     the MMA;
//   * TMEM (512 columns) holds two S buffers, Q, one P buffer and O.  The issuer runs
//     S_0, S_1, P_0 V_0, S_2, P_1 V_1, S_3, ...: S_{j+2} reuses the buffer of S_j as soon
//     as the softmax has read it, and the softmax of tile j+1 runs while the tensor pipe
//     computes P_j V_j and S_{j+2}.  Only K and V pass through shared memory;
//   * warps 2-5 (one per TMEM lane quarter, one query row per thread over all of the
//     tile's columns, so a row's maximum needs no exchange between warps) stage Q into
//     TMEM, then per tile read S from TMEM, apply the tree mask -- prefix tokens always,
//     tree token S+j only when the node's ancestor set holds j ("Tech Radar: SGLang
//     EAGLE-2", section 2 mask M and section 5 bitmask) -- run the online softmax in
//     base 2, write P as packed bf16 into the P buffer once P_{j-1} V_{j-1} has read it,
//     and rescale O in TMEM (after that MMA too) only when a row's running max grows by
//     more than 2^8.
// Every mbarrier wait is bounded; on expiry the CTA records TREESPEC_STATUS_TIMEOUT,
// stops issuing, drains its own copies and tensor-core work, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_tc_parts.cuh"

namespace treespec {

namespace {

using namespace sm100;
using tcparts::kBN;                  // tokens per tile
using tcparts::kD;                   // head dim

constexpr int kM = 128;              // query rows per CTA = TMEM lanes
constexpr int kThreads = 224;        // K producer, MMA issuer, 4 softmax warps, V producer
constexpr int kWarpV = 6;            // the V producer warp
constexpr uint32_t kTmemCols = 512;
constexpr int kSB = 2;               // S buffers in TMEM: columns [0, 256)
constexpr uint32_t kColS = 0;
constexpr uint32_t kColQ = 256;      // Q (bf16 pairs): [256, 320)
constexpr uint32_t kColP = 320;      // P (bf16 pairs): [320, 384)
constexpr uint32_t kColO = 384;      // O: [384, 512)

// Ring geometry.  A stage holds what one CTA copies of one tile, as 128-byte-swizzled
// panels of 64 head dims (128-byte rows).  One CTA: K and V stages are whole tiles, two
// [128 tokens][64 dims] panels.  CTA pair: a K stage is this CTA's 64 tokens as two
// [64][64] panels, a V stage this CTA's 64 head dims of all 128 tokens, one [128][64]
// panel; the halved stages make room for deeper rings.
template <bool kPair>
struct Cfg {
    static constexpr int kNSK = kPair ? 7 : 4;                       // K ring stages
    static constexpr int kNSV = kPair ? 6 : 3;                       // V ring stages
    static constexpr int kKPanel = (kPair ? 64 : 128) * 128;         // bytes of one K panel
    static constexpr int kKStage = 2 * kKPanel;
    static constexpr int kVPanel = 128 * 128;
    static constexpr int kVStage = (kPair ? 1 : 2) * kVPanel;
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kNSK * kKStage;
    static constexpr int kOffBar = kOffV + kNSV * kVStage;
    struct Bars {
        // k/v_full: this CTA's copies landed (TMA bytes + one producer arrive); k/v_peer
        // (rank 0 of a pair): the other CTA's stage landed; k/v_empty: the stage's MMAs
        // completed; s_full, p_full, pv_done, q_full, drain: the S / P / PV / Q hand-offs
        uint64_t k_full[kNSK], k_empty[kNSK], k_peer[kNSK], v_full[kNSV], v_empty[kNSV], v_peer[kNSV];
        uint64_t s_full[kSB], p_full[kSB], pv_done, q_full, drain;
    };
    static constexpr int kOffMisc = kOffBar + int(sizeof(Bars));
    static constexpr int kOffAnc = kOffMisc + 16;
    static constexpr int kSmemBytes = kOffAnc + kMaxNodes * kAncWords * 8;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kKPanel % 1024 == 0 && kVPanel % 1024 == 0, "swizzled panels need 1024-byte alignment");
};

template <bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
    using C = Cfg<kPair>;
    using Bars = typename C::Bars;
    constexpr int kNSK = C::kNSK, kNSV = C::kNSV;
    // the swizzled tiles need 1024-byte alignment: the dynamic shared memory of this
    // kernel (which has no static shared memory) starts at the window's base
    extern __shared__ __align__(1024) unsigned char sm[];
    Bars* bars = reinterpret_cast<Bars*>(sm + C::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(sm + C::kOffMisc + 4);
    uint64_t* anc_s = reinterpret_cast<uint64_t*>(sm + C::kOffAnc);
    grid_dep_wait();                               // the prologue's ancestor words, lengths and counts

    // One CTA: grid (split, kv head x row block, sequence).  Pair: grid (split x 2 + rank,
    // kv head x pair of row blocks, sequence) with clusters of two along x -- the
    // hardware pairs the CTAs whose x differs in its lowest bit; rank 0 holds the even
    // row block of the pair.
    const uint32_t rank = kPair ? uint32_t(blockIdx.x & 1) : 0u;
    const int split = kPair ? int(blockIdx.x >> 1) : int(blockIdx.x);
    const int units_y = kPair ? p.row_blocks / 2 : p.row_blocks;
    const int h = blockIdx.y / units_y;
    const int rb = kPair ? 2 * int(blockIdx.y % units_y) + int(rank) : int(blockIdx.y % units_y);
    const int b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = rb * kM;
    const int S = p.lens[b];

    // Every early return below is taken by both CTAs of a pair alike (same sequence,
    // split and launch shape), so neither waits for a partner that has left.
    if (S < 0) {                                   // invalid sequence: zeros (or the merge writes them)
        if (!p.merge && split == 0) tcparts::zero_rows(p, b, h, r0, kM, kThreads);
        return;
    }
    const int nb = p.nn[b];                        // rows of nodes nb.. are padding: zero output
    const int L = S + nb;
    const int t0 = split * p.split_tokens;
    const int t1 = min(L, t0 + p.split_tokens);
    if (t0 >= t1) return;
    const int ntiles = (t1 - t0 + kBN - 1) / kBN;
    if ((smem_u32(sm) & 1023u) || (kPair && cluster_ctarank() != rank)) {   // never expected
        if (tid == 0) atomicOr(p.status, TREESPEC_STATUS_INTERNAL);
        return;
    }

    // rank 0 of a pair hears from 4 softmax warps of each CTA (one arrive per warp); a single
    // CTA from each of its 128 softmax threads
    constexpr uint32_t kSoftmaxArrivals = kPair ? 8u : uint32_t(kM);
    if (tid == 0) {
        for (int s = 0; s < kNSK; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->k_peer[s], 1);
        }
        for (int s = 0; s < kNSV; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->v_peer[s], 1);
        }
        for (int s = 0; s < kSB; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], kSoftmaxArrivals);
        }
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->q_full, kSoftmaxArrivals);
        mbar_init(&bars->drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int e = tid; e < p.N * kAncWords; e += kThreads) anc_s[e] = p.anc[size_t(b) * p.N * kAncWords + e];
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(tmem_slot, kTmemCols);       // one warp of each CTA of the pair
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (kPair) cluster_sync_all();       // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);

    auto wait_bar = [&](uint64_t* bar, uint32_t parity, uint64_t limit) -> bool {
        return mbar_wait_bounded(bar, parity, limit);
    };
    auto test_bar = [&](uint64_t* bar, uint32_t parity) -> bool { return mbar_try_wait(bar, parity); };

    if (warp == 0 || warp == kWarpV) {
        // ------------------------------------------------------------ TMA producers
        // warp 0 streams K, warp 6 streams V: a K stage is free again as soon as S of its
        // tile has been computed, a V stage only after P V.  This CTA's share of a tile:
        // pages [pg0, pg0 + npg) of its eight, head-dim panels [dp0, dp0 + ndp) of two.
        const bool is_v = warp == kWarpV;
        tcparts::ProducerArgs a;
        a.map = is_v ? &tmv : &tmk;
        a.src = static_cast<const uint16_t*>(is_v ? p.v : p.k);
        a.ring = sm + (is_v ? C::kOffV : C::kOffK);
        a.full = is_v ? bars->v_full : bars->k_full;
        a.empty = is_v ? bars->v_empty : bars->k_empty;
        a.nst = is_v ? kNSV : kNSK;
        a.stage_bytes = is_v ? C::kVStage : C::kKStage;
        a.panel_bytes = is_v ? C::kVPanel : C::kKPanel;
        a.pg0 = (kPair && !is_v) ? 4 * int(rank) : 0;
        a.npg = (kPair && !is_v) ? 4 : 8;
        a.dp0 = (kPair && is_v) ? int(rank) : 0;
        a.ndp = (kPair && is_v) ? 1 : 2;
        int armed = 0;
        tcparts::produce_pages<kBN>(p, a, b, h, t0, t1, L, ntiles, armed, abort_flag);
        tcparts::drain_copies(a, armed);
    } else if (warp == 1 && kPair && rank == 1) {
        // ------------------------------------------------------------ stage forwarder (pair, rank 1)
        // Rank 0's MMAs read this CTA's half of each stage: tell rank 0 when it has landed,
        // in the order the MMAs consume the stages (K_0, K_1, V_0, K_2, V_1, K_3, ...).
        auto forward = [&](bool is_v, int j) -> bool {
            const int nst = is_v ? kNSV : kNSK, st = j % nst;
            uint64_t* f = is_v ? &bars->v_full[st] : &bars->k_full[st];
            uint64_t* peer = is_v ? &bars->v_peer[st] : &bars->k_peer[st];
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(f, uint32_t(j / nst) & 1u, p.wait_ns));
            if (ok && lane == 0) mbar_arrive_cluster(cluster_addr(smem_u32(peer), 0));
            return ok;
        };
        bool ok = true;
        for (int j = 0; ok && j < kSB && j < ntiles; ++j) ok = forward(false, j);
        for (int j = 0; ok && j < ntiles; ++j) {
            ok = *abort_flag == 0 && forward(true, j);
            if (ok && j + kSB < ntiles) ok = forward(false, j + kSB);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (all lanes wait, so control flow stays uniform) and
        // one elected lane issues each group of MMAs with its commits (issue code in a
        // one-lane branch measured 108 cycles per 128x128x16 MMA beside busy softmax
        // warps, the warp-uniform form 69; 64 alone).
        auto ready = [&](uint64_t* x, uint32_t px, uint64_t* y, uint32_t py, uint64_t* z, uint32_t pz) -> bool {
            const bool rx = !x || test_bar(x, px);
            const bool ry = !y || test_bar(y, py);
            const bool rz = !z || test_bar(z, pz);
            bool r = rx && ry && rz;
            if (!__all_sync(0xffffffffu, r)) {
                r = !*abort_flag && (rx || wait_bar(x, px, p.wait_ns)) && (ry || wait_bar(y, py, p.wait_ns)) &&
                    (rz || wait_bar(z, pz, p.wait_ns));
            }
            return __all_sync(0xffffffffu, r);
        };
        // a group's completion reaches this CTA's barrier, and the other CTA's of a pair
        auto commit = [&](uint64_t* bar) {
            if constexpr (kPair) {
                mma_commit_pair(smem_u32(bar));
                mma_commit_pair(cluster_addr(smem_u32(bar), 1));
            } else {
                mma_commit(bar);
            }
        };
        auto mma = [&](uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
            if constexpr (kPair) mma_bf16_ts_pair(d, a, bdesc, idesc, acc);
            else mma_bf16_ts(d, a, bdesc, idesc, acc);
        };
        constexpr uint32_t kIdS = idesc_bf16_f32(kPair ? 256 : 128, 128, false);
        constexpr uint32_t kIdO = idesc_bf16_f32(kPair ? 256 : 128, 128, true);
        // Q is read from TMEM (written there by the softmax warps), K and V from the rings;
        // a K-step or a stage moves only the start-address field of a descriptor (address
        // >> 4 in the low 14 bits, which no offset in the window overflows)
        const uint64_t dk = smem_desc(sbase + C::kOffK, 16, 1024);
        const uint64_t dv = smem_desc(sbase + C::kOffV, C::kVPanel, 1024);
        // S_j into buffer j % 2 (the softmax has read S_{j-2} from it: p_full of tile j-2)
        auto issue_s = [&](int j) -> bool {
            const int stage = j % kNSK, sb = j % kSB;
            const uint32_t kp = uint32_t(j / kNSK) & 1u;
            const bool ok = ready(&bars->k_full[stage], kp, kPair ? &bars->k_peer[stage] : nullptr, kp,
                                  j >= kSB ? &bars->p_full[sb] : nullptr, uint32_t((j / kSB) - 1) & 1u);
            if (!ok) return false;
            tc_fence_after();
            const uint64_t kb = dk + uint64_t((stage * C::kKStage) >> 4);
            const uint32_t d = tbase + kColS + uint32_t(sb) * 128u;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {   // 16 head dims = 8 packed columns of Q
                    const uint64_t koff = uint64_t(((kk >> 2) * C::kKPanel + (kk & 3) * 32) >> 4);
                    mma(d, tbase + kColQ + kk * 8, kb + koff, kIdS, kk > 0);
                }
                commit(&bars->k_empty[stage]);
                commit(&bars->s_full[sb]);
            }
            __syncwarp();
            return true;
        };
        bool ok = __all_sync(0xffffffffu, wait_bar(&bars->q_full, 0, p.wait_ns));
        for (int j = 0; ok && j < kSB && j < ntiles; ++j) ok = issue_s(j);
        for (int j = 0; ok && j < ntiles; ++j) {
            // O += P_j V_j once P_j is in TMEM and V_j has landed, then S_{j+2}
            const int stage = j % kNSV;
            const uint32_t vp = uint32_t(j / kNSV) & 1u;
            ok = ready(&bars->p_full[j % kSB], uint32_t(j / kSB) & 1u, &bars->v_full[stage], vp,
                       kPair ? &bars->v_peer[stage] : nullptr, vp);
            if (!ok) break;
            tc_fence_after();
            const uint64_t vb = dv + uint64_t((stage * C::kVStage) >> 4);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)     // 16 tokens = 8 packed columns of P
                    mma(tbase + kColO, tbase + kColP + kk * 8, vb + uint64_t((kk * 2048) >> 4), kIdO, (j > 0 || kk > 0));
                commit(&bars->v_empty[stage]);
                commit(&bars->pv_done);
            }
            __syncwarp();
            if (j + kSB < ntiles) ok = issue_s(j + kSB);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        }
        if (elect_one()) {                                  // the pipe completes MMAs in issue order
            if constexpr (kPair) mma_commit_pair(smem_u32(&bars->drain));
            else mma_commit(&bars->drain);
        }
        __syncwarp();
        wait_bar(&bars->drain, 0, kDefaultWaitNs);
        __syncwarp();
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------------------ softmax warps
        // Four warps: warp w owns TMEM lane quarter (w % 4) = 32 query rows, one row per
        // thread over all 128 columns of a tile.
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;                   // query row in the block = TMEM lane
        const int r = r0 + t;
        const bool row_in = r < p.R;
        const int i = row_in ? r / p.G : 0;
        const int hq = h * p.G + (row_in ? r % p.G : 0);
        const bool row_ok = row_in && i < nb;                // a padding slot's row is not computed
        const uint64_t anc0 = row_ok ? anc_s[i * kAncWords] : 0ull;     // the node's ancestor-or-self set
        const uint64_t anc1 = row_ok ? anc_s[i * kAncWords + 1] : 0ull;
        const bool warp_rows = __any_sync(0xffffffffu, row_ok);
        const uint32_t tl = tbase + (uint32_t(quarter * 32) << 16);
        // Q and P hand-offs go to the MMA issuer: this CTA's, or rank 0's of a pair
        auto signal_issuer = [&](uint64_t* bar) {
            if constexpr (kPair) {
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(bar);
                    else mbar_arrive_cluster(cluster_addr(smem_u32(bar), 0));
                }
            } else {
                mbar_arrive(bar);
            }
        };
        {
            // this row of Q into TMEM as 64 bf16 pairs (the A operand of S)
            const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                               ((size_t(b) * p.N + i) * p.Hq + hq) * kD);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t qv[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 w = row_ok ? __ldg(qsrc + hh * 8 + c) : make_uint4(0, 0, 0, 0);
                    qv[4 * c] = w.x;
                    qv[4 * c + 1] = w.y;
                    qv[4 * c + 2] = w.z;
                    qv[4 * c + 3] = w.w;
                }
                tmem_st32(tl + kColQ + hh * 32, qv);
                tmem_wait_st();
            }
        }
        tc_fence_before();
        signal_issuer(&bars->q_full);

        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool alive = true;
        uint32_t v[kBN];
        for (int j = 0; j < ntiles; ++j) {
            uint32_t mw[4];
            tcparts::tile_mask<kBN>(mw, t0 + j * kBN, S, t1, anc0, anc1, row_ok);
            const bool full = __all_sync(0xffffffffu, (mw[0] & mw[1] & mw[2] & mw[3]) == 0xffffffffu);
            const int sb = j % kSB;
            const uint32_t scol = tl + kColS + uint32_t(sb) * 128u;
            if (!wait_bar(&bars->s_full[sb], (j / kSB) & 1, p.wait_ns)) { alive = false; break; }
            tc_fence_after();
            if (warp_rows) {
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(scol + c * 32, v + c * 32);
                tmem_wait_ld();
            }
            bool resc = false;
            float alpha = 1.f, ts;
            if (__all_sync(0xffffffffu, tcparts::softmax_tile_fast<kBN>(v, mw, full, sc, m_used, ts))) {
                l += ts;                                     // no row's max moved past m_used + 8
            } else {                                         // S again, and the exact path
                if (warp_rows) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(scol + c * 32, v + c * 32);
                    tmem_wait_ld();
                }
                tcparts::softmax_tile<kBN>(v, mw, full, sc, m_used, l, resc, alpha);
            }
            // the P buffer and O are free once P_{j-1} V_{j-1} has completed
            if (j > 0 && !wait_bar(&bars->pv_done, (j - 1) & 1, p.wait_ns)) {
                alive = false;
                break;
            }
            tc_fence_after();
            if (warp_rows) {
                tmem_st32(tl + kColP, v);
                tmem_st32(tl + kColP + 32, v + 32);
            }
            tmem_wait_st();
            if (__any_sync(0xffffffffu, resc)) tcparts::rescale_o(tl + kColO, resc ? alpha : 1.f);
            tc_fence_before();
            signal_issuer(&bars->p_full[sb]);
        }
        if (!alive || !wait_bar(&bars->pv_done, (ntiles - 1) & 1, p.wait_ns)) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        } else {
            tc_fence_after();
            tcparts::write_row(p, tl + kColO, warp_rows, row_in, row_ok, b, i, hq, h, split, r, m_used, l);
        }
    }

    tc_fence_before();
    __syncthreads();
    // Neither CTA of a pair leaves while the other may still signal its barriers or, for
    // rank 1, while rank 0's tensor-core work may still use its memory (rank 0 drained it
    // above); every wait before this point is bounded, so both CTAs arrive.
    if constexpr (kPair) cluster_sync_all();
    tc_fence_after();
    if (warp == 1) {
        if constexpr (kPair) tmem_dealloc_pair(tbase, kTmemCols);
        else tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 3-D view of a page pool [P][16][Hkv][128] bf16 as (head dim, kv head, pool token),
// copied in boxes of 64 head-dim columns x 1 head x 16 tokens (one page) with
// 128-byte swizzle.
bool make_pool_map(CUtensorMap* map, const void* base, int Hkv, long long pool_tokens) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(Hkv), cuuint64_t(pool_tokens)};
    cuuint64_t strides[2] = {cuuint64_t(kD) * 2, cuuint64_t(Hkv) * kD * 2};
    cuuint32_t box[3] = {64, 1, 16};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool attn_tc_supported(int dtype, int D) { return dtype == TREESPEC_DTYPE_BF16 && D == kD; }

template <bool kPair>
static cudaError_t launch_tc(const AttnParams& p, cudaStream_t s) {
    if (kPair && p.row_blocks % 2 != 0) return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    const long long pool_tokens = (long long)p.num_pool_pages * p.ps;
    if (!make_pool_map(&mk, p.k, p.Hkv, pool_tokens) || !make_pool_map(&mv, p.v, p.Hkv, pool_tokens))
        return cudaErrorInvalidValue;
    auto kern = attn_tc_kernel<kPair>;
    constexpr int smem = Cfg<kPair>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = kPair ? dim3(2 * p.num_splits, p.Hkv * (p.row_blocks / 2), p.B)
                        : dim3(p.num_splits, p.Hkv * p.row_blocks, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;                    // the two row blocks of a pair
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = kPair ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, mk, mv);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s) { return launch_tc<false>(p, s); }
cudaError_t launch_attn_tc_2sm(const AttnParams& p, cudaStream_t s) { return launch_tc<true>(p, s); }

}  // namespace treespec
