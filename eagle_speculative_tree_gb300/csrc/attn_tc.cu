// Split-KV paged tree attention on the 5th-generation tensor cores (bf16, head_dim 128).
//
// Same partial state as the CUDA-core kernel (m, l, acc per query row of one split),
// computed with tcgen05:
//   * one CTA = 128 query rows (row r = node i * G + g of one kv head; padded rows
//     are zero) x one split of the sequence's logical tokens, in 128-token tiles;
//   * warp 0 streams the split's K pages (four-stage ring) and warp 10 its V pages
//     (three stages) with TMA (one 16-token page x 64 head-dim columns per copy,
//     128-byte swizzle; lanes 0-7 issue one page each); the partly filled last page
//     of a sequence and pages past the split are written by the warp itself,
//     zero-filled, so nothing outside the sequence reaches the MMA;
//   * TMEM (512 columns, allocated by warp 1) holds two S buffers, Q and O; P_j is
//     written over S_j.  Warp 1 issues S = Q K^T with Q read from TMEM, warp 11 issues
//     O += P V with P read from TMEM, both as 128x128x16 tcgen05.mma instructions (two
//     issuers, so that the barrier waits of one stream overlap the other's MMAs).  Only
//     K and V pass through shared memory, whose bandwidth the MMAs and TMA share;
//   * warps 2-9 (two per TMEM lane quarter, one query row per thread, each warp one
//     half of the tile's columns) stage Q into TMEM, then per tile read S from TMEM,
//     apply the tree mask -- prefix tokens always, tree token S+j only when bit j of
//     the node's ancestor word is set ("Tech Radar: SGLang EAGLE-2", section 2 mask M
//     and section 5 bitmask) -- run the online softmax in base 2, write P as packed
//     bf16 back to TMEM, and rescale O in TMEM only when a row's running max grows by
//     more than 2^8.
// Every mbarrier wait is bounded; on expiry the CTA records TREESPEC_STATUS_TIMEOUT,
// drains its own tensor-core work, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace treespec {

namespace {

using namespace sm100;

constexpr int kM = 128;              // query rows per CTA = TMEM lanes
constexpr int kD = 128;              // head dim
constexpr int kBN = 128;             // tokens per tile
constexpr int kNSK = 4;              // K ring stages
constexpr int kNSV = 3;              // V ring stages
constexpr int kPanel = 128 * 128;    // one [128 rows][64 bf16] swizzled panel, bytes
constexpr int kTile = 2 * kPanel;    // [128][128] bf16
constexpr int kThreads = 384;        // K producer, S issuer, 8 softmax warps, V producer, PV issuer
constexpr int kWarpV = 10;           // the V producer warp
constexpr int kWarpPV = 11;          // the P V issuer warp
constexpr uint32_t kTmemCols = 512;
constexpr int kSB = 2;               // S buffers in TMEM: columns [0, 256); P_j overwrites S_j
constexpr uint32_t kColS = 0;
constexpr uint32_t kColQ = 256;      // Q (bf16 pairs): [256, 320)
constexpr uint32_t kColO = 384;      // O: [384, 512)
constexpr uint64_t kWaitNs = 2000000000ull;

// shared-memory map (offsets from a 1024-aligned base)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kNSK * kTile;
constexpr int kOffBar = kOffV + kNSV * kTile;
constexpr int kNumBars = 2 * kNSK + 2 * kNSV + 3 * kSB + 1 + 2 + 8;   // k/v full/empty, s_full, p_full, s_free, q_full, drain x2, xchg
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffXch = kOffMisc + 16;                      // softmax half-row exchange, 2 x 2 x 128 floats
constexpr int kOffAnc = kOffXch + 2 * 2 * 128 * 4;
constexpr int kSmemBytes = kOffAnc + kMaxNodes * 8;          // 232,200 bytes: within the 227 KB limit
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Bars {
    uint64_t k_full[kNSK], k_empty[kNSK], v_full[kNSV], v_empty[kNSV], s_full[kSB], p_full[kSB], s_free[kSB], q_full, drain[2], xchg[4][2];
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (d0, d1) = (a0 * b + c, a1 * b + c) as one packed f32x2 instruction
__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, float b, float c) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (d0, d1) += (a0, a1) as one packed f32x2 instruction
__device__ __forceinline__ void add_f32x2(float& d0, float& d1, float a0, float a1) {
    asm("{\n\t.reg .b64 ra, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
        "add.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1));
}

// CL > 1: the CL CTAs of a cluster hold consecutive row blocks of the same
// (sequence, kv head, split); each issues the TMA copies of every CL-th page of a tile
// multicast to all of them, and a stage is refilled only after all CL CTAs released it.
template <int CL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
    // the swizzled tiles need 1024-byte alignment: the dynamic shared memory of this
    // kernel (which has no static shared memory) starts at the window's base
    extern __shared__ __align__(1024) unsigned char sm[];
    Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    uint64_t* anc_s = reinterpret_cast<uint64_t*>(sm + kOffAnc);

    const int split = blockIdx.x;
    const int h = blockIdx.y / p.row_blocks, rb = blockIdx.y % p.row_blocks;
    const int b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = rb * kM;
    const int S = p.lens[b];

    if (S < 0) {                                   // invalid sequence: zeros (or the merge writes them)
        if (!p.merge && split == 0) {
            for (int e = tid; e < kM * (kD / 8); e += kThreads) {
                const int row = r0 + e / (kD / 8), c = e % (kD / 8);
                if (row >= p.R) continue;
                const int i = row / p.G, hq = h * p.G + row % p.G;
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                      ((size_t(b) * p.N + i) * p.Hq + hq) * kD) + c;
                *dst = make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int L = S + p.N;
    const int t0 = split * p.split_tokens;
    const int t1 = min(L, t0 + p.split_tokens);
    if (t0 >= t1) return;
    const int ntiles = (t1 - t0 + kBN - 1) / kBN;
    if (smem_u32(sm) & 1023u) {                    // never expected; refuse rather than misread tiles
        if (tid == 0) atomicOr(p.status, TREESPEC_STATUS_INTERNAL);
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < kNSK; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], CL);
        }
        for (int s = 0; s < kNSV; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], CL);
        }
        for (int s = 0; s < kSB; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->p_full[s], 256);
            mbar_init(&bars->s_free[s], 1);
        }
        mbar_init(&bars->q_full, 256);
        mbar_init(&bars->drain[0], 1);
        mbar_init(&bars->drain[1], 1);
        *abort_flag = 0;
        for (int f = 0; f < 8; ++f) mbar_init(&bars->xchg[f >> 1][f & 1], 2);
        fence_mbar_init();
    }
    for (int e = tid; e < p.N; e += kThreads) anc_s[e] = p.anc[size_t(b) * p.N + e];
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (CL > 1) cluster_sync_all();      // peers' barriers exist before any multicast
    const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
    constexpr uint16_t kMask = uint16_t((1u << CL) - 1u);
    const uint32_t tbase = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);

    if (warp == 0 || warp == kWarpV) {
        // ------------------------------------------------------------ TMA producers
        // warp 0 streams K (4 stages), warp 10 streams V (3 stages): a K stage is free again
        // as soon as S of its tile has been computed, a V stage only after P V.
        const bool is_v = warp == kWarpV;
        const int nst = is_v ? kNSV : kNSK;                 // ring stages
        uint64_t* full = is_v ? bars->v_full : bars->k_full;
        uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
        const uint16_t* src = static_cast<const uint16_t*>(is_v ? p.v : p.k);
        const CUtensorMap* map = is_v ? &tmv : &tmk;
        unsigned char* ring = sm + (is_v ? kOffV : kOffK);
        const int* ptab = p.page_table + size_t(b) * p.max_pages;
        if (lane == 0) tma_prefetch_desc(map);
        // Page ids in batches of four tiles, one warp-wide load each (lane l: page l & 7 of
        // tile 4 * batch + (l >> 3)), fetched a whole batch ahead: a page-table read that
        // waits behind the K/V traffic in L2 then never holds up the ring.
        auto fetch_batch = [&](int bi) -> int {
            const int jt = 4 * bi + (lane >> 3);
            const int pos0 = t0 + jt * kBN + (lane & 7) * 16;
            return (jt < ntiles && pos0 < t1) ? __ldg(ptab + (pos0 >> 4)) : -1;
        };
        int batch_cur = fetch_batch(0), batch_next = fetch_batch(1);
        for (int j = 0; j < ntiles; ++j) {
            const int stage = j % nst;
            if (j > 0 && (j & 3) == 0) {
                batch_cur = batch_next;
                batch_next = fetch_batch((j >> 2) + 1);
            }
            int page = __shfl_sync(0xffffffffu, batch_cur, ((j & 3) << 3) | (lane & 7));
            const int base = t0 + j * kBN;
            // lanes 0..7 own page `lane` of the tile: 1 = full page by TMA, 2 = written here
            // (the sequence's partly filled last page, a bad page id, or past the split)
            const int pos0 = base + lane * 16;
            int kind = 0;
            if (lane < 8) {
                kind = 2;
                if (pos0 < t1) {
                    const bool ok = page >= 0 && page < p.num_pool_pages;
                    if (!ok) atomicOr(p.status, TREESPEC_STATUS_BAD_PAGE);
                    if (ok && pos0 + 16 <= L) kind = 1;
                    if (!ok) page = -1;
                } else {
                    page = -1;
                }
            }
            if (j >= nst && !mbar_wait_bounded(&empty[stage], ((j / nst) - 1) & 1, kWaitNs)) {
                *abort_flag = 1;
                atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            unsigned char* dst = ring + stage * kTile;
            const unsigned manual = __ballot_sync(0xffffffffu, kind == 2);
            if (manual) {
                for (int pg = 0; pg < 8; ++pg) {
                    if (!((manual >> pg) & 1u)) continue;
                    const int pgid = __shfl_sync(0xffffffffu, page, pg);
                    const int q0 = base + pg * 16;
                    for (int c = lane; c < 16 * 16; c += 32) {      // 16 token rows x 16 chunks of 16 bytes
                        const int rr = c >> 4, ch = c & 15;
                        const int pos = q0 + rr;
                        uint4 val = make_uint4(0, 0, 0, 0);
                        if (pgid >= 0 && pos < t1) {
                            const size_t off = ((size_t(pgid) * p.ps + (pos & 15)) * p.Hkv + h) * kD + ch * 8;
                            val = __ldg(reinterpret_cast<const uint4*>(src + off));
                        }
                        *reinterpret_cast<uint4*>(dst + (ch >> 3) * kPanel + sw128_offset(pg * 16 + rr, ch & 7)) = val;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            const unsigned viatma = __ballot_sync(0xffffffffu, kind == 1);
            if (lane == 0) mbar_arrive_expect_tx(&full[stage], uint32_t(__popc(viatma)) * 2u * 2048u);
            __syncwarp();
            if (kind == 1 && (CL == 1 || (lane % CL) == int(rank))) {   // each page's two copies
                const int z = page * 16;
                if constexpr (CL == 1) {
                    tma_load_3d(dst + lane * 2048, map, 0, h, z, &full[stage]);
                    tma_load_3d(dst + kPanel + lane * 2048, map, 64, h, z, &full[stage]);
                } else {
                    tma_load_3d_multicast(dst + lane * 2048, map, 0, h, z, &full[stage], kMask);
                    tma_load_3d_multicast(dst + kPanel + lane * 2048, map, 64, h, z, &full[stage], kMask);
                }
            }
            __syncwarp();
        }
        if constexpr (CL > 1) {
            // every peer's release of every stage has landed here before this CTA may exit
            for (int s2 = 0; s2 < nst && s2 < ntiles; ++s2) {
                const int uses = (ntiles - s2 + nst - 1) / nst;
                if (!mbar_wait_bounded(&empty[s2], (uses - 1) & 1, kWaitNs)) {
                    *abort_flag = 1;
                    atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
                }
            }
        }
    } else if (warp == 1 || warp == kWarpPV) {
        // ------------------------------------------------------------ MMA issuers
        // Two independent streams into the CTA's tensor pipe: warp 1 issues S_j = Q K_j^T,
        // warp 11 issues O += P_j V_j.  They share no TMEM columns and no ring, so the
        // barrier waits of one overlap the other's MMAs instead of draining the pipe.
        // The whole warp runs the loop (all lanes wait, so control flow stays uniform) and
        // one elected lane issues each group of MMAs with its commits.  Each scheduler also
        // runs two busy softmax warps: issue code in a one-lane branch measured 108 cycles
        // per 128x128x16 MMA beside them, the warp-uniform form 69 (64 alone).
        {
            const bool pv = warp == kWarpPV;
            // both barriers of a step tested back to back, then waited (bounded) if needed;
            // the verdict is made warp-uniform
            auto ready2 = [&](uint64_t* x, uint32_t px, uint64_t* y, uint32_t py) -> bool {
                const bool rx = mbar_try_wait(x, px);
                const bool ry = mbar_try_wait(y, py);
                bool r = rx && ry;
                if (!__all_sync(0xffffffffu, r)) {
                    r = !*abort_flag && (rx || mbar_wait_bounded(x, px, kWaitNs)) &&
                        (ry || mbar_wait_bounded(y, py, kWaitNs));
                }
                return __all_sync(0xffffffffu, r);
            };
            bool ok = true;
            if (!pv) {
                constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false);
                // Q is read from TMEM (written there by the softmax warps), K from the ring;
                // a K-step or a stage moves only the start-address field of the K descriptor
                // (address >> 4 in the low 14 bits, which no offset in the window overflows)
                const uint64_t dk = smem_desc(sbase + kOffK, 16, 1024);
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->q_full, 0, kWaitNs));
                for (int j = 0; ok && j < ntiles; ++j) {
                    const int stage = j % kNSK;
                    // K_j has landed; S buffer j%2 is free once P_{j-2} V_{j-2} has read it
                    const int sb = j % kSB;
                    ok = j >= kSB ? ready2(&bars->k_full[stage], (j / kNSK) & 1, &bars->s_free[sb], ((j / kSB) - 1) & 1)
                                  : __all_sync(0xffffffffu, mbar_wait_bounded(&bars->k_full[stage], (j / kNSK) & 1, kWaitNs));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kb = dk + uint64_t((stage * kTile) >> 4);
                    const uint32_t d = tbase + kColS + uint32_t(sb) * 128u;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {   // 16 head dims = 8 packed columns of Q
                            const uint64_t koff = uint64_t(((kk >> 2) * kPanel + (kk & 3) * 32) >> 4);
                            mma_bf16_ts(d, tbase + kColQ + kk * 8, kb + koff, kIdS, kk > 0);
                        }
                        if constexpr (CL == 1) mma_commit(&bars->k_empty[stage]);
                        else mma_commit_multicast(&bars->k_empty[stage], kMask);
                        mma_commit(&bars->s_full[sb]);
                    }
                    __syncwarp();
                }
            } else {
                constexpr uint32_t kIdO = idesc_bf16_f32(128, 128, true);
                const uint64_t dv = smem_desc(sbase + kOffV, kPanel, 1024);
                for (int j = 0; ok && j < ntiles; ++j) {
                    const int stage = j % kNSV;
                    // P_j is in TMEM; V_j has landed
                    const int sb = j % kSB;
                    ok = ready2(&bars->p_full[sb], (j / kSB) & 1, &bars->v_full[stage], (j / kNSV) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vb = dv + uint64_t((stage * kTile) >> 4);
                    // P_j sits in S_j's buffer: tokens 0-63 in columns [0, 32), tokens 64-127 in
                    // [64, 96) (each softmax warp overwrites only its own half of S)
                    const uint32_t pcol = tbase + kColS + uint32_t(sb) * 128u;
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {  // 16 tokens = 8 packed columns of P
                            mma_bf16_ts(tbase + kColO, pcol + (kk >> 2) * 64 + (kk & 3) * 8,
                                        vb + uint64_t((kk * 2048) >> 4), kIdO, (j > 0 || kk > 0));
                        }
                        if constexpr (CL == 1) mma_commit(&bars->v_empty[stage]);
                        else mma_commit_multicast(&bars->v_empty[stage], kMask);
                        mma_commit(&bars->s_free[sb]);
                    }
                    __syncwarp();
                }
            }
            if (!ok && lane == 0) {
                *abort_flag = 1;
                atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
            }
            uint64_t* drain = &bars->drain[pv ? 1 : 0];
            if (elect_one()) mma_commit(drain);             // the pipe completes MMAs in issue order
            __syncwarp();
            mbar_wait_bounded(drain, 0, kWaitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax warps
        // Eight warps: warp w owns TMEM lane quarter (w % 4) = 32 query rows, and one
        // half of the tile's columns (warps 2-5: columns 0-63, warps 6-9: 64-127).  The
        // two warps of a quarter swap their half-row maxima through shared memory.
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;                    // 0 or 1
        const int t = quarter * 32 + lane;                   // query row in the block = TMEM lane
        const int r = r0 + t;
        const bool row_ok = r < p.R;
        const int i = row_ok ? r / p.G : 0;
        const int hq = h * p.G + (row_ok ? r % p.G : 0);
        const uint64_t anc = row_ok ? anc_s[i] : 0ull;
        const bool warp_rows = __any_sync(0xffffffffu, row_ok);
        const uint32_t tl = tbase + (uint32_t(quarter * 32) << 16);
        float* xch = reinterpret_cast<float*>(sm + kOffXch);  // [2 slot][2 half][128 rows]
        // Swap one float per row with the other half's warp of this quarter (both sit on
        // the same scheduler): write the value, arrive on the quarter's barrier of slot
        // seq&1 (two arrivals per phase); collect waits for that phase, sleeping in
        // hardware, and reads the partner's value.  Slot seq&1 is rewritten at seq+2 only
        // after the partner's arrival for seq+1, which follows its collect of seq.
        auto publish = [&](float value, int seq) {
            xch[((seq & 1) * 2 + half) * 128 + t] = value;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->xchg[quarter][seq & 1]);
        };
        auto collect = [&](int seq, bool* ok) -> float {
            *ok = mbar_wait_bounded(&bars->xchg[quarter][seq & 1], ((seq - 1) >> 1) & 1, kWaitNs);
            return xch[((seq & 1) * 2 + (half ^ 1)) * 128 + t];
        };
        {
            // this row's 64 head dims of Q into TMEM as 32 bf16 pairs (the A operand of S)
            const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                               ((size_t(b) * p.N + i) * p.Hq + hq) * kD) + half * 8;
            uint32_t qv[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 w = row_ok ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
                qv[4 * c] = w.x;
                qv[4 * c + 1] = w.y;
                qv[4 * c + 2] = w.z;
                qv[4 * c + 3] = w.w;
            }
            tmem_st32(tl + kColQ + half * 32, qv);
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&bars->q_full);

        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;                   // l: this warp's half of the row sum
        bool alive = true;
        uint32_t v[kBN / 2];
        for (int j = 0; j < ntiles && alive; ++j) {
            const int base = t0 + j * kBN;
            // which of this half's 64 columns the row may see, as two 32-bit words: prefix
            // columns below pref_end, tree columns [tree_lo, tree_hi) via the ancestor word
            const int pref_end = min(S, t1) - base;
            const int tree_lo = S - base, tree_hi = t1 - base;
            uint32_t mw[2];
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const int lo = 64 * half + 32 * w;
                const int np = min(max(pref_end - lo, 0), 32);
                uint32_t bits = np == 32 ? 0xffffffffu : ((1u << np) - 1u);
                const int nh = min(max(tree_hi - lo, 0), 32);
                const uint32_t hi_mask = nh == 32 ? 0xffffffffu : ((1u << nh) - 1u);
                uint32_t tb = 0;
                const int sh = lo - tree_lo;               // anc bit index of column lo
                if (sh >= 0) tb = sh < 64 ? uint32_t(anc >> sh) : 0u;
                else tb = -sh < 32 ? uint32_t(anc << (-sh)) : 0u;
                bits |= tb & hi_mask;
                mw[w] = row_ok ? bits : 0u;
            }
            const bool full = __all_sync(0xffffffffu, (mw[0] & mw[1]) == 0xffffffffu);
            const int sb = j % kSB;
            const uint32_t scol = tl + kColS + uint32_t(sb) * 128u + half * 64;
            // S of this half-row into v, masked columns set to -inf
            auto load_s = [&]() {
                if (warp_rows) {
                    tmem_ld32(scol, v);
                    tmem_ld32(scol + 32, v + 32);
                    tmem_wait_ld();
                }
                constexpr uint32_t kNegInf = 0xff800000u;
                if (!full) {
#pragma unroll
                    for (int c = 0; c < kBN / 2; ++c) v[c] = ((mw[c >> 5] >> (c & 31)) & 1u) ? v[c] : kNegInf;
                }
            };
            // probabilities 2^(s*scale - msub), rounded to bf16 and packed in pairs in place
            // (pair c overwrites v[c], whose value was read at pair c/2); returns their sum
            auto exps = [&](float msub) -> float {
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int c = 0; c < kBN / 4; ++c) {
                    float x0, x1;
                    fma_f32x2(x0, x1, __uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]), sc, -msub);
                    const float p0 = ex2(x0), p1 = ex2(x1);
                    v[c] = pack_bf16x2(p0, p1);
                    if (c & 1) add_f32x2(a2, a3, p0, p1);
                    else add_f32x2(a0, a1, p0, p1);
                }
                return (a0 + a1) + (a2 + a3);
            };
            if (!mbar_wait_bounded(&bars->s_full[sb], (j / kSB) & 1, kWaitNs)) { alive = false; break; }
            tc_fence_after();
            load_s();
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kBN / 2; c += 8) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    mx[e] = fmax3(mx[e], __uint_as_float(v[c + 2 * e]), __uint_as_float(v[c + 2 * e + 1]));
            }
            const float mhalf = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
            publish(mhalf, j + 1);
            // Speculate that the running max stays: the exponentials taken now are final
            // unless some row's max over both halves rises more than 8 above m_used.
            const bool spec = __all_sync(0xffffffffu, mhalf * sc <= m_used + 8.f);
            float lsum = 0.f;
            if (spec) lsum = exps(m_used == -INFINITY ? 0.f : m_used);
            // the row's max over both halves (identical in the two warps of the quarter)
            bool xok = true;
            const float mt = fmaxf(mhalf, collect(j + 1, &xok)) * sc;   // scale > 0 commutes with max
            if (!xok) { alive = false; break; }
            bool resc = false;
            float alpha = 1.f;
            const bool grow = mt > m_used + 8.f;
            if (grow) {
                alpha = ex2(m_used - mt);
                resc = m_used != -INFINITY;
                l *= alpha;
                m_used = mt;
            }
            if (!spec || __any_sync(0xffffffffu, grow)) {
                if (spec) load_s();                        // v holds P: S is still in TMEM
                lsum = exps(m_used == -INFINITY ? 0.f : m_used);
            }
            l += lsum;
            if (__any_sync(0xffffffffu, resc)) {
                // O may only be rescaled once P_{j-1} V_{j-1} is in it (this warp's 64 columns)
                if (!mbar_wait_bounded(&bars->s_free[(j - 1) % kSB], ((j - 1) / kSB) & 1, kWaitNs)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const float f = resc ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tl + kColO + half * 64 + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                    tmem_st32(tl + kColO + half * 64 + c * 32, o);
                }
            }
            tc_fence_after();
            if (warp_rows) tmem_st32(scol, v);             // P over the first 32 columns of this half of S
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[sb]);
        }
        if (!alive) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        } else if (mbar_wait_bounded(&bars->s_free[(ntiles - 1) % kSB], ((ntiles - 1) / kSB) & 1, kWaitNs)) {
            tc_fence_after();
            // the row sum over both halves
            bool xok = true;
            publish(l, ntiles + 1);
            const float lrow = l + collect(ntiles + 1, &xok);
            if (!xok) {
                *abort_flag = 1;
                atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
            }
            const float inv = 1.f / lrow;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                if (warp_rows) {
                    tmem_ld32(tl + kColO + half * 64 + c * 32, o);
                    tmem_wait_ld();
                }
                if (!row_ok) continue;
                const int col0 = half * 64 + c * 32;
                if (!p.merge) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                          ((size_t(b) * p.N + i) * p.Hq + hq) * kD + col0);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t w4[4];
#pragma unroll
                        for (int k2 = 0; k2 < 4; ++k2) {
                            const int idx = e * 8 + k2 * 2;
                            w4[k2] = pack_bf16x2(__uint_as_float(o[idx]) * inv, __uint_as_float(o[idx + 1]) * inv);
                        }
                        dst[e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                } else {
                    const size_t pr = (size_t(b * p.Hkv + h) * p.num_splits + split) * p.R + r;
                    float4* dst = reinterpret_cast<float4*>(p.part_acc + pr * kD + col0);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                             __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
                    if (c == 0 && half == 0) {
                        p.part_ml[pr * 2] = m_used;
                        p.part_ml[pr * 2 + 1] = lrow;
                    }
                }
            }
        } else {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tbase, kTmemCols);
    if constexpr (CL > 1) cluster_sync_all();      // no peer still writes into this CTA
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

}  // namespace

bool attn_tc_supported(int dtype, int D) { return dtype == TREESPEC_DTYPE_BF16 && D == kD; }

template <int CL>
cudaError_t launch_cluster(const AttnParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t s) {
    auto kern = attn_tc_kernel<CL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_splits, p.Hkv * p.row_blocks, p.B);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = CL;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, p, mk, mv);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Pairs of row blocks of one kv head share each K/V copy (multicast): half the L2 reads
// and TMA copies per CTA.  Clusters of 4 fit only 144 of the 152 SMs (whole GPCs),
// clusters of 2 all of them.  Measured on 32 x 8192-token sequences (64 q / 8 kv heads,
// 64 tree nodes): 0.532 ms without clusters, 0.493 ms with pairs, 0.60 ms with 4.
int attn_tc_cluster_size(int row_blocks) { return row_blocks % 2 == 0 ? 2 : 1; }

cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s) {
    CUtensorMap mk, mv;
    const long long pool_tokens = (long long)p.num_pool_pages * p.ps;
    if (!make_pool_map(&mk, p.k, p.Hkv, pool_tokens) || !make_pool_map(&mv, p.v, p.Hkv, pool_tokens))
        return cudaErrorInvalidValue;
    switch (attn_tc_cluster_size(p.row_blocks)) {
        case 4: return launch_cluster<4>(p, mk, mv, s);
        case 2: return launch_cluster<2>(p, mk, mv, s);
        default: return launch_cluster<1>(p, mk, mv, s);
    }
}

}  // namespace treespec
