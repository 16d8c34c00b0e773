// Split-KV paged tree attention on the 5th-generation tensor cores (bf16, head_dim 128).
//
// Same partial state as the CUDA-core kernel (m, l, acc per query row of one split),
// computed with tcgen05:
//   * one CTA = 128 query rows (row r = node i * G + g of one kv head; padded rows
//     are zero) x one split of the sequence's logical tokens, in 128-token tiles;
//   * warp 0 streams the split's K pages and warp 10 its V pages with TMA (one
//     16-token page x 64 head-dim columns per copy, 128-byte swizzle; lanes 0-7 issue
//     one page each) into two three-stage rings; the partly filled last page of a
//     sequence and pages past the split are written by the warp itself, zero-filled,
//     so nothing outside the sequence reaches the MMA;
//   * warp 1 allocates all 512 TMEM columns (S and P double-buffered, O) and issues
//     S = Q K^T from shared memory and O += P V with P read from TMEM, as
//     128x128x16 tcgen05.mma instructions;
//   * warps 2-9 (two per TMEM lane quarter, one query row per thread, each warp one
//     half of the tile's columns) read S from TMEM, apply the tree mask -- prefix tokens always, tree token S+j only when bit
//     j of the node's ancestor word is set ("Tech Radar: SGLang EAGLE-2", section 2
//     mask M and section 5 bitmask) -- run the online softmax in base 2, write P as
//     packed bf16 back to TMEM, and rescale O in TMEM only when a row's running max
//     grows by more than 2^8.
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
constexpr int kNS = 3;               // K/V ring stages
constexpr int kPanel = 128 * 128;    // one [128 rows][64 bf16] swizzled panel, bytes
constexpr int kTile = 2 * kPanel;    // [128][128] bf16
constexpr int kThreads = 352;        // K producer, MMA, 8 softmax warps, V producer
constexpr int kWarpV = 10;           // the V producer warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;        // S double buffer: columns [0, 256)
constexpr uint32_t kColP = 256;      // P double buffer (bf16 pairs): [256, 384)
constexpr uint32_t kColO = 384;      // O: [384, 512)
constexpr uint64_t kWaitNs = 2000000000ull;

// shared-memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;
constexpr int kOffV = kOffK + kNS * kTile;
constexpr int kOffBar = kOffV + kNS * kTile;
constexpr int kNumBars = 4 * kNS + 2 + 2 + 2 + 2 + 2;   // k/v full/empty, s_full/empty, p_full, p_free, q_full, drain
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kOffFlag = kOffMisc + 16;                     // exchange sequence numbers, 4 quarters x 2 halves
constexpr int kOffXch = kOffFlag + 32;                      // softmax half-row exchange, 2 x 2 x 128 floats
constexpr int kOffAnc = kOffXch + 2 * 2 * 128 * 4;
constexpr int kSmemBytes = kOffAnc + kMaxNodes * 8;          // 232,160 bytes: within the 227 KB limit
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Bars {
    uint64_t k_full[kNS], k_empty[kNS], v_full[kNS], v_empty[kNS], s_full[2], s_empty[2], p_full[2], p_free[2], q_full, drain;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], CL);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], CL);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->s_empty[s], 256);
            mbar_init(&bars->p_full[s], 256);
            mbar_init(&bars->p_free[s], 1);
        }
        mbar_init(&bars->q_full, 256);
        mbar_init(&bars->drain, 1);
        *abort_flag = 0;
        for (int f = 0; f < 8; ++f) reinterpret_cast<volatile int*>(sm + kOffFlag)[f] = 0;
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
        // warp 0 streams K, warp 10 streams V: a K stage is free again as soon as S of
        // its tile has been computed, a V stage only after P V, so each has its own ring.
        const bool is_v = warp == kWarpV;
        uint64_t* full = is_v ? bars->v_full : bars->k_full;
        uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
        const uint16_t* src = static_cast<const uint16_t*>(is_v ? p.v : p.k);
        const CUtensorMap* map = is_v ? &tmv : &tmk;
        unsigned char* ring = sm + (is_v ? kOffV : kOffK);
        const int* ptab = p.page_table + size_t(b) * p.max_pages;
        if (lane == 0) tma_prefetch_desc(map);
        // page ids of tile j (lane k < 8 holds page k of the tile), fetched one tile ahead
        auto fetch_pages = [&](int j) -> int {
            const int pos0 = t0 + j * kBN + lane * 16;
            return (lane < 8 && j < ntiles && pos0 < t1) ? __ldg(ptab + (pos0 >> 4)) : -1;
        };
        int page_next = fetch_pages(0);
        for (int j = 0; j < ntiles; ++j) {
            const int stage = j % kNS;
            int page = page_next;
            page_next = fetch_pages(j + 1);
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
            if (j >= kNS && !mbar_wait_bounded(&empty[stage], ((j / kNS) - 1) & 1, kWaitNs)) {
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
            for (int s2 = 0; s2 < kNS && s2 < ntiles; ++s2) {
                const int uses = (ntiles - s2 + kNS - 1) / kNS;
                if (!mbar_wait_bounded(&empty[s2], (uses - 1) & 1, kWaitNs)) {
                    *abort_flag = 1;
                    atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Order S_0, S_1, then S_{j+2} before P_j V_j: the next scores are already queued
        // when the softmax hands over P_j, so the softmax warps never wait for S.
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t kIdO = idesc_bf16_f32(128, 128, true);
            // descriptors of the first K-step of Q, of ring stage 0 of K and of V; a
            // step or a stage moves only the start-address field (address >> 4 in the
            // low 14 bits, which no offset inside the 227 KB window overflows)
            const uint64_t dq = smem_desc(sbase + kOffQ, 16, 1024);
            const uint64_t dk = smem_desc(sbase + kOffK, 16, 1024);
            const uint64_t dv = smem_desc(sbase + kOffV, kPanel, 1024);
            bool ok = mbar_wait_bounded(&bars->q_full, 0, kWaitNs);
            auto issue_s = [&](int j) -> bool {
                const int stage = j % kNS;
                if (!mbar_wait_bounded(&bars->k_full[stage], (j / kNS) & 1, kWaitNs)) return false;
                if (j >= 2 && !mbar_wait_bounded(&bars->s_empty[j & 1], ((j - 2) >> 1) & 1, kWaitNs)) return false;
                tc_fence_after();
                const uint64_t kb = dk + uint64_t((stage * kTile) >> 4);
                const uint32_t d = tbase + kColS + uint32_t(j & 1) * 128u;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t koff = uint64_t(((kk >> 2) * kPanel + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(d, dq + koff, kb + koff, kIdS, kk > 0);
                }
                if constexpr (CL == 1) mma_commit(&bars->k_empty[stage]);
                else mma_commit_multicast(&bars->k_empty[stage], kMask);
                mma_commit(&bars->s_full[j & 1]);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int stage = j % kNS;
                if (!mbar_wait_bounded(&bars->p_full[j & 1], (j >> 1) & 1, kWaitNs)) return false;
                if (!mbar_wait_bounded(&bars->v_full[stage], (j / kNS) & 1, kWaitNs)) return false;
                tc_fence_after();
                const uint64_t vb = dv + uint64_t((stage * kTile) >> 4);
                const uint32_t pcol = tbase + kColP + uint32_t(j & 1) * 64u;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {      // 16 tokens = 8 packed columns of P
                    mma_bf16_ts(tbase + kColO, pcol + kk * 8, vb + uint64_t((kk * 2048) >> 4), kIdO,
                                (j > 0 || kk > 0));
                }
                if constexpr (CL == 1) mma_commit(&bars->v_empty[stage]);
                else mma_commit_multicast(&bars->v_empty[stage], kMask);
                mma_commit(&bars->p_free[j & 1]);
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && ntiles > 1) ok = issue_s(1);
            for (int j = 0; ok && j < ntiles; ++j) {
                if (*abort_flag) { ok = false; break; }
                if (j + 2 < ntiles) ok = issue_s(j + 2);
                if (ok) ok = issue_pv(j);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
            }
            mma_commit(&bars->drain);                        // everything issued above has finished
            mbar_wait_bounded(&bars->drain, 0, kWaitNs);
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
        volatile float* xch = reinterpret_cast<volatile float*>(sm + kOffXch);  // [2 parity][2 half][128 rows]
        volatile int* flags = reinterpret_cast<volatile int*>(sm + kOffFlag);   // [4 quarter][2 half]
        // Swap one float per row with the other half's warp of this quarter: publish the
        // value, then the sequence number; wait (bounded) for the partner's number.  Two
        // parity slots: slot seq&1 is rewritten only after the partner has moved past seq.
        auto exchange = [&](float value, int seq, bool* ok) -> float {
            xch[((seq & 1) * 2 + half) * 128 + t] = value;
            __threadfence_block();
            __syncwarp();
            if (lane == 0) flags[quarter * 2 + half] = seq;
            bool good = true;
            if (lane == 0 && flags[quarter * 2 + (half ^ 1)] < seq) {
                const uint64_t t_start = global_ns();
                while (flags[quarter * 2 + (half ^ 1)] < seq) {
                    if (global_ns() - t_start > kWaitNs) { good = false; break; }
                }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            __threadfence_block();
            *ok = good;
            return xch[((seq & 1) * 2 + (half ^ 1)) * 128 + t];
        };
        {
            const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                               ((size_t(b) * p.N + i) * p.Hq + hq) * kD) + half * 8;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = row_ok ? __ldg(qsrc + c) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(sm + kOffQ + half * kPanel + sw128_offset(t, c)) = v;
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->q_full);

        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;                   // l: this warp's half of the row sum
        bool alive = true;
        for (int j = 0; j < ntiles && alive; ++j) {
            const int base = t0 + j * kBN;
            if (!mbar_wait_bounded(&bars->s_full[j & 1], (j >> 1) & 1, kWaitNs)) { alive = false; break; }
            tc_fence_after();
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
            uint32_t v[kBN / 2];
            if (warp_rows) {
                tmem_ld32(tl + kColS + uint32_t(j & 1) * 128u + half * 64, v);
                tmem_ld32(tl + kColS + uint32_t(j & 1) * 128u + half * 64 + 32, v + 32);
                tmem_wait_ld();
            }
            tc_fence_before();
            mbar_arrive(&bars->s_empty[j & 1]);            // S buffer reusable from here
            constexpr uint32_t kNegInf = 0xff800000u;
            if (!full) {
#pragma unroll
                for (int c = 0; c < kBN / 2; ++c) v[c] = ((mw[c >> 5] >> (c & 31)) & 1u) ? v[c] : kNegInf;
            }
            float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < kBN / 2; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(v[c]));
            float mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
            // the row's max over both halves (identical in the two warps of the quarter)
            bool xok = true;
            mraw = fmaxf(mraw, exchange(mraw, j + 1, &xok));
            if (!xok) { alive = false; break; }
            const float mt = mraw * sc;                    // scale > 0 commutes with max
            bool resc = false;
            float alpha = 1.f;
            if (mt > m_used + 8.f) {
                alpha = ex2(m_used - mt);
                resc = m_used != -INFINITY;
                l *= alpha;
                m_used = mt;
            }
            const float msub = (m_used == -INFINITY) ? 0.f : m_used;
            // probabilities 2^(s*scale - m), rounded to bf16 and packed in pairs in place
            uint32_t* pk = v;
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kBN / 4; ++c) {
                const float p0 = ex2(fmaf(__uint_as_float(v[2 * c]), sc, -msub));
                const float p1 = ex2(fmaf(__uint_as_float(v[2 * c + 1]), sc, -msub));
                pk[c] = pack_bf16x2(p0, p1);
                ls[c & 3] += p0 + p1;
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // P buffer j&1 is free once P_{j-2} V_{j-2} has completed
            if (j >= 2 && !mbar_wait_bounded(&bars->p_free[j & 1], ((j - 2) >> 1) & 1, kWaitNs)) {
                alive = false;
                break;
            }
            if (__any_sync(0xffffffffu, resc)) {
                // O may only be rescaled once P_{j-1} V_{j-1} is in it (this warp's 64 columns)
                if (!mbar_wait_bounded(&bars->p_free[(j - 1) & 1], ((j - 1) >> 1) & 1, kWaitNs)) {
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
            if (warp_rows) tmem_st32(tl + kColP + uint32_t(j & 1) * 64u + half * 32, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_full[j & 1]);
        }
        if (!alive) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        } else if (mbar_wait_bounded(&bars->p_free[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, kWaitNs)) {
            tc_fence_after();
            // the row sum over both halves
            bool xok = true;
            const float lrow = l + exchange(l, ntiles + 1, &xok);
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

int attn_tc_cluster_size(int row_blocks) { return row_blocks % 4 == 0 ? 4 : row_blocks % 2 == 0 ? 2 : 1; }

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
