// Pieces shared by the tensor-core attention kernels (attn_tc.cu, attn_tc_pair.cu): the
// TMA page producer, the tree mask of a 128-token tile, one tile of the online softmax,
// the rescale of O in tensor memory and the epilogue that writes a row block's result.
//
// Layouts they share: a K/V stage holds 128-byte-swizzled panels of 64 head dims (128-byte
// rows, one 16-token page = 16 rows = 2048 bytes of a panel); the query row of a thread
// is its TMEM lane; S, P and O live in tensor memory (P as packed bf16 pairs).
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace treespec {
namespace tcparts {

using namespace sm100;

constexpr int kD = 128;      // head dim
constexpr int kBN = 128;     // tokens per KV tile of the one-tile and CTA-pair kernels (the two-tile kernel: 64)

// ------------------------------------------------------------------ TMA page producer
//
// One warp streams the split's K (or V) pages of sequence b / kv head h into a ring of
// `nst` stages, TILE tokens (TILE / 16 pages) per stage.  This CTA's share of a tile is
// pages [pg0, pg0 + npg) of them and head-dim panels [dp0, dp0 + ndp) of two; stage s starts at ring + s *
// stage_bytes, panel d of it at + d * panel_bytes.  Lanes 0 .. npg-1 own one page each: a
// full page in the pool arrives by TMA (one copy per panel, 2048 bytes), the partly filled
// last page of the sequence, a bad page id (flagged, then zero-filled) and pages past the
// split are written by the warp itself.  A stage is rearmed once `empty` has completed for
// its previous use.  `g` counts the tiles this warp has armed over the CTA's life (stage
// g % nst, its (g / nst)-th use): a CTA that streams several ranges calls this once per
// range and then drain_copies once.  On a timeout or an abort of the CTA the warp stops
// and returns false.
struct ProducerArgs {
    const CUtensorMap* map;
    const uint16_t* src;          // the pool [P][16][Hkv][128] (bf16 bits)
    unsigned char* ring;
    uint64_t* full;               // [nst]: arrive + TMA bytes per use
    uint64_t* empty;              // [nst]
    int nst, stage_bytes, panel_bytes;
    int pg0, npg, dp0, ndp;
};

template <int TILE>
__device__ __forceinline__ bool produce_pages(const AttnParams& p, const ProducerArgs& a, int b, int h, int t0,
                                              int t1, int L, int ntiles, int& g, volatile uint32_t* abort_flag) {
    constexpr int kPPT = TILE / 16;                    // pages per tile
    constexpr int kTPB = 32 / kPPT;                    // tiles per warp-wide page-id load
    const int lane = threadIdx.x & 31;
    const int* ptab = p.page_table + size_t(b) * p.max_pages;
    if (lane == 0) tma_prefetch_desc(a.map);
    // Page ids in batches of kTPB tiles, one warp-wide load each (lane l: page l % kPPT of
    // tile kTPB * batch + l / kPPT), fetched a whole batch ahead: a page-table read that
    // waits behind the K/V traffic in L2 then never holds up the ring.
    auto fetch_batch = [&](int bi) -> int {
        const int jt = kTPB * bi + lane / kPPT;
        const int pos0 = t0 + jt * TILE + (lane % kPPT) * 16;
        return (jt < ntiles && pos0 < t1) ? __ldg(ptab + (pos0 >> 4)) : -1;
    };
    int batch_cur = fetch_batch(0), batch_next = fetch_batch(1);
    for (int j = 0; j < ntiles; ++j, ++g) {
        const int stage = g % a.nst;
        if (j > 0 && (j % kTPB) == 0) {
            batch_cur = batch_next;
            batch_next = fetch_batch(j / kTPB + 1);
        }
        int page = __shfl_sync(0xffffffffu, batch_cur, (j % kTPB) * kPPT + ((a.pg0 + lane) % kPPT));
        const int base = t0 + j * TILE;
        // 1 = full page by TMA, 2 = written here
        const int pos0 = base + (a.pg0 + lane) * 16;
        int kind = 0;
        if (lane < a.npg) {
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
        if (g >= a.nst && !mbar_wait_bounded(&a.empty[stage], ((g / a.nst) - 1) & 1, p.wait_ns)) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
        unsigned char* dst = a.ring + stage * a.stage_bytes;
        const unsigned manual = __ballot_sync(0xffffffffu, kind == 2);
        if (manual) {
            const int nch = 8 * a.ndp;                      // 16-byte chunks of a row this CTA holds
            for (int pg = 0; pg < a.npg; ++pg) {
                if (!((manual >> pg) & 1u)) continue;
                const int pgid = __shfl_sync(0xffffffffu, page, pg);
                const int q0 = base + (a.pg0 + pg) * 16;
                for (int c = lane; c < 16 * nch; c += 32) {  // 16 token rows x nch chunks
                    const int rr = c / nch, cc = c % nch;
                    const int pos = q0 + rr;
                    uint4 val = make_uint4(0, 0, 0, 0);
                    if (pgid >= 0 && pos < t1) {
                        const size_t off = ((size_t(pgid) * p.ps + (pos & 15)) * p.Hkv + h) * kD + (a.dp0 * 8 + cc) * 8;
                        val = __ldg(reinterpret_cast<const uint4*>(a.src + off));
                    }
                    *reinterpret_cast<uint4*>(dst + (cc >> 3) * a.panel_bytes + sw128_offset(pg * 16 + rr, cc & 7)) = val;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        const unsigned viatma = __ballot_sync(0xffffffffu, kind == 1);
        if (lane == 0) mbar_arrive_expect_tx(&a.full[stage], uint32_t(__popc(viatma) * a.ndp) * 2048u);
        __syncwarp();
        if (kind == 1) {                                  // this page's panels
            const int z = page * 16;
            for (int dp = 0; dp < a.ndp; ++dp)
                tma_load_3d(dst + dp * a.panel_bytes + lane * 2048, a.map, 64 * (a.dp0 + dp), h, z, &a.full[stage]);
        }
        __syncwarp();
    }
    return true;
}

// Every copy the warp started (`armed` tiles over the CTA's life) has landed before the
// CTA may end: after an abort the consumers no longer wait for them.  The last phase armed
// on each stage completes once its copies arrive (earlier phases completed before it was
// armed).
__device__ __forceinline__ void drain_copies(const ProducerArgs& a, int armed) {
    for (int s2 = 0; s2 < a.nst && s2 < armed; ++s2) {
        const int last = s2 + ((armed - 1 - s2) / a.nst) * a.nst;
        mbar_wait_bounded(&a.full[s2], uint32_t(last / a.nst) & 1u, kDefaultWaitNs);
    }
}

// ------------------------------------------------------------------ softmax of one tile
//
// Which of the TILE columns of the tile starting at logical token `base` a query row may
// see, as TILE / 32 words: prefix columns below min(S, t1), tree columns [S, t1) when the
// node's ancestor-or-self set {anc0, anc1} holds the column's node ("Tech Radar: SGLang
// EAGLE-2", section 2 mask M and section 5 bitmask).
template <int TILE>
__device__ __forceinline__ void tile_mask(uint32_t (&mw)[TILE / 32], int base, int S, int t1, uint64_t anc0,
                                          uint64_t anc1, bool row_ok) {
    const int pref_end = min(S, t1) - base;
    if (pref_end >= TILE) {                             // a tile of prefix tokens only
#pragma unroll
        for (int w = 0; w < TILE / 32; ++w) mw[w] = row_ok ? 0xffffffffu : 0u;
        return;
    }
    const int tree_lo = S - base, tree_hi = t1 - base;
#pragma unroll
    for (int w = 0; w < TILE / 32; ++w) {
        const int lo = 32 * w;
        const int np = min(max(pref_end - lo, 0), 32);
        uint32_t bits = np == 32 ? 0xffffffffu : ((1u << np) - 1u);
        const int nh = min(max(tree_hi - lo, 0), 32);
        const uint32_t hi_mask = nh == 32 ? 0xffffffffu : ((1u << nh) - 1u);
        const uint32_t tb = anc_bits32(anc0, anc1, lo - tree_lo);   // set bit of column lo: lo - tree_lo
        bits |= tb & hi_mask;
        mw[w] = row_ok ? bits : 0u;
    }
}

// One tile of the online softmax in base 2 for one row: v holds the TILE scores (fp32
// bits) of the tile; columns outside the mask become -inf unless the whole warp sees every
// column (`full`).  The running max m_used moves only when the tile's max exceeds it by
// more than 2^8 (then resc is set and the old O must be scaled by alpha); the
// probabilities 2^(s * sc - m_used), rounded to bf16, leave packed in pairs in
// v[0 .. TILE/2) (pair c overwrites v[c], whose value was read at pair c/2) and add into
// the row sum l.
template <int TILE>
__device__ __forceinline__ void softmax_tile(uint32_t (&v)[TILE], const uint32_t (&mw)[TILE / 32], bool full,
                                             float sc, float& m_used, float& l, bool& resc, float& alpha) {
    if (!full) {
        constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
        for (int c = 0; c < TILE; ++c) v[c] = ((mw[c >> 5] >> (c & 31)) & 1u) ? v[c] : kNegInf;
    }
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < TILE; c += 8) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
            mx[e] = fmax3(mx[e], __uint_as_float(v[c + 2 * e]), __uint_as_float(v[c + 2 * e + 1]));
    }
    const float mt = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * sc;   // scale > 0 commutes with max
    resc = false;
    alpha = 1.f;
    if (mt > m_used + 8.f) {
        alpha = ex2(m_used - mt);
        resc = m_used != -INFINITY;
        l *= alpha;
        m_used = mt;
    }
    const float msub = m_used == -INFINITY ? 0.f : m_used;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int c = 0; c < TILE / 2; ++c) {
        float x0, x1;
        fma_f32x2(x0, x1, __uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]), sc, -msub);
        const float p0 = ex2(x0), p1 = ex2(x1);
        v[c] = pack_bf16x2(p0, p1);
        if (c & 1) add_f32x2(a2, a3, p0, p1);
        else add_f32x2(a0, a1, p0, p1);
    }
    l += (a0 + a1) + (a2 + a3);
}

// The common case of softmax_tile, without the row maximum: P = 2^(s * sc - m_used) against
// the running max in use, and `ts` the tile's sum of P.  The result equals softmax_tile's
// whenever no element of the tile exceeds m_used + 8 (then softmax_tile keeps m_used), and
// a sum of at most 2^8 shows exactly that; false otherwise (also while m_used is -inf and
// the row sees a column), and then v holds partial results: the caller reloads S and calls
// softmax_tile.  Skipping the maximum removes half an instruction per element and the
// maximum -> exponential dependency from nearly every tile.
template <int TILE>
__device__ __forceinline__ bool softmax_tile_fast(uint32_t (&v)[TILE], const uint32_t (&mw)[TILE / 32], bool full,
                                                  float sc, float m_used, float& ts) {
    ts = 0.f;
    if (m_used == -INFINITY) {                          // no column seen yet
        uint32_t seen = 0u;
#pragma unroll
        for (int w = 0; w < TILE / 32; ++w) seen |= mw[w];
        if (seen) return false;                         // the first visible column: the exact path sets the max
#pragma unroll
        for (int c = 0; c < TILE / 2; ++c) v[c] = 0u;   // nothing visible: P = 0
        return true;
    }
    if (!full) {
        constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
        for (int c = 0; c < TILE; ++c) v[c] = ((mw[c >> 5] >> (c & 31)) & 1u) ? v[c] : kNegInf;
    }
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int c = 0; c < TILE / 2; ++c) {
        float x0, x1;
        fma_f32x2(x0, x1, __uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1]), sc, -m_used);
        const float p0 = ex2(x0), p1 = ex2(x1);
        v[c] = pack_bf16x2(p0, p1);
        if (c & 1) add_f32x2(a2, a3, p0, p1);
        else add_f32x2(a0, a1, p0, p1);
    }
    ts = (a0 + a1) + (a2 + a3);
    return ts <= 256.f;                                 // false for inf / NaN too
}

// O (128 fp32 columns of this thread's lane, from `ocol`) *= f; the whole warp takes part.
__device__ __forceinline__ void rescale_o(uint32_t ocol, float f) {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(ocol + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
        tmem_st32(ocol + c * 32, o);
        tmem_wait_st();
    }
}

// ------------------------------------------------------------------ epilogue
//
// Row r of the block (node i, query head hq of kv head h) leaves O / l as bf16 into out,
// or -- when the plan splits the sequence -- O, m and l as float partials for the merge.
// A padding slot's row (row_in && !row_ok) is written as zeros (the merge writes them
// otherwise); rows past R are not written.  The whole warp takes part (TMEM loads).
__device__ __forceinline__ void write_row(const AttnParams& p, uint32_t ocol, bool warp_rows, bool row_in,
                                          bool row_ok, int b, int i, int hq, int h, int split, int r, float m_used,
                                          float l) {
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (warp_rows) {
            tmem_ld32(ocol + c * 32, o);
            tmem_wait_ld();
        }
        const int col0 = c * 32;
        if (!row_ok) {
            if (row_in && !p.merge) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                                      ((size_t(b) * p.N + i) * p.Hq + hq) * kD + col0);
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = make_uint4(0, 0, 0, 0);
            }
            continue;
        }
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
            if (c == 0) {
                p.part_ml[pr * 2] = m_used;
                p.part_ml[pr * 2 + 1] = l;
            }
        }
    }
}

// Zero rows [r0, r0 + rows) of an invalid sequence's output (one split writes them; with
// several the merge does).  All threads of the CTA take part.
__device__ __forceinline__ void zero_rows(const AttnParams& p, int b, int h, int r0, int rows, int nthreads) {
    for (int e = threadIdx.x; e < rows * (kD / 8); e += nthreads) {
        const int row = r0 + e / (kD / 8), c = e % (kD / 8);
        if (row >= p.R) continue;
        const int i = row / p.G, hq = h * p.G + row % p.G;
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + ((size_t(b) * p.N + i) * p.Hq + hq) * kD) + c;
        *dst = make_uint4(0, 0, 0, 0);
    }
}

}  // namespace tcparts
}  // namespace treespec
