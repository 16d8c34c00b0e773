// Split-KV paged tree attention on the 5th-generation tensor cores, two query tiles
// per CTA (bf16, head_dim 128, an even number of 128-row blocks per kv head).
//
// Same partial state as the other kernels (m, l, acc per query row).  A CTA holds 256
// query rows of one kv head (a "unit": sequence b, kv head h, row-block pair pr) as two
// 128-row query tiles (row r = node i * G + g) and runs over a range of the sequence's
// logical tokens in 64-token KV tiles:
//   * shared memory: Q of both query tiles (written by the softmax warps, 128-byte
//     swizzle), a five-stage K ring (warp 8) and a five-stage V ring (warp 9) filled by
//     TMA one 16-token page x 64 head dims per copy (the page producer shared with the
//     other tensor-core kernels: the partly filled last page of a sequence and pages
//     past the range are written by the producer warp itself, zero-filled);
//   * TMEM (all 512 columns): for each query tile t two 64-column S buffers and O_t;
//     P_t(j) is written over the first 32 columns of S buffer j % 2 as packed bf16;
//   * warp 10 issues the MMAs of query tile 0 and warp 11 those of tile 1, in the order
//     S_t(0), S_t(1), P_t(0) V(0), S_t(2), P_t(1) V(1), ...: S of the next KV tile is
//     computed while the softmax works on the current one, and S_t(j) reuses buffer
//     j % 2 only after P_t(j-2) V(j-2) has completed;
//   * warps 0-3 run the softmax of query tile 0 and warps 4-7 that of tile 1, one query
//     row per thread over all columns of a KV tile (the row maximum needs no exchange
//     between warps).  Per KV tile: read S from TMEM, apply the tree mask -- prefix
//     tokens always, tree token S+j only when bit j of the node's ancestor set holds
//     ("Tech Radar: SGLang EAGLE-2", section 2 mask M and section 5 bitmask) -- take the
//     online softmax in base 2, rescale O in TMEM only when a row's running max grows by
//     more than 2^8 (after P_t(j-1) V(j-1) has completed), and write P back to TMEM.
//
// Two launch forms share this body:
//   * one range per CTA (kStream = false): grid (splits, Hkv * pairs, B), a CTA is one
//     split of one unit; with several splits the partials go to the merge kernel;
//   * persistent (kStream = true): one CTA per SM.  The units' KV tiles, ordered
//     (pr, b, h, tile), are cut into as many equal contiguous ranges as there are CTAs, so
//     every SM gets the same number of tiles whatever the batch (no partly filled last
//     wave), and a CTA walks its range unit by unit without refilling its pipeline.  With
//     pr outermost, the CTAs holding the two row-block pairs of one (b, h) run over the
//     same K/V at about the same time and share it in L2.  A unit cut between CTAs has
//     its head piece (its first tiles) in the last range of CTA c0 and its other pieces
//     in the first (or only) ranges of CTAs c0 + 1 .. c1, which end long before c0's last
//     range.  Those pieces leave their partial (m, l, O) in the CTA's slot and raise the
//     slot's ready flag; at the end of its last range c0 waits (bounded) for the flags and
//     merges the partials into its own O as it writes the rows.  A CTA only ever waits
//     for the first ranges of later CTAs, which wait for nothing before those end, so the
//     waits finish whether or not all CTAs are resident at once.  The softmax warps copy the next
//     unit's Q in (cp.async) while they work on the current unit's last tile, as soon as
//     its S is in TMEM, so the MMA warps compute S of the next unit while O of the
//     current one is read out; P V of the next unit waits for that read (o_free).
// Every mbarrier wait is bounded; on expiry the CTA records TREESPEC_STATUS_TIMEOUT,
// drains its own tensor-core work, frees TMEM and exits.
#include "attn_tc_parts.cuh"

namespace treespec {

namespace {

using namespace sm100;
using tcparts::kD;                   // head dim

constexpr int kM = 128;              // query rows per tile = TMEM lanes
constexpr int kNQ = 2;               // query tiles per CTA
constexpr int kBN = 64;              // tokens per KV tile
constexpr int kNSK = 5;              // K ring stages
constexpr int kNSV = 5;              // V ring stages
constexpr int kQPanel = kM * 128;    // one [128 rows][64 bf16] swizzled panel of Q, bytes
constexpr int kQTile = 2 * kQPanel;  // [128][128] bf16
constexpr int kPanel = kBN * 128;    // one [64 tokens][64 bf16] swizzled panel of K or V
constexpr int kTile = 2 * kPanel;    // [64][128] bf16
constexpr int kThreads = 384;        // 8 softmax warps, K producer, V producer, 2 MMA issuers
constexpr int kWarpK = 8;
constexpr int kWarpV = 9;
constexpr int kWarpMma = 10;         // warps 10 and 11 issue the MMAs of tiles 0 and 1
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;        // S buffer b of tile t: [128 t + 64 b, 128 t + 64 b + 64)
constexpr uint32_t kColO = 256;      // O_t: [256 + 128 t, 256 + 128 t + 128)
// registers per thread: 168 at launch (384 threads); then the producer / issuer
// warpgroup (warps 8-11) drops to 56 and the two softmax warpgroups rise to 200:
// 128 x (200 + 200 + 56) = 58,368 <= 384 x 168 = 64,512
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsOther = 56;
static_assert(128 * (2 * kRegsSoftmax + kRegsOther) <= kThreads * 168, "register split exceeds the launch allocation");

// shared-memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kNQ * kQTile;
constexpr int kOffV = kOffK + kNSK * kTile;
constexpr int kOffBar = kOffV + kNSV * kTile;

struct Bars {
    uint64_t k_full[kNSK], k_empty[kNSK], v_full[kNSV], v_empty[kNSV];
    uint64_t q_full[kNQ], s_full[kNQ][2], p_full[kNQ][2], pv_done[kNQ][2], o_full[kNQ], o_free[kNQ], drain[kNQ];
    uint64_t piece_out[kNQ];          // persistent form: the tile's rows of a piece are in memory
};
constexpr int kOffMisc = kOffBar + int(sizeof(Bars));
// the ancestor sets of one sequence (one range per CTA), or the tile offsets of the
// sequences (persistent form, kStreamMaxBatch + 1 ints)
constexpr int kOffAnc = kOffMisc + 16;
constexpr int kSmemBytes = kOffAnc + kMaxNodes * kAncWords * 8;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert((kStreamMaxBatch + 2) * 4 <= kMaxNodes * kAncWords * 8, "tile offsets fit the ancestor area");

// One contiguous range of KV tiles of one unit that a CTA computes.
struct Seg {
    int b, h, pr;          // sequence, kv head, row-block pair
    int S, nb, L;          // prefix length, tree nodes, logical tokens
    int t0, t1, ntiles;    // logical tokens [t0, t1), in ntiles KV tiles
    int split;             // one range per CTA: the split index
    bool whole;            // the range is the whole unit: final rows, no partials
    int slot;              // persistent form, a piece: this CTA's partial slot
    int ub, ue;            // persistent form: the unit's tiles [ub, ue) in the global order
};

// Persistent form: the unit holding global tile T, ordered (pr, b, h, tile) over the
// sequences' tile offsets tcum[0 .. B]; j0 is T's tile within the unit, n the unit's tiles.
__device__ __forceinline__ void unit_at(int T, const int* tcum, int B, int Hkv, int& pr, int& b, int& h, int& j0,
                                        int& n) {
    const int per_pr = Hkv * tcum[B];
    pr = T / per_pr;
    const int rem = T - pr * per_pr;
    const int x = rem / Hkv;                        // the sequence b has tcum[b] <= x < tcum[b + 1]
    int lo_b = 0, hi_b = B;                         // the last b with tcum[b] <= x
    while (hi_b - lo_b > 1) {
        const int mid = (lo_b + hi_b) >> 1;
        if (tcum[mid] <= x) lo_b = mid;
        else hi_b = mid;
    }
    b = lo_b;
    n = tcum[b + 1] - tcum[b];
    const int off = rem - Hkv * tcum[b];
    h = off / n;
    j0 = off - h * n;
}

// The sequences' tile offsets (an invalid sequence has no tiles, a valid one at least
// one), by one warp; tcum[B + 1] is 1 if some sequence has no tiles.
__device__ __forceinline__ void tile_offsets(const AttnParams& p, int* tcum) {
    const int lane = threadIdx.x & 31;
    int run = 0;
    bool empty = false;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int bb = b0 + lane;
        int n = 0;
        if (bb < p.B) {
            const int S = p.lens[bb];
            if (S >= 0) n = (S + p.nn[bb] + kBN - 1) / kBN;
        }
        empty |= __any_sync(0xffffffffu, bb < p.B && n == 0);
        int inc = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (bb < p.B) tcum[bb] = run + inc - n;
        run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
        tcum[p.B] = run;
        tcum[p.B + 1] = empty ? 1 : 0;
    }
}

// The persistent form's cut: CTA c owns global tiles [lo(c), lo(c + 1)).  The cut is even
// in a weighted position, where each unit costs kCutKappa tiles more than its own tiles
// (about what a piece's epilogue and the restart of the pipeline take), so that a range
// that touches one unit more holds fewer tiles.  The weighted start of tile T of unit
// (pr, b, h), tile j0 of n, is pr WP + Hkv (tcum[b] + k b) + h (k + n) + k + j0, with WP
// the weight of one row-block pair's units.  With a sequence that has no tiles, or ranges
// too short for the weights, the cut is even in tiles (k = 0).  All positions are below
// 2^31 (the host checks the batch's tile count); weighted ones are kept in 64 bits.
constexpr int kCutKappa = 7;
struct Cut {
    long long WP, Wt;      // weight of one pair's units; of all units
    int k;                 // weight of a unit beyond its tiles (0: the plain cut)
};
__device__ __forceinline__ long long cut_wb(const int* tcum, int b, int Hkv, int k) {
    return (long long)Hkv * (tcum[b] + (long long)k * b);
}
__device__ __forceinline__ Cut make_cut(const int* tcum, int B, int Hkv, int pairs, int G) {
    Cut c;
    c.k = tcum[B + 1] ? 0 : kCutKappa;
    c.WP = cut_wb(tcum, B, Hkv, c.k);
    c.Wt = c.WP * pairs;
    if (c.k && c.Wt < (long long)(c.k + 2) * G) {
        c.k = 0;
        c.WP = cut_wb(tcum, B, Hkv, 0);
        c.Wt = c.WP * pairs;
    }
    return c;
}
// lo(c): the first tile whose weighted start is at or past c Wt / G
__device__ __forceinline__ int cut_lo(const Cut& q, const int* tcum, int B, int Hkv, int W, int G, int c) {
    if (c >= G) return W;
    if (q.k == 0) return int((long long)c * W / G);
    const long long X = (long long)c * q.Wt / G;
    const int pr = int(X / q.WP);
    const long long rem = X - pr * q.WP;
    int lo_b = 0, hi_b = B;                         // the last b with cut_wb(b) <= rem
    while (hi_b - lo_b > 1) {
        const int mid = (lo_b + hi_b) >> 1;
        if (cut_wb(tcum, mid, Hkv, q.k) <= rem) lo_b = mid;
        else hi_b = mid;
    }
    const int n = tcum[lo_b + 1] - tcum[lo_b];
    const long long off = rem - cut_wb(tcum, lo_b, Hkv, q.k);
    const int h = int(off / (q.k + n));
    const int x = int(off - (long long)h * (q.k + n));
    return pr * Hkv * tcum[B] + Hkv * tcum[lo_b] + h * n + max(0, x - q.k);
}
// The CTA whose range holds tile T: the largest c with floor(c Wt / G) <= the weighted
// start of T.
__device__ __forceinline__ int cut_owner(const Cut& q, const int* tcum, int B, int Hkv, int W, int G, int T) {
    if (q.k == 0) return int(((long long)(T + 1) * G - 1) / W);
    int pr, b, h, j0, n;
    unit_at(T, tcum, B, Hkv, pr, b, h, j0, n);
    const long long ws = pr * q.WP + cut_wb(tcum, b, Hkv, q.k) + (long long)h * (q.k + n) + q.k + j0;
    return int(((ws + 1) * G - 1) / q.Wt);
}

// Every role of a CTA walks the same ranges in the same order.  A range is named by the
// global position of its first tile (persistent form; 0 for the single range of the other
// form) and its fields are recomputed from that position where they are needed, so that
// no role keeps more than a position or two in registers.
template <bool kStream>
struct SegWalk {
    const AttnParams* p;
    const int* tcum;       // persistent form: [B + 1] exclusive tile offsets of the sequences
    int W, lo, hi;
    int G, c, pairs;

    __device__ int begin() const { return kStream ? lo : 0; }
    __device__ bool more(int T) const { return kStream ? T < hi : T == 0; }

    __device__ void at(int T, Seg& s) const {
        if constexpr (!kStream) {
            s.b = blockIdx.z;
            s.h = blockIdx.y / pairs;
            s.pr = blockIdx.y % pairs;
            s.split = blockIdx.x;
            s.S = p->lens[s.b];
            s.nb = p->nn[s.b];
            s.L = s.S + s.nb;
            s.t0 = s.split * p->split_tokens;
            s.t1 = min(s.L, s.t0 + p->split_tokens);
            s.ntiles = (s.t1 - s.t0 + kBN - 1) / kBN;
            s.whole = !p->merge;
        } else {
            int j0, n;
            unit_at(T, tcum, p->B, p->Hkv, s.pr, s.b, s.h, j0, n);
            const int j1 = min(n, j0 + (hi - T));
            s.S = p->lens[s.b];
            s.nb = p->nn[s.b];
            s.L = s.S + s.nb;
            s.t0 = j0 * kBN;
            s.t1 = min(s.L, j1 * kBN);
            s.ntiles = j1 - j0;
            s.split = 0;
            s.whole = j0 == 0 && j1 == n;
            s.slot = 2 * c + (T == lo ? 0 : 1);
            s.ub = T - j0;
            s.ue = s.ub + n;
        }
    }
};

// Persistent form, one query row of a non-head piece: the partial (O, m, l) into the
// CTA's slot (the slot's flag is raised once all rows of the tile are written).
__device__ __forceinline__ void write_piece(const AttnParams& p, uint32_t ocol, bool warp_rows, int slot, int t,
                                            int row, float m_used, float l) {
    const size_t pr = (size_t(slot) * kNQ + t) * kM + row;
    float4* dst = reinterpret_cast<float4*>(p.part_acc + pr * kD);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (warp_rows) {
            tmem_ld32(ocol + c * 32, o);
            tmem_wait_ld();
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
            __stcg(dst + c * 8 + e, make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                                __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3])));
    }
    __stcg(reinterpret_cast<float2*>(p.part_ml) + pr, make_float2(m_used, l));
}

// Persistent form, one query row of a unit's head piece: its own (O in TMEM, m, l) merged
// with the partials of the unit's other pieces (slot 2c of CTAs c0 + 1 .. c1: their first
// ranges), once their flags are up, as splits merge: M = max m_k, l = sum l_k 2^(m_k - M),
// O = sum O_k 2^(m_k - M); O / l leaves as bf16.  False if a flag did not come up in time.
__device__ __forceinline__ bool merge_head(const AttnParams& p, uint32_t ocol, bool warp_rows, const Seg& s,
                                           const int* tcum, int W, int G, int t, int row, bool row_in, bool row_ok,
                                           int i, int hq, float m_own, float l_own) {
    const Cut q = make_cut(tcum, p.B, p.Hkv, p.row_blocks / kNQ, G);
    const int c0 = cut_owner(q, tcum, p.B, p.Hkv, W, G, s.ub), c1 = cut_owner(q, tcum, p.B, p.Hkv, W, G, s.ue - 1);
    bool ok = true;
    const uint64_t t_start = global_ns();
    for (int c = c0 + 1; c <= c1; ++c) {             // every piece's partial is in memory
        const int* flag = p.stream_flags + 2 * c * kNQ + t;
        int v;
        for (;;) {
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
            if (v != 0) break;
            if (global_ns() - t_start > p.wait_ns) { ok = false; break; }
            __nanosleep(256);
        }
        if (!ok) break;
    }
    const float2* ml2 = reinterpret_cast<const float2*>(p.part_ml);
    float M = m_own;
    for (int c = c0 + 1; ok && c <= c1; ++c) M = fmaxf(M, __ldcg(ml2 + (size_t(2 * c) * kNQ + t) * kM + row).x);
    const float w_own = m_own == -INFINITY ? 0.f : ex2(m_own - M);
    float l = l_own * w_own;
    for (int c = c0 + 1; ok && c <= c1; ++c) {
        const float2 ml = __ldcg(ml2 + (size_t(2 * c) * kNQ + t) * kM + row);
        l += ml.x == -INFINITY ? 0.f : ml.y * ex2(ml.x - M);
    }
    const float inv = 1.f / l;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + ((size_t(s.b) * p.N + i) * p.Hq + hq) * kD);
#pragma unroll 1
    for (int q = 0; q < kD / 32; ++q) {              // 32 columns at a time
        uint32_t o[32];
        if (warp_rows) {
            tmem_ld32(ocol + q * 32, o);
            tmem_wait_ld();
        }
        float acc[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = __uint_as_float(o[e]) * w_own;
        for (int c = c0 + 1; ok && c <= c1; ++c) {
            const size_t pr = (size_t(2 * c) * kNQ + t) * kM + row;
            const float mk = __ldcg(ml2 + pr).x;
            const float w = mk == -INFINITY ? 0.f : ex2(mk - M);
            const float4* src = reinterpret_cast<const float4*>(p.part_acc + pr * kD + q * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float4 x = __ldcg(src + e);
                acc[4 * e] += x.x * w;
                acc[4 * e + 1] += x.y * w;
                acc[4 * e + 2] += x.z * w;
                acc[4 * e + 3] += x.w * w;
            }
        }
        if (!row_in) continue;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint32_t w4[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2)
                w4[k2] = row_ok ? pack_bf16x2(acc[8 * e + 2 * k2] * inv, acc[8 * e + 2 * k2 + 1] * inv) : 0u;
            dst[q * 4 + e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
    }
    return ok;
}

template <bool kStream>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_pair_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ __align__(1024) unsigned char sm[];
    Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    uint64_t* anc_s = reinterpret_cast<uint64_t*>(sm + kOffAnc);
    int* tcum = reinterpret_cast<int*>(sm + kOffAnc);
    grid_dep_wait();                               // the prologue's ancestor words, lengths, counts and flags

    const int pairs = p.row_blocks / kNQ;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (smem_u32(sm) & 1023u) {                    // never expected; refuse rather than misread tiles
        if (tid == 0) atomicOr(p.status, TREESPEC_STATUS_INTERNAL);
        return;
    }

    SegWalk<kStream> walk{};
    walk.p = &p;
    walk.pairs = pairs;
    if constexpr (!kStream) {
        const int b = blockIdx.z, h = blockIdx.y / pairs, pr = blockIdx.y % pairs;
        const int S = p.lens[b];
        if (S < 0) {                               // invalid sequence: zeros (or the merge writes them)
            if (!p.merge && blockIdx.x == 0) tcparts::zero_rows(p, b, h, pr * kNQ * kM, kNQ * kM, kThreads);
            return;
        }
        if (int(blockIdx.x) * p.split_tokens >= S + p.nn[b]) return;
    } else {
        if (warp == 0) tile_offsets(p, tcum);
        __syncthreads();
        walk.tcum = tcum;
        walk.c = blockIdx.x;
        walk.W = pairs * p.Hkv * tcum[p.B];
        // the cut runs over min(CTAs, tiles) CTAs, so that each of them has a tile at least
        // (a unit's pieces are then the CTAs owner(ub) .. owner(ue - 1), all of them)
        walk.G = min(int(gridDim.x), walk.W);
        walk.lo = walk.hi = 0;
        if (walk.c < walk.G) {
            const Cut q = make_cut(tcum, p.B, p.Hkv, pairs, walk.G);
            walk.lo = cut_lo(q, tcum, p.B, p.Hkv, walk.W, walk.G, walk.c);
            walk.hi = cut_lo(q, tcum, p.B, p.Hkv, walk.W, walk.G, walk.c + 1);
        }
        // the units of invalid sequences are zeroed, each by one CTA
        for (int b = 0; b < p.B; ++b) {
            if (tcum[b + 1] != tcum[b]) continue;
            for (int u = 0; u < p.Hkv * pairs; ++u)
                if ((b * p.Hkv * pairs + u) % int(gridDim.x) == walk.c)
                    tcparts::zero_rows(p, b, u / pairs, (u % pairs) * kNQ * kM, kNQ * kM, kThreads);
        }
        if (walk.lo >= walk.hi) return;
    }

    if (tid == 0) {
        for (int s = 0; s < kNSK; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], kNQ);
        }
        for (int s = 0; s < kNSV; ++s) {
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], kNQ);
        }
        for (int t = 0; t < kNQ; ++t) {
            mbar_init(&bars->q_full[t], kM);
            for (int bf = 0; bf < 2; ++bf) {
                mbar_init(&bars->s_full[t][bf], 1);
                mbar_init(&bars->p_full[t][bf], kM);
                mbar_init(&bars->pv_done[t][bf], 1);
            }
            mbar_init(&bars->o_full[t], 1);
            mbar_init(&bars->o_free[t], kM);
            mbar_init(&bars->drain[t], 1);
            mbar_init(&bars->piece_out[t], kM);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (!kStream) {
        const int b = blockIdx.z;
        for (int e = tid; e < p.N * kAncWords; e += kThreads) anc_s[e] = p.anc[size_t(b) * p.N * kAncWords + e];
    }
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);
    Seg sg;
    if (warp >= kWarpK) {
      // one setmaxnreg for the whole warpgroup, then its producer or issuer role
      regs_lower<kRegsOther>();
      if (warp == kWarpK || warp == kWarpV) {
        // ------------------------------------------------------------ TMA producers
        const bool is_v = warp == kWarpV;
        tcparts::ProducerArgs a;
        a.map = is_v ? &tmv : &tmk;
        a.src = static_cast<const uint16_t*>(is_v ? p.v : p.k);
        a.ring = sm + (is_v ? kOffV : kOffK);
        a.full = is_v ? bars->v_full : bars->k_full;
        a.empty = is_v ? bars->v_empty : bars->k_empty;
        a.nst = is_v ? kNSV : kNSK;
        a.stage_bytes = kTile;
        a.panel_bytes = kPanel;
        a.pg0 = 0;
        a.npg = kBN / 16;
        a.dp0 = 0;
        a.ndp = 2;
        int armed = 0;
        for (int T = walk.begin(); walk.more(T); T += sg.ntiles) {
            walk.at(T, sg);
            if (!tcparts::produce_pages<kBN>(p, a, sg.b, sg.h, sg.t0, sg.t1, sg.L, sg.ntiles, armed, abort_flag))
                break;
        }
        tcparts::drain_copies(a, armed);
      } else {
        // ------------------------------------------------------------ MMA issuers
        // Warp 10 + t issues every MMA of tile t.  The whole warp runs the loop (all lanes
        // wait, so control flow stays uniform); one elected lane issues each group and its
        // commits.  g counts the KV tiles over the CTA's life (ring stages, S buffers and
        // their phases); k counts the ranges (Q, O and their phases).
        const int t = warp - kWarpMma;
        auto ready = [&](uint64_t* x, uint32_t px) -> bool {     // polled: its wake-ups are on the critical path
            const uint64_t t0 = global_ns();
            for (;;) {
                if (__all_sync(0xffffffffu, mbar_test_wait(x, px))) return true;
                if (*abort_flag || global_ns() - t0 > p.wait_ns) return false;
            }
        };
        constexpr uint32_t kIdS = idesc_bf16_f32(128, kBN, false);
        constexpr uint32_t kIdO = idesc_bf16_f32(128, 128, true);
        const uint32_t dS = tbase + kColS + uint32_t(t) * 128u;
        const uint32_t dO = tbase + kColO + uint32_t(t) * 128u;
        // a K-step or a stage moves only the start-address field of a descriptor
        // (address >> 4 in the low 14 bits, which no offset in the window overflows)
        const uint64_t dq = smem_desc(sbase + kOffQ + t * kQTile, 16, 1024);
        const uint64_t dk = smem_desc(sbase + kOffK, 16, 1024);
        const uint64_t dv = smem_desc(sbase + kOffV, kPanel, 1024);
        bool ok = true;
        int g = 0, k = 0;
        for (int T = walk.begin(); ok && walk.more(T); T += sg.ntiles, ++k) {
            walk.at(T, sg);
            const int ntiles = sg.ntiles;
            ok = ready(&bars->q_full[t], k & 1);
            for (int j = 0; ok && j <= ntiles; ++j) {
                const int gj = g + j;
                if (j < ntiles) {
                    // S_t(gj) = Q_t K(gj)^T into buffer gj % 2, once K(gj) has landed and
                    // P_t(gj-2) V(gj-2) has read that buffer
                    const int ks = gj % kNSK, bf = gj & 1;
                    ok = ready(&bars->k_full[ks], (gj / kNSK) & 1) &&
                         (gj < 2 || ready(&bars->pv_done[t][bf], ((gj >> 1) - 1) & 1));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t kb = dk + uint64_t((ks * kTile) >> 4);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint64_t qoff = uint64_t(((kk >> 2) * kQPanel + (kk & 3) * 32) >> 4);
                            const uint64_t koff = uint64_t(((kk >> 2) * kPanel + (kk & 3) * 32) >> 4);
                            mma_bf16_ss(dS + bf * 64u, dq + qoff, kb + koff, kIdS, kk > 0);
                        }
                        mma_commit(&bars->k_empty[ks]);
                        mma_commit(&bars->s_full[t][bf]);
                    }
                    __syncwarp();
                }
                if (j > 0) {
                    // O_t += P_t(gp) V(gp): P in the first 32 columns of buffer gp % 2; the
                    // range's first one overwrites O, once the last range's O has been read
                    const int jp = j - 1, gp = gj - 1, vs = gp % kNSV, bf = gp & 1;
                    ok = ready(&bars->p_full[t][bf], (gp >> 1) & 1) && ready(&bars->v_full[vs], (gp / kNSV) & 1) &&
                         (jp > 0 || k == 0 || ready(&bars->o_free[t], (k - 1) & 1));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vb = dv + uint64_t((vs * kTile) >> 4);
                    if (elect_one()) {
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)     // 16 tokens = 8 packed columns of P
                            mma_bf16_ts(dO, dS + bf * 64u + kk * 8, vb + uint64_t((kk * 2048) >> 4), kIdO,
                                        (jp > 0 || kk > 0));
                        mma_commit(&bars->v_empty[vs]);
                        mma_commit(&bars->pv_done[t][bf]);
                        if (jp == ntiles - 1) mma_commit(&bars->o_full[t]);
                    }
                    __syncwarp();
                }
            }
            g += ntiles;
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        }
        if (elect_one()) mma_commit(&bars->drain[t]);      // the pipe completes MMAs in issue order
        __syncwarp();
        mbar_wait_bounded(&bars->drain[t], 0, kDefaultWaitNs);
        __syncwarp();
      }
    } else {
        // ------------------------------------------------------------ softmax warps
        regs_raise<kRegsSoftmax>();
        const int t = warp >> 2;                             // query tile
        const int quarter = warp & 3;                        // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;                 // row in the tile = TMEM lane
        const uint32_t tl = tbase + (uint32_t(quarter * 32) << 16);
        const uint32_t scol0 = tl + kColS + uint32_t(t) * 128u;
        const uint32_t ocol = tl + kColO + uint32_t(t) * 128u;
        const float sc = p.scale_log2;
        bool alive = true;
        uint32_t v[kBN];
        // this thread's query row of a range: its node and query head
        struct RowOf {
            int r, i, hq;
            bool in, ok;
        };
        auto row_of = [&](const Seg& s) -> RowOf {
            RowOf ro;
            ro.r = s.pr * kNQ * kM + t * kM + row;
            ro.in = ro.r < p.R;
            ro.i = ro.in ? ro.r / p.G : 0;
            ro.hq = s.h * p.G + (ro.in ? ro.r % p.G : 0);
            ro.ok = ro.in && ro.i < s.nb;                    // a padding slot's row is not computed
            return ro;
        };
        // What the tile loop of a range needs: its tokens and this row's ancestor-or-self set.
        struct Run {
            int t0, S, t1, ntiles;
            bool ok;
            uint64_t anc0, anc1;
        };
        auto run_of = [&](const Seg& s) -> Run {
            const RowOf ro = row_of(s);
            Run u{s.t0, s.S, s.t1, s.ntiles, ro.ok, 0ull, 0ull};
            if (ro.ok) {
                const uint64_t* ar = kStream ? p.anc + (size_t(s.b) * p.N + ro.i) * kAncWords : anc_s + ro.i * kAncWords;
                u.anc0 = ar[0];
                u.anc1 = ar[1];
            }
            return u;
        };
        // The row of Q of the range at position T into the tile's swizzled shared-memory image
        // (the A operand of S) by cp.async, which needs no registers; finish_q waits for the
        // copies and hands the image to the MMA warp.
        auto issue_q = [&](int T) {
            Seg s;
            walk.at(T, s);
            const RowOf ro = row_of(s);
            const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                               ((size_t(s.b) * p.N + ro.i) * p.Hq + ro.hq) * kD);
            unsigned char* qt = sm + kOffQ + t * kQTile;
#pragma unroll
            for (int ch = 0; ch < kD / 8; ++ch)
                cp_async_16_zfill(qt + (ch >> 3) * kQPanel + sw128_offset(row, ch & 7), ro.ok ? qsrc + ch : p.q,
                                  ro.ok ? 16 : 0);
        };
        auto finish_q = [&]() {
            cp_async_wait_all_groups();
            fence_proxy_async_smem();
            mbar_arrive(&bars->q_full[t]);
        };
        // One KV tile: S from TMEM, the mask, the online softmax, P back to TMEM.  Once S of a
        // range's last tile is in TMEM no S MMA reads Q_t any more: the Q of the range at
        // position tq (if any) is copied in while this tile's softmax runs.  False on a timeout.
        auto tile = [&](const Run& u, bool warp_rows, int j, int gj, float& m_used, float& l, int tq) -> bool {
            const int bf = gj & 1;
            const uint32_t scol = scol0 + bf * 64u;
            uint32_t mw[kBN / 32];
            tcparts::tile_mask<kBN>(mw, u.t0 + j * kBN, u.S, u.t1, u.anc0, u.anc1, u.ok);
            const bool full = __all_sync(0xffffffffu, (mw[0] & mw[1]) == 0xffffffffu);
            if (!mbar_wait_spin(&bars->s_full[t][bf], (gj >> 1) & 1, p.wait_ns)) return false;
            tc_fence_after();
            if (kStream && tq >= 0) issue_q(tq);
            if (warp_rows) {
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) tmem_ld32(scol + c * 32, v + c * 32);
                tmem_wait_ld();
            }
            bool resc = false;
            float alpha = 1.f, ts;
            if (__all_sync(0xffffffffu, tcparts::softmax_tile_fast<kBN>(v, mw, full, sc, m_used, ts))) {
                l += ts;                                     // no row's max moved past m_used + 8
            } else {                                         // S again, and the exact path
                if (warp_rows) {
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c) tmem_ld32(scol + c * 32, v + c * 32);
                    tmem_wait_ld();
                }
                tcparts::softmax_tile<kBN>(v, mw, full, sc, m_used, l, resc, alpha);
            }
            if (warp_rows) tmem_st32(scol, v);               // P over the first 32 columns of the buffer
            tmem_wait_st();
            if (__any_sync(0xffffffffu, resc)) {
                // O_t may be rescaled once P_t(gj-1) V(gj-1) is in it (P_t(gj) V(gj) waits for
                // p_full); never at a range's first tile (m_used was -inf)
                if (!mbar_wait_bounded(&bars->pv_done[t][bf ^ 1], ((gj - 1) >> 1) & 1, p.wait_ns)) return false;
                tc_fence_after();
                tcparts::rescale_o(ocol, resc ? alpha : 1.f);
            }
            tc_fence_before();
            mbar_arrive(&bars->p_full[t][bf]);
            return true;
        };
        if constexpr (!kStream) {
            // one range: Q in, the tiles, the epilogue
            Seg sa;
            walk.at(0, sa);
            const RowOf ra = row_of(sa);
            const Run RA = run_of(sa);
            issue_q(0);
            finish_q();
            float m_used = -INFINITY, l = 0.f;
            const bool wr = __any_sync(0xffffffffu, RA.ok);
            for (int j = 0; alive && j < RA.ntiles; ++j) alive = tile(RA, wr, j, j, m_used, l, -1);
            if (alive && mbar_wait_bounded(&bars->o_full[t], 0, p.wait_ns)) {
                tc_fence_after();
                tcparts::write_row(p, ocol, wr, ra.in, ra.ok, sa.b, ra.i, ra.hq, sa.h, sa.split, ra.r, m_used, l);
            } else {
                alive = false;
            }
        } else {
        // Range A starts at position TA; the next range's Q is copied in during A's last
        // tile and handed over before A's epilogue.
        int TA = walk.begin();
        int head_T = -1;                                     // the head piece to merge after the loop
        float head_m = 0.f, head_l = 0.f;
        Seg sa;
        walk.at(TA, sa);                                     // a CTA that gets here has a range
        Run RA = run_of(sa);
        issue_q(TA);
        finish_q();
        int g = 0;
        for (int k = 0;; ++k) {
            const int TB = TA + RA.ntiles;
            const bool haveB = walk.more(TB);
            float m_used = -INFINITY, l = 0.f;
            {
                const bool wr = __any_sync(0xffffffffu, RA.ok);
                // the last tile apart: only it copies the next range's Q in, so the loop's
                // instance of the tile carries no copy
                for (int j = 0; alive && j + 1 < RA.ntiles; ++j) alive = tile(RA, wr, j, g + j, m_used, l, -1);
                if (alive) alive = tile(RA, wr, RA.ntiles - 1, g + RA.ntiles - 1, m_used, l, haveB ? TB : -1);
            }
            if (!alive) break;
            g += RA.ntiles;
            Run RB{};
            if (haveB) {
                finish_q();                                  // the next range's Q has landed
                Seg sb;
                walk.at(TB, sb);
                RB = run_of(sb);
            }
            if (!mbar_wait_bounded(&bars->o_full[t], k & 1, p.wait_ns)) { alive = false; break; }
            tc_fence_after();
            {
                Seg A;
                walk.at(TA, A);
                const RowOf ra = row_of(A);
                const bool wr = __any_sync(0xffffffffu, ra.ok);
                if (A.whole) {
                    tcparts::write_row(p, ocol, wr, ra.in, ra.ok, A.b, ra.i, ra.hq, A.h, A.split, ra.r, m_used, l);
                } else if (TA == A.ub) {                     // a unit's head piece: the CTA's last range
                    head_m = m_used;
                    head_l = l;
                    head_T = TA;
                    break;
                } else {                                     // another piece: its partial, then its flag
                    write_piece(p, ocol, wr, A.slot, t, row, m_used, l);
                    __threadfence();
                    mbar_arrive(&bars->piece_out[t]);
                    if (row == 0) {                          // a CTA has one such piece at most
                        if (mbar_wait_bounded(&bars->piece_out[t], 0, p.wait_ns)) {
                            __threadfence();
                            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.stream_flags + A.slot * kNQ + t),
                                         "r"(1)
                                         : "memory");
                        } else {
                            alive = false;
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&bars->o_free[t]);
                if (!alive) break;
            }
            if (!haveB) break;
            TA = TB;
            RA = RB;
        }
        if (alive && head_T >= 0) {
            // the unit's head piece, merged with its other pieces as its rows are written
            Seg A;
            walk.at(head_T, A);
            const RowOf ra = row_of(A);
            const bool wr = __any_sync(0xffffffffu, ra.ok);
            alive = merge_head(p, ocol, wr, A, walk.tcum, walk.W, walk.G, t, row, ra.in, ra.ok, ra.i, ra.hq, head_m,
                               head_l);
            tc_fence_before();
            mbar_arrive(&bars->o_free[t]);
        }
        }
        if (!alive) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tbase, kTmemCols);
}

template <bool kStream>
cudaError_t launch_two_tile(const AttnParams& p, cudaStream_t s, dim3 grid) {
    if (p.row_blocks % kNQ != 0 || p.rows_per_block != kM) return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    const long long pool_tokens = (long long)p.num_pool_pages * p.ps;
    if (!make_pool_map(&mk, p.k, p.Hkv, pool_tokens) || !make_pool_map(&mv, p.v, p.Hkv, pool_tokens))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_pair_kernel<kStream>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, attn_tc_pair_kernel<kStream>, p, mk, mv);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc_pair(const AttnParams& p, cudaStream_t s) {
    return launch_two_tile<false>(p, s, dim3(p.num_splits, p.Hkv * (p.row_blocks / kNQ), p.B));
}

cudaError_t launch_attn_tc_stream(const AttnParams& p, cudaStream_t s) {
    if (p.B > kStreamMaxBatch || p.stream_ctas < 1 || p.stream_ctas > kStreamMaxCtas || p.merge)
        return cudaErrorInvalidValue;
    if (!p.stream_flags) return cudaErrorInvalidValue;
    return launch_two_tile<true>(p, s, dim3(p.stream_ctas));
}

}  // namespace treespec
