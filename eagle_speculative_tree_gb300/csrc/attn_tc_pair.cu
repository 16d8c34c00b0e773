// Split-KV paged tree attention on the 5th-generation tensor cores, two query tiles
// per CTA (bf16, head_dim 128, an even number of 128-row blocks per kv head).
//
// Same partial state as the other kernels (m, l, acc per query row of one split).  One
// CTA holds 256 query rows of one kv head as two 128-row query tiles (row r = node i * G
// + g) and one split of the sequence's logical tokens, in 64-token KV tiles:
//   * shared memory: Q of both query tiles (written once by the softmax warps, 128-byte
//     swizzle), a five-stage K ring (warp 8) and a five-stage V ring (warp 9) filled by
//     TMA one 16-token page x 64 head dims per copy (the page producer shared with the
//     other tensor-core kernels: the partly filled last page of a sequence and pages
//     past the split are written by the producer warp itself, zero-filled);
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
    uint64_t q_full[kNQ], s_full[kNQ][2], p_full[kNQ][2], pv_done[kNQ][2], o_full[kNQ], drain[kNQ];
};
constexpr int kOffMisc = kOffBar + int(sizeof(Bars));
constexpr int kOffAnc = kOffMisc + 16;
constexpr int kSmemBytes = kOffAnc + kMaxNodes * kAncWords * 8;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_pair_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ __align__(1024) unsigned char sm[];
    Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
    volatile uint32_t* abort_flag = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    uint64_t* anc_s = reinterpret_cast<uint64_t*>(sm + kOffAnc);

    const int pairs = p.row_blocks / kNQ;
    const int split = blockIdx.x;
    const int h = blockIdx.y / pairs, pr = blockIdx.y % pairs;
    const int b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = pr * kNQ * kM;
    const int S = p.lens[b];

    if (S < 0) {                                   // invalid sequence: zeros (or the merge writes them)
        if (!p.merge && split == 0) tcparts::zero_rows(p, b, h, r0, kNQ * kM, kThreads);
        return;
    }
    const int nb = p.nn[b];                        // rows of nodes nb.. are padding: zero output
    const int L = S + nb;
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
            mbar_init(&bars->drain[t], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    for (int e = tid; e < p.N * kAncWords; e += kThreads) anc_s[e] = p.anc[size_t(b) * p.N * kAncWords + e];
    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    const uint32_t sbase = smem_u32(sm);
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
        tcparts::produce_pages<kBN>(p, a, b, h, t0, t1, L, ntiles, abort_flag);
      } else {
        // ------------------------------------------------------------ MMA issuers
        // Warp 10 + t issues every MMA of tile t.  The whole warp runs the loop (all lanes
        // wait, so control flow stays uniform); one elected lane issues each group and its
        // commits.
        const int t = warp - kWarpMma;
        auto ready = [&](uint64_t* x, uint32_t px) -> bool {
            bool r = mbar_try_wait(x, px);
            if (!__all_sync(0xffffffffu, r)) r = !*abort_flag && (r || mbar_wait_bounded(x, px, p.wait_ns));
            return __all_sync(0xffffffffu, r);
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
        bool ok = ready(&bars->q_full[t], 0);
        for (int j = 0; ok && j <= ntiles; ++j) {
            if (j < ntiles) {
                // S_t(j) = Q_t K(j)^T into buffer j % 2, once K(j) has landed and P_t(j-2) V(j-2)
                // has read that buffer
                const int ks = j % kNSK, bf = j & 1;
                ok = ready(&bars->k_full[ks], (j / kNSK) & 1) &&
                     (j < 2 || ready(&bars->pv_done[t][bf], ((j >> 1) - 1) & 1));
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
                // O_t += P_t(j-1) V(j-1): P in the first 32 columns of buffer (j-1) % 2
                const int jp = j - 1, vs = jp % kNSV, bf = jp & 1;
                ok = ready(&bars->p_full[t][bf], (jp >> 1) & 1) && ready(&bars->v_full[vs], (jp / kNSV) & 1);
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
        const int r = r0 + t * kM + row;
        const bool row_in = r < p.R;
        const int i = row_in ? r / p.G : 0;
        const int hq = h * p.G + (row_in ? r % p.G : 0);
        const bool row_ok = row_in && i < nb;                // a padding slot's row is not computed
        const uint64_t anc0 = row_ok ? anc_s[i * kAncWords] : 0ull;     // the node's ancestor-or-self set
        const uint64_t anc1 = row_ok ? anc_s[i * kAncWords + 1] : 0ull;
        const bool warp_rows = __any_sync(0xffffffffu, row_ok);
        const uint32_t tl = tbase + (uint32_t(quarter * 32) << 16);
        const uint32_t scol0 = tl + kColS + uint32_t(t) * 128u;
        const uint32_t ocol = tl + kColO + uint32_t(t) * 128u;
        {
            // this row of Q into the tile's swizzled shared-memory image (the A operand of S)
            const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                               ((size_t(b) * p.N + i) * p.Hq + hq) * kD);
            unsigned char* qt = sm + kOffQ + t * kQTile;
#pragma unroll
            for (int ch = 0; ch < kD / 8; ++ch) {
                const uint4 w = row_ok ? __ldg(qsrc + ch) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(qt + (ch >> 3) * kQPanel + sw128_offset(row, ch & 7)) = w;
            }
            fence_proxy_async_smem();
        }
        mbar_arrive(&bars->q_full[t]);

        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool alive = true;
        uint32_t v[kBN];
        for (int j = 0; j < ntiles; ++j) {
            const int bf = j & 1;
            const uint32_t scol = scol0 + bf * 64u;
            uint32_t mw[kBN / 32];
            tcparts::tile_mask<kBN>(mw, t0 + j * kBN, S, t1, anc0, anc1, row_ok);
            const bool full = __all_sync(0xffffffffu, (mw[0] & mw[1]) == 0xffffffffu);
            if (!mbar_wait_bounded(&bars->s_full[t][bf], (j >> 1) & 1, p.wait_ns)) { alive = false; break; }
            tc_fence_after();
            if (warp_rows) {
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) tmem_ld32(scol + c * 32, v + c * 32);
                tmem_wait_ld();
            }
            bool resc;
            float alpha;
            tcparts::softmax_tile<kBN>(v, mw, full, sc, m_used, l, resc, alpha);
            if (warp_rows) tmem_st32(scol, v);             // P over the first 32 columns of the buffer
            tmem_wait_st();
            if (__any_sync(0xffffffffu, resc)) {
                // O_t may be rescaled once P_t(j-1) V(j-1) is in it (P_t(j) V(j) waits for p_full)
                if (!mbar_wait_bounded(&bars->pv_done[t][bf ^ 1], ((j - 1) >> 1) & 1, p.wait_ns)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                tcparts::rescale_o(ocol, resc ? alpha : 1.f);
            }
            tc_fence_before();
            mbar_arrive(&bars->p_full[t][bf]);
        }
        if (!alive || !mbar_wait_bounded(&bars->o_full[t], 0, p.wait_ns)) {
            *abort_flag = 1;
            atomicOr(p.status, TREESPEC_STATUS_TIMEOUT);
        } else {
            tc_fence_after();
            tcparts::write_row(p, ocol, warp_rows, row_in, row_ok, b, i, hq, h, split, r, m_used, l);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

cudaError_t launch_attn_tc_pair(const AttnParams& p, cudaStream_t s) {
    if (p.row_blocks % kNQ != 0 || p.rows_per_block != kM) return cudaErrorInvalidValue;
    CUtensorMap mk, mv;
    const long long pool_tokens = (long long)p.num_pool_pages * p.ps;
    if (!make_pool_map(&mk, p.k, p.Hkv, pool_tokens) || !make_pool_map(&mv, p.v, p.Hkv, pool_tokens))
        return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(attn_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attn_tc_pair_kernel<<<dim3(p.num_splits, p.Hkv * (p.row_blocks / kNQ), p.B), kThreads, kSmemBytes, s>>>(p, mk,
                                                                                                          mv);
    return cudaGetLastError();
}

}  // namespace treespec
