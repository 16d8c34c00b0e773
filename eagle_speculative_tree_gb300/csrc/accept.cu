// Accept walk over the verified draft tree.
//
// Greedy ("EAGLE-2 & Lookahead Decoding", section 4): a child is accepted iff its token
// is the argmax (lowest id on ties) of the current node's target row; the bonus token
// is the argmax at the node where the walk stops.
//
// Stochastic ("Speculative Decoding in Production: EAGLE-3 Dynamic Trees", section
// "Mathematical Proof of Lossless Speedup", steps 1-3, and "From Linear Sequences to
// Dynamic Draft Trees" for trying the next sibling after a rejection): with
// p = softmax(logits / T) and q the node's draft distribution, children c_1, c_2, ...
// are tested in ascending node index; c_j (token x) is accepted iff r_{j-1}(x) > 0 and
// u_c * q(x) <= r_{j-1}(x), where r_0 = p and r_j = max(0, r_{j-1} - q) / Z_j,
// Z_j = sum_v max(0, r_{j-1}(v) - q(v)) (a zero Z_j leaves r unchanged).  When the
// walk stops at node cur after rejecting k children, the bonus token is the smallest
// v whose running sum of r_k exceeds u_0 * sum(r_k).
//
// Two schedules compute the same result:
//   all rows  -- accept_rows (one CTA per (sequence, node), vocab-parallel) reduces
//                every row up front (argmax; or max, sum of exp and the sibling Z chain),
//                then accept_walk (one CTA per sequence) walks on those scalars and draws
//                the bonus token.  Best when there are few rows (small batch).
//   path only -- walks depth by depth and reduces only the rows it visits, plus one
//                residual pass per rejected sibling that has a successor; it reads about
//                (accepted + 1) rows per sequence instead of N.  accept_cluster (the
//                default for float4 rows up to 131072 tokens) holds a row in the
//                registers of one thread-block cluster per sequence, takes the softmax
//                max and sum in one cluster round, stages the draft row in shared memory
//                at its first pass, and draws the bonus token from float32 prefix sums;
//                accept_path (one CTA per sequence) covers the other shapes.
// The all-rows kernels and accept_path use float4 loads when the vocabulary is a multiple
// of 4, compensated float sums per thread and float64 across threads; their bonus draw
// scans one row with float terms and float64 running sums.
#include <cooperative_groups.h>

#include "common.cuh"

namespace treespec {

namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Ask the L2 for the 128-byte line holding `p` (no data comes back to the thread).
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Softmax probability of one logit, evaluated identically everywhere:
// p = 2^(logit * c - M2) / S with c = log2(e) / T and M2 = max(logit * c).
__device__ __forceinline__ float prob_at(float logit, float c, float M2, float invS) {
    return ex2(fmaf(logit, c, -M2)) * invS;
}

// r_j(v) from p(v), q(v) and 1/Z_1 .. 1/Z_j (0 marks a zero-mass residual, left unchanged).
__device__ __forceinline__ float residual_at(float pv, float qv, const float* izs, int j) {
    float r = pv;
    for (int m = 0; m < j; ++m) {
        const float iz = izs[m];
        if (iz > 0.f) r = fmaxf(r - qv, 0.f) * iz;
    }
    return r;
}

// Neumaier-compensated float accumulation.
struct KSum {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float x) {
        const float t = s + x;
        c += (fabsf(s) >= fabsf(x)) ? ((s - t) + x) : ((x - t) + s);
        s = t;
    }
    __device__ __forceinline__ double value() const { return double(s) + double(c); }
};

// ------------------------------------------------------------ block reductions

template <int NT>
__device__ __forceinline__ double block_sum_d(double v, double* red) {
    v = warp_sum_d(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        double t = lane < NT / 32 ? red[lane] : 0.0;
        t = warp_sum_d(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

template <int NT>
__device__ __forceinline__ float block_sum_f(float v, float* red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < NT / 32 ? red[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

template <int NT>
__device__ __forceinline__ float block_max_f(float v, float* red) {
    v = warp_max(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < NT / 32 ? red[lane] : -INFINITY;
        t = warp_max(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

// ------------------------------------------------------------ row passes

// Visit every element of a row (all NT threads, coalesced; float4 when VEC).
template <int NT, bool VEC, typename F>
__device__ __forceinline__ void for_each(const float* row, int V, F f) {
    if constexpr (VEC) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
        for (int v4 = threadIdx.x; v4 < V / 4; v4 += NT) {
            const float4 x = __ldg(r4 + v4);
            f(4 * v4, x.x);
            f(4 * v4 + 1, x.y);
            f(4 * v4 + 2, x.z);
            f(4 * v4 + 3, x.w);
        }
    } else {
        for (int v = threadIdx.x; v < V; v += NT) f(v, __ldg(row + v));
    }
}

template <int NT, bool VEC, typename F>
__device__ __forceinline__ void for_each_pair(const float* a, const float* b, int V, F f) {
    if constexpr (VEC) {
        const float4* a4 = reinterpret_cast<const float4*>(a);
        const float4* b4 = reinterpret_cast<const float4*>(b);
#pragma unroll 2
        for (int v4 = threadIdx.x; v4 < V / 4; v4 += NT) {
            const float4 x = __ldg(a4 + v4), y = __ldg(b4 + v4);
            f(x.x, y.x);
            f(x.y, y.y);
            f(x.z, y.z);
            f(x.w, y.w);
        }
    } else {
        for (int v = threadIdx.x; v < V; v += NT) f(__ldg(a + v), __ldg(b + v));
    }
}

// Visitors that pass the float4 lane k (0..3) so callers can keep four independent
// accumulators per thread.
template <int NT, bool VEC, typename F>
__device__ __forceinline__ void for_each4(const float* row, int V, F f) {
    if constexpr (VEC) {
        const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 2
        for (int v4 = threadIdx.x; v4 < V / 4; v4 += NT) {
            const float4 x = __ldg(r4 + v4);
            f(0, x.x);
            f(1, x.y);
            f(2, x.z);
            f(3, x.w);
        }
    } else {
        for (int v = threadIdx.x; v < V; v += NT) f(v & 3, __ldg(row + v));
    }
}

template <int NT, bool VEC, typename F>
__device__ __forceinline__ void for_each_pair4(const float* a, const float* b, int V, F f) {
    if constexpr (VEC) {
        const float4* a4 = reinterpret_cast<const float4*>(a);
        const float4* b4 = reinterpret_cast<const float4*>(b);
#pragma unroll 2
        for (int v4 = threadIdx.x; v4 < V / 4; v4 += NT) {
            const float4 x = __ldg(a4 + v4), y = __ldg(b4 + v4);
            f(0, x.x, y.x);
            f(1, x.y, y.y);
            f(2, x.z, y.z);
            f(3, x.w, y.w);
        }
    } else {
        for (int v = threadIdx.x; v < V; v += NT) f(v & 3, __ldg(a + v), __ldg(b + v));
    }
}

// Lowest index of the row maximum (broadcast to every thread).
template <int NT, bool VEC>
__device__ int row_argmax(const float* lg, int V, float* redf, int* redi) {
    float bv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    int bix[4] = {0x7fffffff, 0x7fffffff, 0x7fffffff, 0x7fffffff};
    if constexpr (VEC) {
        const float4* r4 = reinterpret_cast<const float4*>(lg);
#pragma unroll 2
        for (int v4 = threadIdx.x; v4 < V / 4; v4 += NT) {     // ascending v per lane: keeps the first
            const float4 x = __ldg(r4 + v4);
            if (x.x > bv[0]) { bv[0] = x.x; bix[0] = 4 * v4; }
            if (x.y > bv[1]) { bv[1] = x.y; bix[1] = 4 * v4 + 1; }
            if (x.z > bv[2]) { bv[2] = x.z; bix[2] = 4 * v4 + 2; }
            if (x.w > bv[3]) { bv[3] = x.w; bix[3] = 4 * v4 + 3; }
        }
    } else {
        for (int v = threadIdx.x; v < V; v += NT) {
            const float x = __ldg(lg + v);
            if (x > bv[0]) { bv[0] = x; bix[0] = v; }
        }
    }
    float best = bv[0];
    int bi = bix[0];
#pragma unroll
    for (int k = 1; k < 4; ++k)
        if (bv[k] > best || (bv[k] == best && bix[k] < bi)) { best = bv[k]; bi = bix[k]; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) { redf[warp] = best; redi[warp] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < NT / 32; ++w)
            if (redf[w] > best || (redf[w] == best && redi[w] < bi)) { best = redf[w]; bi = redi[w]; }
        redi[0] = bi == 0x7fffffff ? 0 : bi;
    }
    __syncthreads();
    return redi[0];
}

// (M2, S): M2 = max(logits * c), S = sum 2^(logits * c - M2) with c = log2(e) / T
// (broadcast).  Two passes over the row: the second one hits L2.
template <int NT, bool VEC>
__device__ float2 row_softmax_stats(const float* lg, int V, float c, float* redf, double* redd) {
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    for_each4<NT, VEC>(lg, V, [&](int k, float x) { m[k] = fmaxf(m[k], x); });
    const float mx = block_max_f<NT>(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), redf);
    const float M2 = mx * c;                     // c > 0 commutes with max
    KSum s[4];
    for_each4<NT, VEC>(lg, V, [&](int k, float x) { s[k].add(ex2(fmaf(x, c, -M2))); });
    const double S = block_sum_d<NT>((s[0].value() + s[1].value()) + (s[2].value() + s[3].value()), redd);
    return make_float2(M2, float(S));
}

// Z_{j+1} = sum_v max(0, r_j(v) - q(v)) for the row (broadcast).
template <int NT, bool VEC>
__device__ float row_residual_mass(const float* lg, const float* qr, int V, float c, float M2, float invS,
                                   const float* izs, int j, double* redd) {
    KSum z[4];
    for_each_pair4<NT, VEC>(lg, qr, V, [&](int k, float x, float qv) {
        z[k].add(fmaxf(residual_at(prob_at(x, c, M2, invS), qv, izs, j) - qv, 0.f));
    });
    return float(block_sum_d<NT>((z[0].value() + z[1].value()) + (z[2].value() + z[3].value()), redd));
}

// Term of the bonus distribution at token v: r_rej(v) up to normalisation.
struct BonusTerm {
    const float* lg;
    const float* qr;
    const float* izs;
    float c, M2, invS;
    int rej;          // number of rejected children at the final node
    bool unchanged;   // the last residual had zero mass: use r_{rej-1} itself
    __device__ __forceinline__ float operator()(int v) const {
        const float pv = prob_at(__ldg(lg + v), c, M2, invS);
        if (rej == 0) return pv;
        const float qv = __ldg(qr + v);
        const float r = residual_at(pv, qv, izs, rej - 1);
        return unchanged ? r : fmaxf(r - qv, 0.f);
    }
};

__device__ __forceinline__ double warp_inclusive_scan_d(double x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Smallest v with sum_{w <= v} term(w) > u0 * sum_w term(w) (whole CTA; broadcast).
// Pass 1: the warps sum segments of `seg_len` tokens (float64 per segment).  Then warp 0
// scans the segment sums in order to find the segment holding the threshold and scans
// that segment 32 tokens at a time.  A threshold at or above the total (rounding)
// yields the largest token with mass; a residual with no mass falls back to r_{rej-1}.
template <int NT>
__device__ int bonus_scan(BonusTerm term, int V, float u0) {
    constexpr int NW = NT / 32;
    constexpr int kMaxSeg = 2048;
    __shared__ double segsum[kMaxSeg];
    __shared__ int s_state, s_result;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int seg_len = 512;
    while ((V + seg_len - 1) / seg_len > kMaxSeg) seg_len *= 2;
    const int nseg = (V + seg_len - 1) / seg_len;
    for (int attempt = 0; attempt < 2; ++attempt) {
        term.unchanged = attempt == 1;
        for (int sg = warp; sg < nseg; sg += NW) {
            const int a = sg * seg_len, e = min(V, a + seg_len);
            double part = 0.0;
            for (int v = a + lane; v < e; v += 32) part += double(term(v));
            part = warp_sum_d(part);
            if (lane == 0) segsum[sg] = part;
        }
        __syncthreads();
        if (warp == 0) {
            double total = 0.0;
            for (int k0 = 0; k0 < nseg; k0 += 32) total += warp_sum_d(k0 + lane < nseg ? segsum[k0 + lane] : 0.0);
            int state = 1, result = -1;
            if (total > 0.0) {
                const double thr = double(u0) * total;
                double run = 0.0;
                int hit = -1;
                for (int k0 = 0; k0 < nseg && hit < 0; k0 += 32) {
                    const double x = k0 + lane < nseg ? segsum[k0 + lane] : 0.0;
                    const double inc = warp_inclusive_scan_d(x);
                    const unsigned hb = __ballot_sync(0xffffffffu, run + inc > thr);
                    if (hb) {
                        const int l = __ffs(hb) - 1;
                        hit = k0 + l;
                        run += __shfl_sync(0xffffffffu, inc - x, l);
                    } else {
                        run += __shfl_sync(0xffffffffu, inc, 31);
                    }
                }
                if (hit >= 0) {
                    const int a = hit * seg_len, e = min(V, a + seg_len);
                    int last_nz = -1;
                    for (int v0 = a; v0 < e; v0 += 32) {
                        const int v = v0 + lane;
                        const double x = v < e ? double(term(v)) : 0.0;
                        const double inc = warp_inclusive_scan_d(x);
                        const unsigned hb = __ballot_sync(0xffffffffu, run + inc > thr);
                        const unsigned nz = __ballot_sync(0xffffffffu, x > 0.0);
                        if (nz) last_nz = v0 + 31 - __clz(nz);
                        if (hb) { result = v0 + __ffs(hb) - 1; break; }
                        run += __shfl_sync(0xffffffffu, inc, 31);
                    }
                    if (result < 0) result = last_nz;        // rounding between the two passes
                } else {
                    for (int sg = nseg - 1; sg >= 0 && result < 0; --sg) {
                        if (!(segsum[sg] > 0.0)) continue;
                        const int a = sg * seg_len, e = min(V, a + seg_len);
                        int ln = -1;
                        for (int v = a + lane; v < e; v += 32)
                            if (term(v) > 0.f) ln = v;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) ln = max(ln, __shfl_xor_sync(0xffffffffu, ln, o));
                        result = ln;
                    }
                }
            } else if (term.rej > 0 && attempt == 0) {
                state = 2;                                 // zero residual mass: keep r_{rej-1}
            }
            if (lane == 0) {
                s_state = state;
                s_result = result;
            }
        }
        __syncthreads();
        if (s_state != 2) break;
    }
    const int v = s_result;
    __syncthreads();
    return v < 0 ? 0 : v;
}

// Topological parent array, possibly padded with kAbsent after the tree's own nodes (a
// batch may hold trees of different sizes); a padding slot is never anyone's child.
__device__ __forceinline__ uint32_t check_parents(const int* par, int N) {
    uint32_t st = (par[0] != -1) ? TREESPEC_STATUS_BAD_PARENT : 0u;
    bool pad = false;
    for (int c = 1; c < N; ++c) {
        if (par[c] == kAbsent) {
            pad = true;
            continue;
        }
        if (pad || par[c] < 0 || par[c] >= c) st |= TREESPEC_STATUS_BAD_PARENT;
    }
    return st;
}

// The children of every node in ascending index, as the walks test them: kid0[c] is the
// smallest k > c with par[k] == c and sib[c] the smallest k > c with par[k] == par[c]
// (-1: none), so the children of c are kid0[c], sib[kid0[c]], ...  The same nodes a scan
// of par from c + 1 finds, in O(1) per test instead of O(N) for one thread while the CTA
// waits at the next barrier.  Threads c < N of the block, one node each.
__device__ __forceinline__ void child_tables(const int* par, int N, int* kid0, int* sib, int tid, int nt) {
    for (int c = tid; c < N; c += nt) {
        const int pc = par[c];
        int k0 = -1, sb = -1;
        for (int k = c + 1; k < N && (k0 < 0 || sb < 0); ++k) {
            const int pk = par[k];
            if (k0 < 0 && pk == c) k0 = k;
            if (sb < 0 && pk == pc) sb = k;
        }
        kid0[c] = k0;
        sib[c] = sb;
    }
}

// ------------------------------------------------------------ all-rows schedule

template <int NT, bool VEC, bool STOCH>
__global__ void __launch_bounds__(NT) accept_rows_kernel(AcceptParams p) {
    __shared__ double redd[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ float izs[kMaxNodes];
    const int row = blockIdx.x;                 // b * N + i
    const int b = row / p.N, i = row % p.N;
    if (i > 0 && p.parents[row] == kAbsent) return;   // a padding slot's row is never visited
    const float* lg = p.logits + size_t(row) * p.V;
    if constexpr (!STOCH) {
        const int a = row_argmax<NT, VEC>(lg, p.V, redf, redi);
        if (threadIdx.x == 0) p.amax[row] = a;
    } else {
        const float2 st = row_softmax_stats<NT, VEC>(lg, p.V, p.c, redf, redd);
        const float invS = 1.f / st.y;
        if (threadIdx.x == 0) {
            p.stats[size_t(row) * 2] = st.x;
            p.stats[size_t(row) * 2 + 1] = st.y;
        }
        int k = 0;
        for (int c = i + 1; c < p.N; ++c) k += (p.parents[size_t(b) * p.N + c] == i);
        const float* qr = p.probs + size_t(row) * p.V;
        for (int j = 1; j < k; ++j) {                // Z_1 .. Z_{k-1}
            const float Z = row_residual_mass<NT, VEC>(lg, qr, p.V, p.c, st.x, invS, izs, j - 1, redd);
            if (threadIdx.x == 0) {
                const float iz = Z > 0.f ? 1.f / Z : 0.f;
                izs[j - 1] = iz;
                p.izs[size_t(row) * kMaxNodes + (j - 1)] = iz;
            }
            __syncthreads();
        }
    }
}

template <int NT, bool STOCH>
__global__ void __launch_bounds__(NT) accept_walk_kernel(AcceptParams p) {
    __shared__ int par[kMaxNodes], tok[kMaxNodes], path[kMaxNodes];
    __shared__ float izs[kMaxNodes];
    __shared__ int s_cur, s_rej, s_len;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int N = p.N, V = p.V;
    for (int c = tid; c < N; c += NT) {
        par[c] = p.parents[size_t(b) * N + c];
        tok[c] = p.tokens[size_t(b) * N + c];
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t st = check_parents(par, N);
        int cur = 0, len = 0, rej = 0;
        for (;;) {
            const size_t row = size_t(b) * N + cur;
            int accepted = -1, jj = 0;
            float M2 = 0.f, invS = 0.f;
            const float* rz = p.izs + row * kMaxNodes;
            if (STOCH) {
                M2 = p.stats[row * 2];
                invS = 1.f / p.stats[row * 2 + 1];
            }
            for (int c = cur + 1; c < N; ++c) {
                if (par[c] != cur) continue;
                const int x = tok[c];
                const bool valid = x >= 0 && x < V;
                if (!valid) st |= TREESPEC_STATUS_BAD_TOKEN;
                bool ok = false;
                if (valid) {
                    if (!STOCH) {
                        ok = (x == p.amax[row]);
                    } else {
                        const float qx = p.probs[row * V + x];
                        const float r = residual_at(prob_at(p.logits[row * V + x], p.c, M2, invS), qx, rz, jj);
                        ok = r > 0.f && p.uniforms[size_t(b) * N + c] * qx <= r;
                    }
                }
                if (ok) { accepted = c; break; }
                ++jj;
            }
            if (accepted < 0) { rej = jj; break; }
            path[len++] = accepted;
            cur = accepted;
        }
        if (st) atomicOr(p.status, st);
        s_cur = cur;
        s_rej = rej;
        s_len = len;
        if (!STOCH) p.bonus[b] = p.amax[size_t(b) * N + cur];
    }
    __syncthreads();
    for (int c = tid; c < N; c += NT) p.path[size_t(b) * N + c] = c < s_len ? path[c] : -1;
    if (tid == 0) p.len[b] = s_len;
    if constexpr (STOCH) {
        const size_t row = size_t(b) * N + s_cur;
        const int rej = s_rej;
        for (int t = tid; t < kMaxNodes; t += NT) izs[t] = (t < rej) ? p.izs[row * kMaxNodes + t] : 0.f;
        __syncthreads();
        const BonusTerm term{p.logits + row * V, p.probs + row * V, izs, p.c, p.stats[row * 2],
                             1.f / p.stats[row * 2 + 1], rej, false};
        const int v = bonus_scan<NT>(term, V, p.uniforms[size_t(b) * N]);
        if (tid == 0) p.bonus[b] = v;
    }
}

// ------------------------------------------------------------ path-only schedule

template <int NT, bool VEC, bool STOCH>
__global__ void __launch_bounds__(NT) accept_path_kernel(AcceptParams p) {
    __shared__ int par[kMaxNodes], tok[kMaxNodes], path[kMaxNodes];
    __shared__ float izs[kMaxNodes];
    __shared__ double redd[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ int s_cur, s_len, s_action, s_child;
    __shared__ int kid0[kMaxNodes], sib[kMaxNodes];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int N = p.N, V = p.V;
    for (int c = tid; c < N; c += NT) {
        par[c] = p.parents[size_t(b) * N + c];
        tok[c] = p.tokens[size_t(b) * N + c];
    }
    __syncthreads();
    child_tables(par, N, kid0, sib, tid, NT);
    uint32_t st = 0;
    if (tid == 0) {
        st = check_parents(par, N);
        s_cur = 0;
        s_len = 0;
    }
    __syncthreads();
    int amax = 0, rej = 0;
    float M2 = 0.f, invS = 1.f;
    for (int depth = 0; depth < N; ++depth) {
        const int cur = s_cur;
        const size_t row = size_t(b) * N + cur;
        const float* lg = p.logits + row * V;
        const float* qr = STOCH ? p.probs + row * V : nullptr;
        if constexpr (!STOCH) {
            amax = row_argmax<NT, VEC>(lg, V, redf, redi);
        } else {
            const float2 sm = row_softmax_stats<NT, VEC>(lg, V, p.c, redf, redd);
            M2 = sm.x;
            invS = 1.f / sm.y;
        }
        // try the children of cur in ascending node index
        int jj = 0, pos = cur, action = 0, child = -1;
        for (;;) {
            if (tid == 0) {
                const int nc = pos == cur ? kid0[cur] : sib[pos];
                int act = 0;                              // 0: no child left
                if (nc >= 0) {
                    const int x = tok[nc];
                    const bool valid = x >= 0 && x < V;
                    if (!valid) st |= TREESPEC_STATUS_BAD_TOKEN;
                    bool ok = false;
                    if (valid) {
                        if (!STOCH) {
                            ok = x == amax;
                        } else {
                            const float qx = qr[x];
                            const float r = residual_at(prob_at(lg[x], p.c, M2, invS), qx, izs, jj);
                            ok = r > 0.f && p.uniforms[size_t(b) * N + nc] * qx <= r;
                        }
                    }
                    if (ok) {
                        act = 1;                          // accepted
                    } else {
                        const int more = sib[nc];
                        act = more >= 0 ? 2 : 3;          // rejected; 2: a sibling follows
                    }
                }
                s_action = act;
                s_child = nc;
            }
            __syncthreads();
            action = s_action;
            child = s_child;
            __syncthreads();
            if (action == 1 || action == 0) break;
            ++jj;
            if (action == 3) break;
            if constexpr (STOCH) {                        // next sibling sees the residual
                const float Z = row_residual_mass<NT, VEC>(lg, qr, V, p.c, M2, invS, izs, jj - 1, redd);
                if (tid == 0) izs[jj - 1] = Z > 0.f ? 1.f / Z : 0.f;
                __syncthreads();
            }
            pos = child;
        }
        if (action != 1) {
            rej = jj;
            break;
        }
        if (tid == 0) {
            path[s_len] = child;
            s_len = s_len + 1;
            s_cur = child;
        }
        __syncthreads();
    }
    if (tid == 0 && st) atomicOr(p.status, st);
    const int len = s_len;
    for (int c = tid; c < N; c += NT) p.path[size_t(b) * N + c] = c < len ? path[c] : -1;
    if (tid == 0) p.len[b] = len;
    if constexpr (!STOCH) {
        if (tid == 0) p.bonus[b] = amax;
    } else {
        const size_t row = size_t(b) * N + s_cur;
        const BonusTerm term{p.logits + row * V, p.probs + row * V, izs, p.c, M2, invS, rej, false};
        const int v = bonus_scan<NT>(term, V, p.uniforms[size_t(b) * N]);
        if (tid == 0) p.bonus[b] = v;
    }
}

// ------------------------------------------------------------ path-only, one cluster per sequence
//
// The same walk as accept_path_kernel, for large vocabularies: a cluster of CL CTAs
// holds the current row in registers (thread t of CTA k owns tokens
// [k*NT*E + t*E, +E)), so a residual pass is a few register operations per token
// plus one cluster-wide reduction through distributed shared memory.  Every CTA takes
// the same decisions from the same reduced scalars; CTA 0 writes the walk.

namespace cg = cooperative_groups;

template <int CL>
struct ClusterRed {
    float f[2][CL], g[2][CL];
    int i[2][CL];
};

// Cluster-wide reductions: each CTA publishes one value, every CTA combines all CL
// values in rank order (identical result everywhere).  Two alternating slots let a
// slot be rewritten only after the next cluster barrier.
template <int NT, int CL>
struct ClusterReducer {
    ClusterRed<CL>* cr;
    float* redf;
    float* redg;
    int* redi;
    int phase = 0;

    // float sum (partials combined in rank order, so every CTA gets the same value)
    __device__ float sumf(float v) {
        cg::cluster_group cl = cg::this_cluster();
        v = block_sum_f<NT>(v, redf);
        if (threadIdx.x == 0) cr->f[phase][cl.block_rank()] = v;
        cl.sync();
        float t = 0.f;
        for (int k = 0; k < CL; ++k) t += cl.map_shared_rank(cr, k)->f[phase][k];
        phase ^= 1;
        return t;
    }
    __device__ float max(float v) {
        cg::cluster_group cl = cg::this_cluster();
        v = block_max_f<NT>(v, redf);
        if (threadIdx.x == 0) cr->f[phase][cl.block_rank()] = v;
        cl.sync();
        float t = -INFINITY;
        for (int k = 0; k < CL; ++k) t = fmaxf(t, cl.map_shared_rank(cr, k)->f[phase][k]);
        phase ^= 1;
        return t;
    }
    // (value, index): the largest value, lowest index on ties
    __device__ int argmax(float best, int bi) {
        cg::cluster_group cl = cg::this_cluster();
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
        }
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        __syncthreads();
        if (lane == 0) { redf[warp] = best; redi[warp] = bi; }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < NT / 32; ++w)
                if (redf[w] > best || (redf[w] == best && redi[w] < bi)) { best = redf[w]; bi = redi[w]; }
            cr->f[phase][cl.block_rank()] = best;
            cr->i[phase][cl.block_rank()] = bi;
        }
        cl.sync();
        float gb = -INFINITY;
        int gi = 0x7fffffff;
        for (int k = 0; k < CL; ++k) {
            const ClusterRed<CL>* r = cl.map_shared_rank(cr, k);
            const float vb = r->f[phase][k];
            const int vi = r->i[phase][k];
            if (vb > gb || (vb == gb && vi < gi)) { gb = vb; gi = vi; }
        }
        phase ^= 1;
        return gi == 0x7fffffff ? 0 : gi;
    }
    // exclusive prefix (in rank order) of one float per CTA, and the total
    __device__ float exclusive(float v, float* total) {
        cg::cluster_group cl = cg::this_cluster();
        if (threadIdx.x == 0) cr->f[phase][cl.block_rank()] = v;
        cl.sync();
        float pre = 0.f, t = 0.f;
        for (int k = 0; k < CL; ++k) {
            const float x = cl.map_shared_rank(cr, k)->f[phase][k];
            if (k < int(cl.block_rank())) pre += x;
            t += x;
        }
        phase ^= 1;
        *total = t;
        return pre;
    }
    // (max, sum) of softmax partials in one round: every thread brings an integer offset m
    // at or above the max of its values (log2 units; -inf if it has none) and s = sum
    // 2^(x - m); partials combine as M = max(m1, m2) and s1 2^(m1 - M) + s2 2^(m2 - M).  The
    // offsets being integers, the rescales are exact powers of two and only the additions
    // round, as in a plain sum.  Returns (M, S), the same everywhere.
    __device__ float2 maxsum(float m, float s) {
        cg::cluster_group cl = cg::this_cluster();
        auto combine = [](float& m1, float& s1, float m2, float s2) {
            const float M = fmaxf(m1, m2);
            if (M == -INFINITY) return;                        // both empty
            const float a = m1 == -INFINITY ? 0.f : ldexpf(s1, int(m1 - M));
            const float c = m2 == -INFINITY ? 0.f : ldexpf(s2, int(m2 - M));
            s1 = a + c;
            m1 = M;
        };
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
            combine(m, s, m2, s2);
        }
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        __syncthreads();
        if (lane == 0) { redf[warp] = m; redg[warp] = s; }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < NT / 32; ++w) combine(m, s, redf[w], redg[w]);
            cr->f[phase][cl.block_rank()] = m;
            cr->g[phase][cl.block_rank()] = s;
        }
        cl.sync();
        float M = -INFINITY, S = 0.f;
        for (int k = 0; k < CL; ++k) {                         // rank order: identical everywhere
            const ClusterRed<CL>* r = cl.map_shared_rank(cr, k);
            combine(M, S, r->f[phase][k], r->g[phase][k]);
        }
        phase ^= 1;
        return make_float2(M, S);
    }
};

__device__ __forceinline__ float warp_inclusive_scan_f(float x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

template <int CL, int NT, int E, bool STOCH>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 1) accept_cluster_kernel(AcceptParams p) {
    __shared__ int par[kMaxNodes], tok[kMaxNodes], path[kMaxNodes];
    __shared__ float izs[kMaxNodes], uni[kMaxNodes];
    __shared__ float redf[32], redg[32], scan[NT / 32 + 1];
    __shared__ int redi[32];
    __shared__ int s_cur, s_len, s_action, s_child, s_found;
    __shared__ float ch_lg[kMaxNodes], ch_q[kMaxNodes];     // target logit / draft prob of each child's token
    __shared__ int kid0[kMaxNodes], sib[kMaxNodes];
    __shared__ ClusterRed<CL> cred;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int b = blockIdx.y, tid = threadIdx.x;
    const int N = p.N, V = p.V;
    const int lane = tid & 31, warp = tid >> 5;
    // Token layout: warp w of CTA `rank` owns the contiguous range wbase .. wbase + 32 E,
    // and element e of lane l is token wbase + (e / 4) * 128 + 4 l + e % 4: every
    // warp-wide float4 load reads 512 contiguous bytes.
    const int wbase = (rank * (NT / 32) + warp) * 32 * E;
    auto tok_of = [&](int e) { return wbase + (e >> 2) * 128 + lane * 4 + (e & 3); };
    ClusterReducer<NT, CL> red{&cred, redf, redg, redi, 0};

    for (int c = tid; c < N; c += NT) {
        par[c] = p.parents[size_t(b) * N + c];
        tok[c] = p.tokens[size_t(b) * N + c];
        if (STOCH) uni[c] = p.uniforms[size_t(b) * N + c];
    }
    if (tid == 0) {
        s_cur = 0;
        s_len = 0;
    }
    __syncthreads();
    uint32_t st = (tid == 0 && rank == 0) ? check_parents(par, N) : 0u;

    float r[E];
    // The draft row is read only where a child is rejected (and for the bonus draw).  The
    // first pass over it at a node stages this thread's E values in its own slots of shared
    // memory ([E/4][NT] float4, conflict-free), and the later passes (the next siblings'
    // residuals, the deferred rescale, the bonus draw) read them there: no other thread
    // touches those slots, so no barrier is needed, and a row in host memory crosses the
    // link once.
    extern __shared__ float4 qstage[];
    bool q_staged = false;                                  // the current node's row is staged
    auto q_at = [&](const float* q, int e) -> float4 {        // e a multiple of 4
        float4* slot = qstage + (e >> 2) * NT + tid;
        if (q_staged) return *slot;
        const int v = tok_of(e);
        const float4 x = v < V ? __ldg(reinterpret_cast<const float4*>(q + v)) : make_float4(0.f, 0.f, 0.f, 0.f);
        *slot = x;
        return x;
    };
    const float* q_last = nullptr;                          // the draft row of the last visited node
    int amax = 0, rej = 0;
    float M2 = 0.f, invS = 1.f;
    for (int depth = 0; depth < N; ++depth) {
        const int cur = s_cur;
        const size_t row = size_t(b) * N + cur;
        const float* lg = p.logits + row * V;
        const float* qr = STOCH ? p.probs + row * V : nullptr;
        q_last = qr;
        q_staged = false;
        // this warp's draft tokens, into L2 early.  Not over the CPU-GPU link: there the
        // link's rate bounds the walk, and the row is needed only if a child is rejected
        // (the first child is accepted at about half of the levels).
        if (STOCH && !p.probs_on_host) {
#pragma unroll
            for (int m = 0; m < E / 32; ++m) {
                const int v = wbase + (lane + 32 * m) * 32;    // one 128-byte line per lane
                if (v < V) prefetch_line_l2(qr + v);
            }
        }
        if (STOCH) {                                        // what the sibling tests below will need
            for (int c = tid; c < N; c += NT) {
                const int x = tok[c];
                if (par[c] == cur && x >= 0 && x < V) {
                    ch_lg[c] = __ldg(lg + x);
                    ch_q[c] = __ldg(qr + x);
                }
            }
        }
        float piz = 0.f;                                    // a rescale of r still to apply (0: none)
#pragma unroll
        for (int e = 0; e < E; e += 4) {
            const int v = tok_of(e);
            float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (v < V) x = __ldg(reinterpret_cast<const float4*>(lg + v));
            r[e] = x.x; r[e + 1] = x.y; r[e + 2] = x.z; r[e + 3] = x.w;
        }
        if (depth == 0) {                                   // while the root's row is in flight
            child_tables(par, N, kid0, sib, tid, NT);
            __syncthreads();
        }
        if constexpr (!STOCH) {
            float best = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int v = tok_of(e);
                if (v < V && (r[e] > best || (r[e] == best && v < bi))) { best = r[e]; bi = v; }
            }
            amax = red.argmax(best, bi);
        } else {
            // max and sum in one cluster round: each thread's partial sum is taken against
            // an integer offset at or above its own max, the reduction rescales the partials
            // exactly, then p = 2^(x c - M2) / S is formed as prob_at forms it for the child
            // tests (M2 the largest offset: at most one above the row's max)
            float m = -INFINITY;
#pragma unroll
            for (int e = 0; e < E; ++e) m = fmaxf(m, r[e]);
            const float mloc = m == -INFINITY ? -INFINITY : ceilf(m * p.c);   // c > 0 commutes with max
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            if (mloc != -INFINITY) {
#pragma unroll
                for (int e = 0; e < E; ++e) ls[e & 3] += ex2(fmaf(r[e], p.c, -mloc));
            }
            const float2 ms = red.maxsum(mloc, (ls[0] + ls[1]) + (ls[2] + ls[3]));
            M2 = ms.x;
            invS = 1.f / ms.y;
            // r = p (the row's probabilities) is formed only where it is used -- the residual
            // after a rejection and the bonus draw where the walk stops -- not at a node whose
            // child is accepted (the child tests take p of the child's token from its logit)
        }
        bool r_is_p = !STOCH;
        auto form_p = [&]() {
            if (r_is_p) return;
#pragma unroll
            for (int e = 0; e < E; ++e) r[e] = ex2(fmaf(r[e], p.c, -M2)) * invS;   // -inf (padding) -> 0
            r_is_p = true;
        };
        int jj = 0, pos = cur, action = 0, child = -1;
        for (;;) {
            if (tid == 0) {
                const int nc = pos == cur ? kid0[cur] : sib[pos];
                int act = 0;
                if (nc >= 0) {
                    const int x = tok[nc];
                    const bool valid = x >= 0 && x < V;
                    if (!valid && rank == 0) st |= TREESPEC_STATUS_BAD_TOKEN;
                    bool ok = false;
                    if (valid) {
                        if (!STOCH) {
                            ok = x == amax;
                        } else {
                            const float qx = ch_q[nc];
                            const float rx = residual_at(prob_at(ch_lg[nc], p.c, M2, invS), qx, izs, jj);
                            ok = rx > 0.f && uni[nc] * qx <= rx;
                        }
                    }
                    if (ok) {
                        act = 1;
                    } else {
                        const int more = sib[nc];
                        act = more >= 0 ? 2 : 3;
                    }
                }
                s_action = act;
                s_child = nc;
            }
            __syncthreads();
            action = s_action;
            child = s_child;
            __syncthreads();
            if (action == 1 || action == 0) break;
            ++jj;
            if (action == 3) break;
            if constexpr (STOCH) {                          // the next sibling sees the residual
                // the previous sibling's rescale r = max(r - q, 0) / Z is applied here, in the
                // same pass over q as this residual's mass (same operations, one read of q)
                form_p();
                float zs4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < E; e += 4) {
                    const float4 q4 = q_at(qr, e);
                    if (piz > 0.f) {
                        r[e] = fmaxf(r[e] - q4.x, 0.f) * piz;
                        r[e + 1] = fmaxf(r[e + 1] - q4.y, 0.f) * piz;
                        r[e + 2] = fmaxf(r[e + 2] - q4.z, 0.f) * piz;
                        r[e + 3] = fmaxf(r[e + 3] - q4.w, 0.f) * piz;
                    }
                    zs4[0] += fmaxf(r[e] - q4.x, 0.f);
                    zs4[1] += fmaxf(r[e + 1] - q4.y, 0.f);
                    zs4[2] += fmaxf(r[e + 2] - q4.z, 0.f);
                    zs4[3] += fmaxf(r[e + 3] - q4.w, 0.f);
                }
                q_staged = true;
                const float Z = red.sumf((zs4[0] + zs4[1]) + (zs4[2] + zs4[3]));
                const float iz = Z > 0.f ? 1.f / Z : 0.f;
                if (tid == 0) izs[jj - 1] = iz;
                piz = iz;
            }
            pos = child;
        }
        if (action != 1) {
            rej = jj;
            form_p();                                       // the bonus draw reads r
            if (STOCH && piz > 0.f) {                       // the last deferred rescale
#pragma unroll
                for (int e = 0; e < E; e += 4) {
                    const float4 q4 = q_at(qr, e);
                    r[e] = fmaxf(r[e] - q4.x, 0.f) * piz;
                    r[e + 1] = fmaxf(r[e + 1] - q4.y, 0.f) * piz;
                    r[e + 2] = fmaxf(r[e + 2] - q4.z, 0.f) * piz;
                    r[e + 3] = fmaxf(r[e + 3] - q4.w, 0.f) * piz;
                }
                q_staged = true;
            }
            break;
        }
        if (tid == 0) {
            path[s_len] = child;
            s_len = s_len + 1;
            s_cur = child;
        }
        __syncthreads();
    }
    const int len = s_len;
    if (rank == 0) {
        if (tid == 0 && st) atomicOr(p.status, st);
        for (int c = tid; c < N; c += NT) p.path[size_t(b) * N + c] = c < len ? path[c] : -1;
        if (tid == 0) p.len[b] = len;
        if (!STOCH && tid == 0) p.bonus[b] = amax;
    }
    if constexpr (STOCH) {
        // bonus token: inverse CDF of r_rej (up to normalisation) in token order; the weights
        // w = r (no rejection at this node, or zero residual mass) or max(r - q, 0)
        bool unchanged = false;
        auto weight4 = [&](int e) -> float4 {
            if (rej == 0 || unchanged) return make_float4(r[e], r[e + 1], r[e + 2], r[e + 3]);
            const float4 q4 = q_at(q_last, e);
            return make_float4(fmaxf(r[e] - q4.x, 0.f), fmaxf(r[e + 1] - q4.y, 0.f), fmaxf(r[e + 2] - q4.z, 0.f),
                               fmaxf(r[e + 3] - q4.w, 0.f));
        };
        // Sums in float32 (GB300's float64 rate is a small fraction of its float32 rate):
        // each thread's four running sums of at most 16 terms, then trees over the warp, the
        // CTA and the cluster; the crossing warp walks its chunks with a compensated running
        // sum.  Any prefix of the weights is then off by at most about (16 + 5 + 4 + 2 + 6)
        // float32 roundings, 2e-6 of the total -- a tenth of the 2e-5 margin below which a
        // decision counts as a rounding tie.
        float total = 0.f, wsum = 0.f;                        // wsum: this warp's weight
        for (int attempt = 0; attempt < 2; ++attempt) {
            float m4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int e = 0; e < E; e += 4) {
                const float4 w4 = weight4(e);
                m4[0] += w4.x;
                m4[1] += w4.y;
                m4[2] += w4.z;
                m4[3] += w4.w;
            }
            const float lane_sum = (m4[0] + m4[1]) + (m4[2] + m4[3]);
            if (rej > 0 && !unchanged) q_staged = true;       // weight4 read every q slot
            wsum = __shfl_sync(0xffffffffu, warp_sum(lane_sum), 0);
            total = red.sumf(lane_sum);
            if (total > 0.f || rej == 0 || unchanged) break;
            unchanged = true;                                // zero residual mass: keep r_{rej-1}
        }
        // each warp's interval [base, end) of the cumulative weight, in token order: warps of
        // this CTA, then the CTAs of the cluster.  A warp's end is the next warp's base, the
        // same float expression, so the intervals tile the total without rounding gaps.
        if (lane == 0) scan[warp] = wsum;
        __syncthreads();
        float pre_warp = 0.f, pre_next = 0.f, cta_total = 0.f;
        for (int w2 = 0; w2 < NT / 32; ++w2) {
            if (w2 < warp) pre_warp += scan[w2];
            if (w2 <= warp) pre_next += scan[w2];
            cta_total += scan[w2];
        }
        float all = 0.f;
        const float pre_cta = red.exclusive(cta_total, &all);
        const float thr = uni[0] * all;
        const float base = pre_cta + pre_warp;
        const float end = pre_cta + pre_next;
        if (tid == 0 && rank == 0) s_found = 0;
        cluster.sync();
        if (base <= thr && thr < end) {                      // warp-uniform: the crossing is in this warp
            // walk the warp's 128-token chunks in order; in the chunk that crosses, a scan
            // over the lanes' four tokens finds the lane, the lane finds the token
            float run = base, comp = 0.f;                    // compensated running sum
            int v = -1, lnz = -1;
            bool done = false;
#pragma unroll
            for (int e = 0; e < E; e += 4) {
                const float4 w4 = weight4(e);
                const float w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (w[u] > 0.f) lnz = max(lnz, tok_of(e + u));
                if (done) continue;
                const float ls = ((w[0] + w[1]) + w[2]) + w[3];
                const float incl = warp_inclusive_scan_f(ls);
                const float ctot = __shfl_sync(0xffffffffu, incl, 31);
                if (run + ctot > thr) {
                    const unsigned pass = __ballot_sync(0xffffffffu, run + incl > thr);
                    const int L = pass ? __ffs(pass) - 1 : 31;
                    if (lane == L) {
                        float rr = run + (incl - ls);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            rr += w[u];
                            if (v < 0 && rr > thr) v = tok_of(e + u);
                        }
                    }
                    v = __shfl_sync(0xffffffffu, v, L);
                    done = true;
                }
                const float y = ctot - comp, tsum = run + y;
                comp = (tsum - run) - y;
                run = tsum;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lnz = max(lnz, __shfl_xor_sync(0xffffffffu, lnz, o));
            if (lane == 0) {
                p.bonus[b] = v >= 0 ? v : lnz;               // not found: rounding at a boundary
                *cluster.map_shared_rank(&s_found, 0) = 1;
            }
        }
        cluster.sync();
        if (rank == 0 && tid == 0 && s_found == 0) s_found = 2;     // nobody: rounding at the top end
        cluster.sync();
        const int none = *cluster.map_shared_rank(&s_found, 0) == 2;
        if (none) {
            int last_nz = -1;
#pragma unroll
            for (int e = 0; e < E; e += 4) {
                const float4 w4 = weight4(e);
                if (w4.x > 0.f) last_nz = max(last_nz, tok_of(e));
                if (w4.y > 0.f) last_nz = max(last_nz, tok_of(e + 1));
                if (w4.z > 0.f) last_nz = max(last_nz, tok_of(e + 2));
                if (w4.w > 0.f) last_nz = max(last_nz, tok_of(e + 3));
            }
            const int ln = red.argmax(float(last_nz), last_nz);  // largest index with mass
            if (rank == 0 && tid == 0) p.bonus[b] = ln < 0 ? 0 : ln;
        }
    }
    cluster.sync();                      // peers may still read this CTA's shared memory
}

// ------------------------------------------------------------ launches

template <int NT, bool STOCH>
void rows_launch(const AcceptParams& p, cudaStream_t s) {
    const unsigned grid = unsigned(p.B) * unsigned(p.N);
    if (p.V % 4 == 0) accept_rows_kernel<NT, true, STOCH><<<grid, NT, 0, s>>>(p);
    else accept_rows_kernel<NT, false, STOCH><<<grid, NT, 0, s>>>(p);
}

template <int NT, bool STOCH>
void path_launch(const AcceptParams& p, cudaStream_t s) {
    if (p.V % 4 == 0) accept_path_kernel<NT, true, STOCH><<<p.B, NT, 0, s>>>(p);
    else accept_path_kernel<NT, false, STOCH><<<p.B, NT, 0, s>>>(p);
}

// The stochastic walk stages a draft row in NT * E floats of dynamic shared memory.
template <int CL, int NT, int E, bool STOCH>
void cluster_launch(const AcceptParams& p, cudaStream_t s) {
    const int smem = STOCH ? NT * E * int(sizeof(float)) : 0;
    if (STOCH)                                              // per call: the attribute is per device
        cudaFuncSetAttribute(accept_cluster_kernel<CL, NT, E, STOCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    accept_cluster_kernel<CL, NT, E, STOCH><<<dim3(CL, p.B), NT, smem, s>>>(p);
}

template <bool STOCH>
int launch_schedule(const AcceptParams& p, int mode, cudaStream_t s) {
    if (mode == TREESPEC_ACCEPT_PATH_ONLY) {
        const bool vec = p.V % 4 == 0 && p.B <= 65535;
        // A row per cluster, held in registers: clusters of 2 (76 fit on the GPU at once) up
        // to 65,536 tokens, of 4 (36 at once) up to 131,072, with 32 or 64 tokens a thread.
        // Where the batch leaves SMs idle the cluster doubles and each thread holds half as
        // many tokens: the walk of a sequence is a chain of row loads and cluster-wide
        // reductions, and both shorten with more SMs per row.
        const bool wide = (long long)p.B * 8 <= p.sms;
        if (vec && p.V > 16384 && p.V <= 32768) {
            if (wide) cluster_launch<4, 512, 16, STOCH>(p, s);
            else cluster_launch<2, 512, 32, STOCH>(p, s);
            return 1;
        }
        if (vec && p.V > 32768 && p.V <= 65536) {
            if (wide) cluster_launch<4, 512, 32, STOCH>(p, s);
            else cluster_launch<2, 512, 64, STOCH>(p, s);
            return 1;
        }
        if (vec && p.V > 65536 && p.V <= 131072) {
            if (wide) cluster_launch<8, 512, 32, STOCH>(p, s);
            else cluster_launch<4, 512, 64, STOCH>(p, s);
            return 1;
        }
        if (p.V >= 32768) path_launch<512, STOCH>(p, s);
        else if (p.V >= 1024) path_launch<256, STOCH>(p, s);
        else path_launch<32, STOCH>(p, s);
        return 1;
    }
    if (p.V >= 16384) rows_launch<512, STOCH>(p, s);
    else if (p.V >= 2048) rows_launch<256, STOCH>(p, s);
    else if (p.V >= 256) rows_launch<128, STOCH>(p, s);
    else rows_launch<32, STOCH>(p, s);
    if (!STOCH) accept_walk_kernel<32, false><<<p.B, 32, 0, s>>>(p);
    else if (p.V >= 32768) accept_walk_kernel<512, true><<<p.B, 512, 0, s>>>(p);
    else if (p.V >= 1024) accept_walk_kernel<256, true><<<p.B, 256, 0, s>>>(p);
    else accept_walk_kernel<32, true><<<p.B, 32, 0, s>>>(p);
    return 2;
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, int mode, cudaStream_t s, int* kernels) {
    *kernels = p.temperature > 0.f ? launch_schedule<true>(p, mode, s) : launch_schedule<false>(p, mode, s);
    return cudaGetLastError();
}

}  // namespace treespec
