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
//   path only -- accept_path (one CTA per sequence) walks depth by depth and reduces
//                only the rows it visits, plus one residual pass per rejected sibling
//                that has a successor; it reads about (accepted + 1) rows per sequence
//                instead of N.
// Row passes use float4 loads when the vocabulary is a multiple of 4, compensated
// float sums per thread and float64 across threads; the bonus draw scans one row with
// float terms and float64 running sums.
#include "common.cuh"

namespace treespec {

namespace {

// Softmax probability of one logit, evaluated identically everywhere.
__device__ __forceinline__ float prob_at(float logit, float inv_t, float M, float invS) {
    return expf(fmaf(logit, inv_t, -M)) * invS;
}

// r_j(v) from p(v), q(v) and Z_1..Z_j.
__device__ __forceinline__ float residual_at(float pv, float qv, const float* zs, int j) {
    float r = pv;
    for (int m = 0; m < j; ++m) {
        const float z = zs[m];
        if (z > 0.f) r = fmaxf(r - qv, 0.f) / z;
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

// Lowest index of the row maximum (broadcast to every thread).
template <int NT, bool VEC>
__device__ int row_argmax(const float* lg, int V, float* redf, int* redi) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for_each<NT, VEC>(lg, V, [&](int v, float x) {
        if (x > best) { best = x; bi = v; }           // ascending v per thread: keeps the first
    });
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

// (M, S): M = max(logits / T), S = sum exp(logits / T - M) (broadcast).
template <int NT, bool VEC>
__device__ float2 row_softmax_stats(const float* lg, int V, float inv_t, float* redf, double* redd) {
    float m = -INFINITY;
    KSum s;
    for_each<NT, VEC>(lg, V, [&](int, float x) {
        const float y = x * inv_t;
        if (y > m) {
            const float a = expf(m - y);
            s.s *= a;
            s.c *= a;
            m = y;
        }
        s.add(expf(y - m));
    });
    const float M = block_max_f<NT>(m, redf);
    const double part = (m == -INFINITY) ? 0.0 : s.value() * double(expf(m - M));
    const double S = block_sum_d<NT>(part, redd);
    return make_float2(M, float(S));
}

// Z_{j+1} = sum_v max(0, r_j(v) - q(v)) for the row (broadcast).
template <int NT, bool VEC>
__device__ float row_residual_mass(const float* lg, const float* qr, int V, float inv_t, float M, float invS,
                                   const float* zs, int j, double* redd) {
    KSum z;
    for_each_pair<NT, VEC>(lg, qr, V, [&](float x, float qv) {
        z.add(fmaxf(residual_at(prob_at(x, inv_t, M, invS), qv, zs, j) - qv, 0.f));
    });
    return float(block_sum_d<NT>(z.value(), redd));
}

// Term of the bonus distribution at token v: r_rej(v) up to normalisation.
struct BonusTerm {
    const float* lg;
    const float* qr;
    const float* zs;
    float inv_t, M, invS;
    int rej;          // number of rejected children at the final node
    bool unchanged;   // the last residual had zero mass: use r_{rej-1} itself
    __device__ __forceinline__ float operator()(int v) const {
        const float pv = prob_at(__ldg(lg + v), inv_t, M, invS);
        if (rej == 0) return pv;
        const float qv = __ldg(qr + v);
        const float r = residual_at(pv, qv, zs, rej - 1);
        return unchanged ? r : fmaxf(r - qv, 0.f);
    }
};

// Smallest v with sum_{w <= v} term(w) > u0 * sum_w term(w) (whole CTA; broadcast).
template <int NT>
__device__ int bonus_scan(BonusTerm term, int V, float u0) {
    constexpr int NW = NT / 32;
    __shared__ double segsum[NW];
    __shared__ double s_base, s_thr;
    __shared__ int s_seg, s_found, s_unchanged;
    __shared__ int lastnz[NW];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = ((V + NW - 1) / NW + 31) / 32 * 32;
    const int s0 = warp * seg, s1 = min(V, s0 + seg);
    __syncthreads();
    if (threadIdx.x == 0) s_unchanged = 0;
    __syncthreads();
    for (int attempt = 0; attempt < 2; ++attempt) {
        term.unchanged = s_unchanged != 0;
        double part = 0.0;
        for (int v = s0 + lane; v < s1; v += 32) part += double(term(v));
        part = warp_sum_d(part);
        if (lane == 0) segsum[warp] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
            double total = 0.0;
            for (int w = 0; w < NW; ++w) total += segsum[w];
            s_found = 0;
            if (total > 0.0) {
                const double thr = double(u0) * total;
                double pre = 0.0;
                s_seg = -1;
                for (int w = 0; w < NW; ++w) {
                    if (pre + segsum[w] > thr) { s_seg = w; break; }
                    pre += segsum[w];
                }
                s_base = pre;
                s_thr = thr;
                s_found = 1;
            } else if (term.rej > 0 && !s_unchanged) {
                s_unchanged = 1;          // zero residual mass: the distribution stays r_{rej-1}
                s_found = 2;
            }
        }
        __syncthreads();
        if (s_found != 2) break;
    }
    const int sel = (s_found == 1) ? s_seg : -1;
    if (sel >= 0 && warp == sel) {
        double run = s_base;
        const double thr = s_thr;
        int v_hit = -1, last_nz = -1;
        for (int v0 = s0; v0 < s1; v0 += 32) {
            const int v = v0 + lane;
            const double x = v < s1 ? double(term(v)) : 0.0;
            double inc = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, run + inc > thr);
            const unsigned nz = __ballot_sync(0xffffffffu, x > 0.0);
            if (nz) last_nz = v0 + 31 - __clz(nz);
            if (hit) { v_hit = v0 + __ffs(hit) - 1; break; }
            run += __shfl_sync(0xffffffffu, inc, 31);
        }
        if (v_hit < 0) v_hit = last_nz;        // rounding between the two passes
        if (lane == 0) lastnz[0] = v_hit;
    }
    if (sel < 0) {                             // threshold at or above the total by rounding
        int ln = -1;
        for (int v = s0 + lane; v < s1; v += 32)
            if (term(v) > 0.f) ln = v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ln = max(ln, __shfl_xor_sync(0xffffffffu, ln, o));
        if (lane == 0) lastnz[warp] = ln;
    }
    __syncthreads();
    int v = -1;
    if (sel >= 0) {
        v = lastnz[0];
    } else {
        for (int w = 0; w < NW; ++w) v = max(v, lastnz[w]);
    }
    __syncthreads();
    return v < 0 ? 0 : v;
}

__device__ __forceinline__ uint32_t check_parents(const int* par, int N) {
    uint32_t st = (par[0] != -1) ? TREESPEC_STATUS_BAD_PARENT : 0u;
    for (int c = 1; c < N; ++c)
        if (par[c] < 0 || par[c] >= c) st |= TREESPEC_STATUS_BAD_PARENT;
    return st;
}

// ------------------------------------------------------------ all-rows schedule

template <int NT, bool VEC, bool STOCH>
__global__ void __launch_bounds__(NT) accept_rows_kernel(AcceptParams p) {
    __shared__ double redd[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ float zsm[kMaxNodes];
    const int row = blockIdx.x;                 // b * N + i
    const int b = row / p.N, i = row % p.N;
    const float* lg = p.logits + size_t(row) * p.V;
    if constexpr (!STOCH) {
        const int a = row_argmax<NT, VEC>(lg, p.V, redf, redi);
        if (threadIdx.x == 0) p.amax[row] = a;
    } else {
        const float2 st = row_softmax_stats<NT, VEC>(lg, p.V, p.inv_t, redf, redd);
        const float invS = 1.f / st.y;
        if (threadIdx.x == 0) {
            p.stats[size_t(row) * 2] = st.x;
            p.stats[size_t(row) * 2 + 1] = st.y;
        }
        int k = 0;
        for (int c = i + 1; c < p.N; ++c) k += (p.parents[size_t(b) * p.N + c] == i);
        const float* qr = p.probs + size_t(row) * p.V;
        for (int j = 1; j < k; ++j) {                // Z_1 .. Z_{k-1}
            const float Z = row_residual_mass<NT, VEC>(lg, qr, p.V, p.inv_t, st.x, invS, zsm, j - 1, redd);
            if (threadIdx.x == 0) {
                zsm[j - 1] = Z;
                p.zs[size_t(row) * kMaxNodes + (j - 1)] = Z;
            }
            __syncthreads();
        }
    }
}

template <int NT, bool STOCH>
__global__ void __launch_bounds__(NT) accept_walk_kernel(AcceptParams p) {
    __shared__ int par[kMaxNodes], tok[kMaxNodes], path[kMaxNodes];
    __shared__ float zsm[kMaxNodes];
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
            float M = 0.f, invS = 0.f;
            const float* zs = p.zs + row * kMaxNodes;
            if (STOCH) {
                M = p.stats[row * 2];
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
                        const float r = residual_at(prob_at(p.logits[row * V + x], p.inv_t, M, invS), qx, zs, jj);
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
        for (int t = tid; t < kMaxNodes; t += NT) zsm[t] = (t < rej) ? p.zs[row * kMaxNodes + t] : 0.f;
        __syncthreads();
        const BonusTerm term{p.logits + row * V, p.probs + row * V, zsm, p.inv_t, p.stats[row * 2],
                             1.f / p.stats[row * 2 + 1], rej, false};
        const int v = bonus_scan<NT>(term, V, p.uniforms[size_t(b) * N]);
        if (tid == 0) p.bonus[b] = v;
    }
}

// ------------------------------------------------------------ path-only schedule

template <int NT, bool VEC, bool STOCH>
__global__ void __launch_bounds__(NT) accept_path_kernel(AcceptParams p) {
    __shared__ int par[kMaxNodes], tok[kMaxNodes], path[kMaxNodes];
    __shared__ float zsm[kMaxNodes];
    __shared__ double redd[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ int s_cur, s_len, s_action, s_child;
    const int b = blockIdx.x, tid = threadIdx.x;
    const int N = p.N, V = p.V;
    for (int c = tid; c < N; c += NT) {
        par[c] = p.parents[size_t(b) * N + c];
        tok[c] = p.tokens[size_t(b) * N + c];
    }
    __syncthreads();
    uint32_t st = 0;
    if (tid == 0) {
        st = check_parents(par, N);
        s_cur = 0;
        s_len = 0;
    }
    __syncthreads();
    int amax = 0, rej = 0;
    float M = 0.f, invS = 1.f;
    for (int depth = 0; depth < N; ++depth) {
        const int cur = s_cur;
        const size_t row = size_t(b) * N + cur;
        const float* lg = p.logits + row * V;
        const float* qr = STOCH ? p.probs + row * V : nullptr;
        if constexpr (!STOCH) {
            amax = row_argmax<NT, VEC>(lg, V, redf, redi);
        } else {
            const float2 sm = row_softmax_stats<NT, VEC>(lg, V, p.inv_t, redf, redd);
            M = sm.x;
            invS = 1.f / sm.y;
        }
        // try the children of cur in ascending node index
        int jj = 0, pos = cur, action = 0, child = -1;
        for (;;) {
            if (tid == 0) {
                int nc = -1;
                for (int k = pos + 1; k < N; ++k)
                    if (par[k] == cur) { nc = k; break; }
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
                            const float r = residual_at(prob_at(lg[x], p.inv_t, M, invS), qx, zsm, jj);
                            ok = r > 0.f && p.uniforms[size_t(b) * N + nc] * qx <= r;
                        }
                    }
                    if (ok) {
                        act = 1;                          // accepted
                    } else {
                        int more = -1;
                        for (int k = nc + 1; k < N; ++k)
                            if (par[k] == cur) { more = k; break; }
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
                const float Z = row_residual_mass<NT, VEC>(lg, qr, V, p.inv_t, M, invS, zsm, jj - 1, redd);
                if (tid == 0) zsm[jj - 1] = Z;
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
        const BonusTerm term{p.logits + row * V, p.probs + row * V, zsm, p.inv_t, M, invS, rej, false};
        const int v = bonus_scan<NT>(term, V, p.uniforms[size_t(b) * N]);
        if (tid == 0) p.bonus[b] = v;
    }
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

template <bool STOCH>
int launch_schedule(const AcceptParams& p, int mode, cudaStream_t s) {
    if (mode == TREESPEC_ACCEPT_PATH_ONLY) {
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
