// Accept walk over the verified draft tree: per-row statistics, then one walk per
// sequence.
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
// Kernel 1 (accept_rows, one CTA per (sequence, node) row, vocab-parallel, float4
// loads): greedy -> the row's argmax; stochastic -> M = max(logits/T),
// S = sum exp(logits/T - M) and Z_1 .. Z_{k-1} for the row's k children (each Z is one
// more vocab pass; r_j(v) is evaluated pointwise from p(v), q(v) and the previous Z's).
// Kernel 2 (accept_walk, one CTA per sequence): thread 0 walks the tree using those
// scalars and two gathered values per tested child; the whole CTA then draws the bonus
// token by an inverse-CDF scan of one row (float32 terms, float64 running sums).
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

template <int NT>
__device__ __forceinline__ double block_sum_d(double v, double* red) {
    v = warp_sum_d(v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (warp == 0) {
        t = lane < NT / 32 ? red[lane] : 0.0;
        t = warp_sum_d(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

template <int NT, bool VEC, bool STOCH>
__global__ void __launch_bounds__(NT) accept_rows_kernel(AcceptParams p) {
    __shared__ double red[32];
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ float zsm[kMaxNodes];
    __shared__ int nkids;
    const int row = blockIdx.x;                 // b * N + i
    const int b = row / p.N, i = row % p.N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* lg = p.logits + size_t(row) * p.V;
    const int V = p.V;

    if constexpr (!STOCH) {
        float best = -INFINITY;
        int bi = 0x7fffffff;
        if constexpr (VEC) {
            const float4* l4 = reinterpret_cast<const float4*>(lg);
            for (int v4 = tid; v4 < V / 4; v4 += NT) {
                const float4 x = __ldg(l4 + v4);
                const int v = v4 * 4;
                if (x.x > best) { best = x.x; bi = v; }
                if (x.y > best) { best = x.y; bi = v + 1; }
                if (x.z > best) { best = x.z; bi = v + 2; }
                if (x.w > best) { best = x.w; bi = v + 3; }
            }
        } else {
            for (int v = tid; v < V; v += NT) {
                const float x = __ldg(lg + v);
                if (x > best) { best = x; bi = v; }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
        }
        if (lane == 0) { redf[warp] = best; redi[warp] = bi; }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < NT / 32; ++w)
                if (redf[w] > best || (redf[w] == best && redi[w] < bi)) { best = redf[w]; bi = redi[w]; }
            p.amax[row] = bi == 0x7fffffff ? 0 : bi;
        }
        return;
    } else {
        // ---- pass 1: online max / sum of exp(logits/T - max)
        const float inv_t = p.inv_t;
        float m = -INFINITY;
        KSum s;
        auto visit = [&](float x) {
            const float y = x * inv_t;
            if (y > m) {
                const float a = expf(m - y);
                s.s *= a;
                s.c *= a;
                m = y;
            }
            s.add(expf(y - m));
        };
        if constexpr (VEC) {
            const float4* l4 = reinterpret_cast<const float4*>(lg);
            for (int v4 = tid; v4 < V / 4; v4 += NT) {
                const float4 x = __ldg(l4 + v4);
                visit(x.x); visit(x.y); visit(x.z); visit(x.w);
            }
        } else {
            for (int v = tid; v < V; v += NT) visit(__ldg(lg + v));
        }
        // block max, then rescale and sum in double
        float bm = warp_max(m);
        if (lane == 0) redf[warp] = bm;
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < NT / 32; ++w) bm = fmaxf(bm, redf[w]);
            redf[0] = bm;
        }
        __syncthreads();
        const float M = redf[0];
        const double part = (m == -INFINITY) ? 0.0 : s.value() * double(expf(m - M));
        const double Sd = block_sum_d<NT>(part, red);
        const float S = float(Sd);
        const float invS = 1.f / S;
        if (tid == 0) {
            p.stats[size_t(row) * 2] = M;
            p.stats[size_t(row) * 2 + 1] = S;
            int k = 0;
            for (int c = i + 1; c < p.N; ++c) k += (p.parents[size_t(b) * p.N + c] == i);
            nkids = k;
        }
        __syncthreads();
        const int k = nkids;
        const float* qr = p.probs + size_t(row) * p.V;
        // ---- passes 2..k: Z_1 .. Z_{k-1}
        for (int j = 1; j < k; ++j) {
            KSum z;
            if constexpr (VEC) {
                const float4* l4 = reinterpret_cast<const float4*>(lg);
                const float4* q4 = reinterpret_cast<const float4*>(qr);
                for (int v4 = tid; v4 < V / 4; v4 += NT) {
                    const float4 x = __ldg(l4 + v4), qv = __ldg(q4 + v4);
                    z.add(fmaxf(residual_at(prob_at(x.x, inv_t, M, invS), qv.x, zsm, j - 1) - qv.x, 0.f));
                    z.add(fmaxf(residual_at(prob_at(x.y, inv_t, M, invS), qv.y, zsm, j - 1) - qv.y, 0.f));
                    z.add(fmaxf(residual_at(prob_at(x.z, inv_t, M, invS), qv.z, zsm, j - 1) - qv.z, 0.f));
                    z.add(fmaxf(residual_at(prob_at(x.w, inv_t, M, invS), qv.w, zsm, j - 1) - qv.w, 0.f));
                }
            } else {
                for (int v = tid; v < V; v += NT) {
                    const float qv = __ldg(qr + v);
                    z.add(fmaxf(residual_at(prob_at(__ldg(lg + v), inv_t, M, invS), qv, zsm, j - 1) - qv, 0.f));
                }
            }
            const double Z = block_sum_d<NT>(z.value(), red);
            if (tid == 0) {
                zsm[j - 1] = float(Z);
                p.zs[size_t(row) * kMaxNodes + (j - 1)] = float(Z);
            }
            __syncthreads();
        }
    }
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

template <int NT, bool STOCH>
__global__ void __launch_bounds__(NT) accept_walk_kernel(AcceptParams p) {
    constexpr int NW = NT / 32;
    __shared__ int par[kMaxNodes], tok[kMaxNodes], path[kMaxNodes];
    __shared__ float zsm[kMaxNodes];
    __shared__ int s_cur, s_rej, s_len, s_seg, s_found, s_unchanged;
    __shared__ double segsum[NW], s_base, s_thr;
    __shared__ int lastnz[NW];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = p.N, V = p.V;
    for (int c = tid; c < N; c += NT) {
        par[c] = p.parents[size_t(b) * N + c];
        tok[c] = p.tokens[size_t(b) * N + c];
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t st = 0;
        if (par[0] != -1) st |= TREESPEC_STATUS_BAD_PARENT;
        for (int c = 1; c < N; ++c)
            if (par[c] < 0 || par[c] >= c) st |= TREESPEC_STATUS_BAD_PARENT;
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
        s_unchanged = 0;
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
        BonusTerm term{p.logits + row * V, p.probs + row * V, zsm, p.inv_t, p.stats[row * 2],
                       1.f / p.stats[row * 2 + 1], rej, false};
        const int seg = ((V + NW - 1) / NW + 31) / 32 * 32;
        const int s0 = warp * seg, s1 = min(V, s0 + seg);
        for (int attempt = 0; attempt < 2; ++attempt) {
            term.unchanged = s_unchanged != 0;
            double part = 0.0;
            for (int v = s0 + lane; v < s1; v += 32) part += double(term(v));
            part = warp_sum_d(part);
            if (lane == 0) segsum[warp] = part;
            __syncthreads();
            if (tid == 0) {
                double total = 0.0;
                for (int w = 0; w < NW; ++w) total += segsum[w];
                s_found = 0;
                if (total > 0.0) {
                    const double thr = double(p.uniforms[size_t(b) * N]) * total;
                    double pre = 0.0;
                    s_seg = -1;
                    for (int w = 0; w < NW; ++w) {
                        if (pre + segsum[w] > thr) { s_seg = w; break; }
                        pre += segsum[w];
                    }
                    s_base = pre;
                    s_thr = thr;
                    s_found = 1;
                } else if (rej > 0 && !s_unchanged) {
                    s_unchanged = 1;          // zero residual mass: the distribution stays r_{rej-1}
                    s_found = 2;
                }
            }
            __syncthreads();
            if (s_found != 2) break;
        }
        // locate the crossing inside the chosen segment
        int v_hit = -1;
        const int sel = (s_found == 1) ? s_seg : -1;
        if (sel >= 0 && warp == sel) {
            double run = s_base;
            const double thr = s_thr;
            int last_nz = -1;
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
        // no crossing anywhere (threshold at or above the total by rounding): the
        // largest token with positive mass
        if (sel < 0) {
            int ln = -1;
            for (int v = s0 + lane; v < s1; v += 32)
                if (term(v) > 0.f) ln = v;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ln = max(ln, __shfl_xor_sync(0xffffffffu, ln, o));
            if (lane == 0) lastnz[warp] = ln;
        }
        __syncthreads();
        if (tid == 0) {
            int v = -1;
            if (sel >= 0) {
                v = lastnz[0];
            } else {
                for (int w = 0; w < NW; ++w) v = max(v, lastnz[w]);
            }
            p.bonus[b] = v < 0 ? 0 : v;
        }
    }
}

template <int NT, bool STOCH>
cudaError_t launch_rows(const AcceptParams& p, cudaStream_t s) {
    const bool vec = (p.V % 4) == 0;
    const unsigned grid = unsigned(p.B) * unsigned(p.N);
    if (vec) accept_rows_kernel<NT, true, STOCH><<<grid, NT, 0, s>>>(p);
    else accept_rows_kernel<NT, false, STOCH><<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

template <bool STOCH>
cudaError_t launch_all(const AcceptParams& p, cudaStream_t s) {
    cudaError_t e;
    if (p.V >= 16384) e = launch_rows<512, STOCH>(p, s);
    else if (p.V >= 2048) e = launch_rows<256, STOCH>(p, s);
    else if (p.V >= 256) e = launch_rows<128, STOCH>(p, s);
    else e = launch_rows<32, STOCH>(p, s);
    if (e != cudaSuccess) return e;
    if (!STOCH) {
        accept_walk_kernel<32, false><<<p.B, 32, 0, s>>>(p);
    } else if (p.V >= 32768) {
        accept_walk_kernel<1024, true><<<p.B, 1024, 0, s>>>(p);
    } else if (p.V >= 1024) {
        accept_walk_kernel<256, true><<<p.B, 256, 0, s>>>(p);
    } else {
        accept_walk_kernel<32, true><<<p.B, 32, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t s) {
    return p.temperature > 0.f ? launch_all<true>(p, s) : launch_all<false>(p, s);
}

}  // namespace treespec
