// Draft-tree construction: one beam-expansion step (tree_draft_step) and the final
// rerank (tree_rerank, tree_rerank_pool).  Every scored candidate becomes a node; the k
// best of a step form the next frontier; the rerank chooses among all nodes or among a
// given pool of them.
//
// Confidence of a draft path = product of its conditional probabilities ("EAGLE-2 &
// Lookahead Decoding", section 4); in log space a node's score is its parent's score
// plus its log-probability (float32).  Each step branches every frontier node into its
// top-k tokens and keeps the k best candidates; the rerank keeps the root and the
// N - 1 best nodes ("Speculative Decoding" (SGLang), EAGLE decoding: expansion with
// speculative_eagle_topk per step, then rerank to speculative_num_draft_tokens).
// Ties: lower token id within a row, lower candidate index (frontier f, rank r ->
// f * k + r) across a step, lower node index in the rerank.
#include <climits>

#include "common.cuh"

namespace treespec {

namespace {

constexpr int kTopkThreads = 512;

// a ranks before b: larger value, or equal value and smaller index
__device__ __forceinline__ bool before(float av, int at, float bv, int bt) {
    return av > bv || (av == bv && at < bt);
}

// Order-preserving map of a float onto int (for atomicMax on shared memory): x < y iff
// key(x) < key(y), for every float but NaN.
__device__ __forceinline__ int order_key(float x) {
    const int b = __float_as_int(x);
    return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float from_order_key(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// Top-k tokens of one part of a frontier row (a row's vocabulary is cut into p.S parts
// of p.chunk tokens, one CTA each, so that the SMs share every row: one CTA per row left
// most of them idle).  Each warp keeps one sorted list spread over its lanes (lane i
// holds rank i, i < k) and a copy of its k-th entry in every lane; the lanes test their
// elements against that threshold with one ballot, and the rare winners are inserted one
// at a time by shifting the list down a lane.  (With a private list per thread, some
// lane of a warp inserts at almost every element and the warp runs the insertion nearly
// always.)  The warps also share a floor in shared memory, below which no element can be
// in the row's top k: the largest of their lists' k-th values (that warp's k entries beat
// anything below it), and at the start the k-th largest of each warp's lane maxima over
// its first batch (k distinct elements are at or above it).  Elements equal to the floor
// are still looked at (their token decides).  Without the seed a warp's first batch met
// an empty list and all 32 lanes' elements went in one by one.  At the end the CTA ranks
// the list entries at or above the floor.
template <bool VEC>
__global__ void __launch_bounds__(kTopkThreads) draft_topk_kernel(const DraftParams p) {
    constexpr int kWarps = kTopkThreads / 32;
    __shared__ float sv[kWarps * kMaxTopk];
    __shared__ int st[kWarps * kMaxTopk];
    __shared__ int floor_key;                            // order_key of the warps' largest k-th value
    __shared__ int n_cand;
    grid_dep_release();                                   // the select kernel may launch; it waits for this grid
    const int row = blockIdx.x / p.S, part = blockIdx.x % p.S;   // row = b * F + f
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0 && tid == 0) *p.status = 0;       // only the select kernel after this grid sets bits
    const int k = p.k;
    const int v_lo = part * p.chunk, v_hi = min(p.V, v_lo + p.chunk);
    const float* lp = p.logprobs + size_t(row) * p.V;
    float wv = -INFINITY, tv = -INFINITY;                // this lane's list entry; the warp's k-th entry
    int wt = INT_MAX, tt = INT_MAX;
    if (tid == 0) floor_key = order_key(-INFINITY);
    __syncthreads();
    float fl = -INFINITY;                                 // this warp's last look at the floor
    auto look = [&]() {                                   // publish this warp's k-th value, read the floor
        if (tv > fl) {
            if (lane == 0) atomicMax(&floor_key, order_key(tv));
            fl = tv;
        }
        fl = fmaxf(fl, from_order_key(*reinterpret_cast<volatile int*>(&floor_key)));
    };
    // The k-th largest of the lanes' maxima over a batch (a bitonic sort across the warp,
    // largest first): k distinct elements are at or above it, so it is a floor too.
    // Without it a warp's first batch meets an empty list, every lane wins the ballot,
    // and the winners go in one at a time.
    auto seed = [&](float lm) {
#pragma unroll
        for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                const float o = __shfl_xor_sync(0xffffffffu, lm, stride);
                const bool keep_max = ((lane & size) == 0) == ((lane & stride) == 0);
                lm = keep_max ? fmaxf(lm, o) : fminf(lm, o);
            }
        }
        const float kth = __shfl_sync(0xffffffffu, lm, k - 1);
        if (kth > fl) {
            if (lane == 0) atomicMax(&floor_key, order_key(kth));
            fl = kth;
        }
    };
    auto consider = [&](float x, int t) {                 // called by all lanes together
        unsigned m = __ballot_sync(0xffffffffu, x >= fl && before(x, t, tv, tt));
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const float nv = __shfl_sync(0xffffffffu, x, src);
            const int nt = __shfl_sync(0xffffffffu, t, src);
            if (!before(nv, nt, tv, tt)) continue;        // displaced by an earlier winner of this round
            const float uv = __shfl_up_sync(0xffffffffu, wv, 1);
            const int ut = __shfl_up_sync(0xffffffffu, wt, 1);
            const bool from_above = lane > 0 && before(nv, nt, uv, ut);
            const bool take_new = before(nv, nt, wv, wt);
            if (lane < k) {
                if (from_above) {
                    wv = uv;
                    wt = ut;
                } else if (take_new) {
                    wv = nv;
                    wt = nt;
                }
            }
            tv = __shfl_sync(0xffffffffu, wv, k - 1);
            tt = __shfl_sync(0xffffffffu, wt, k - 1);
        }
    };
    // eight independent loads per lane in flight before they are consumed (four left a
    // CTA latency-bound at about 10 GB/s)
    constexpr int kU = 8;
    if constexpr (VEC) {                                  // p.chunk is a multiple of 4
        bool first = true;
        for (int v0 = v_lo; v0 < v_hi; v0 += kTopkThreads * 4 * kU) {
            float4 x[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int v = v0 + (u * kTopkThreads + tid) * 4;
                x[u] = v < v_hi ? __ldg(reinterpret_cast<const float4*>(lp + v))
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
            if (first) {                                  // the warp's first batch seeds the floor
                float lm = -INFINITY;
#pragma unroll
                for (int u = 0; u < kU; ++u) lm = fmaxf(lm, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)));
                seed(lm);
                first = false;
            }
            look();
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                // one vote per float4: only a group holding a value at or above the warp's
                // k-th entry can change the list (exact: a tie needs the token test below)
                const float m4 = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
                if (!__any_sync(0xffffffffu, m4 >= fmaxf(tv, fl))) continue;
                const int v = v0 + (u * kTopkThreads + tid) * 4;
                const bool in = v < v_hi;
                consider(x[u].x, in ? v : INT_MAX);
                consider(x[u].y, in ? v + 1 : INT_MAX);
                consider(x[u].z, in ? v + 2 : INT_MAX);
                consider(x[u].w, in ? v + 3 : INT_MAX);
            }
        }
    } else {
        bool first = true;
        for (int v0 = v_lo; v0 < v_hi; v0 += kTopkThreads * kU) {
            float x[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int v = v0 + u * kTopkThreads + tid;
                x[u] = v < v_hi ? __ldg(lp + v) : -INFINITY;
            }
            if (first) {
                float lm = -INFINITY;
#pragma unroll
                for (int u = 0; u < kU; ++u) lm = fmaxf(lm, x[u]);
                seed(lm);
                first = false;
            }
            look();
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int v = v0 + u * kTopkThreads + tid;
                consider(x[u], v < v_hi ? v : INT_MAX);
            }
        }
    }
    // The part's top k are among the list entries at or above the final floor (an entry
    // below it has the k entries of the floor's warp ahead of it): gather those, then rank
    // each against the others, all threads at once.  Ranks break equal (value, token)
    // pairs -- only the (-inf, INT_MAX) fillers of a part shorter than k -- by slot.
    look();
    __syncthreads();
    const float fin = from_order_key(floor_key);
    if (tid == 0) n_cand = 0;
    __syncthreads();
    if (lane < k && wv >= fin) {
        const int c = atomicAdd(&n_cand, 1);
        sv[c] = wv;
        st[c] = wt;
    }
    __syncthreads();
    const int n = n_cand;
    for (int c = tid; c < n; c += kTopkThreads) {
        const float cv = sv[c];
        const int ct = st[c];
        int rank = 0;
        for (int o = 0; o < n; ++o) {
            const float ov = sv[o];
            const int ot = st[o];
            rank += (before(ov, ot, cv, ct) || (ov == cv && ot == ct && o < c)) ? 1 : 0;
        }
        if (rank < k) {
            p.tk_tok[size_t(blockIdx.x) * k + rank] = ct;
            p.tk_lp[size_t(blockIdx.x) * k + rank] = cv;
        }
    }
}

// One CTA per sequence.  First each frontier row's top k out of the S partial lists of
// its parts (ties: lower token id); then the F * k candidates become nodes base + (f * k
// + r), and the k best of them (ties: lower candidate index) the next frontier, best first.
constexpr int kSelectThreads = 256;
__global__ void __launch_bounds__(kSelectThreads) draft_select_kernel(const DraftParams p) {
    __shared__ float cs[kMaxFrontier * kMaxTopk];
    __shared__ float mv[kMaxFrontier * kMaxTopk];
    __shared__ int mt[kMaxFrontier * kMaxTopk];
    grid_dep_wait();                                      // every part's list, and the cleared status word
    const int b = blockIdx.x, tid = threadIdx.x;
    const int k = p.k, F = p.F, S = p.S, nc = F * k;
    int* par = p.node_parent + size_t(b) * p.M;
    int* tok = p.node_token + size_t(b) * p.M;
    float* sc = p.node_score + size_t(b) * p.M;
    const int base = p.step == 0 ? 1 : 1 + k + (p.step - 1) * k * k;
    // merge: entry e = (f, part, r) of the F * S * k partial entries takes its rank within row f
    const size_t e0 = size_t(b) * F * S * k;
    for (int e = tid; e < F * S * k; e += kSelectThreads) {
        const int f = e / (S * k);
        const float ev = p.tk_lp[e0 + e];
        const int et = p.tk_tok[e0 + e];
        int rank = 0;
#pragma unroll 8
        for (int o = f * S * k; o < (f + 1) * S * k; ++o) rank += before(p.tk_lp[e0 + o], p.tk_tok[e0 + o], ev, et) ? 1 : 0;
        if (rank < k) {
            mv[f * k + rank] = ev;
            mt[f * k + rank] = et;
            if (et == INT_MAX) atomicOr(p.status, TREESPEC_STATUS_BAD_TOKEN);   // fewer than k usable values
        }
    }
    __syncthreads();
    for (int c = tid; c < nc; c += kSelectThreads) {
        const int f = c / k;
        const int node = p.step == 0 ? 0 : p.frontier_in[size_t(b) * F + f];
        const float parent_score = p.step == 0 ? 0.f : sc[node];
        const float score = parent_score + mv[c];
        cs[c] = score;
        par[base + c] = node;
        tok[base + c] = mt[c];
        sc[base + c] = score;
    }
    __syncthreads();
    for (int c = tid; c < nc; c += kSelectThreads) {
        int rank = 0;
        const float cc = cs[c];
#pragma unroll 8
        for (int o = 0; o < nc; ++o) rank += before(cs[o], o, cc, c) ? 1 : 0;
        if (rank < k) p.frontier_out[size_t(b) * k + rank] = base + c;
    }
    if (p.step == 0 && tid == 0) {
        par[0] = -1;
        tok[0] = -1;
        sc[0] = 0.f;
    }
}

// One CTA per sequence: keep the root and the N - 1 best eligible nodes (every node, or
// the pool's), numbered by original index, parents remapped; a pool with fewer eligible
// nodes leaves the rest of the row as padding (parent kAbsent, token -1).
constexpr int kRerankThreads = 256;
__global__ void __launch_bounds__(kRerankThreads) rerank_kernel(const RerankParams p) {
    __shared__ int wsum[kRerankThreads / 32];
    __shared__ float s[kMaxDraftNodes];
    __shared__ int par[kMaxDraftNodes];
    __shared__ int kept[kMaxDraftNodes], newidx[kMaxDraftNodes];
    __shared__ unsigned char elig[kMaxDraftNodes];
    const int b = blockIdx.x, tid = threadIdx.x, M = p.M, N = p.N;
    for (int i = tid; i < M; i += blockDim.x) {
        s[i] = p.node_score[size_t(b) * M + i];
        int q = p.node_parent[size_t(b) * M + i];
        if (i > 0 && (q < 0 || q >= i)) {                 // not a topologically ordered tree
            atomicOr(p.status, TREESPEC_STATUS_BAD_PARENT);
            q = 0;
        }
        par[i] = q;
        elig[i] = p.pool == nullptr && i > 0;
    }
    __syncthreads();
    if (p.pool) {                                         // ids outside 1 .. M-1 are ignored
        for (int e = tid; e < p.P; e += blockDim.x) {
            const int id = p.pool[size_t(b) * p.P + e];
            if (id > 0 && id < M) elig[id] = 1;
        }
        __syncthreads();
    }
    for (int i = tid; i < M; i += kRerankThreads) {
        int rank = 0;
        if (elig[i]) {
            const float si = s[i];
#pragma unroll 8
            for (int j = 1; j < M; ++j) rank += (elig[j] && before(s[j], j, si, i)) ? 1 : 0;
        }
        kept[i] = i == 0 || (elig[i] && rank < N - 1);
    }
    __syncthreads();
    {   // newidx = the kept nodes before i (root -> 0, kept nodes -> 1, 2, ...): a block scan,
        // four consecutive nodes a thread
        static_assert(kRerankThreads * 4 >= kMaxDraftNodes, "four nodes a thread cover the arrays");
        const int lane = tid & 31, warp = tid >> 5, i0 = tid * 4;
        int c[4], run = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            c[e] = i0 + e < M ? kept[i0 + e] : 0;
            run += c[e];
        }
        int inc = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        int ex = inc - run;
        for (int w = 0; w < warp; ++w) ex += wsum[w];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (i0 + e < M) newidx[i0 + e] = ex;
            ex += c[e];
        }
    }
    __syncthreads();
    const int nk = newidx[M - 1] + kept[M - 1];           // nodes kept, root included
    for (int q = nk + tid; q < N; q += blockDim.x) {
        p.parents[size_t(b) * N + q] = kAbsent;
        p.tokens[size_t(b) * N + q] = -1;
    }
    for (int i = tid; i < M; i += blockDim.x) {
        if (!kept[i]) continue;
        const int ni = newidx[i];
        int q = -1;
        if (i > 0) {
            q = par[i];
            if (!kept[q]) {                               // parent dropped: only with positive log-probs
                atomicOr(p.status, TREESPEC_STATUS_BAD_PARENT);
                q = 0;
            }
            q = newidx[q];
        }
        p.parents[size_t(b) * N + ni] = q;
        p.tokens[size_t(b) * N + ni] = p.node_token[size_t(b) * M + i];
    }
}

}  // namespace

cudaError_t launch_draft_step(const DraftParams& p, cudaStream_t s) {
    const unsigned grid = unsigned(p.B) * unsigned(p.F) * unsigned(p.S);
    if (p.V % 4 == 0) draft_topk_kernel<true><<<grid, kTopkThreads, 0, s>>>(p);
    else draft_topk_kernel<false><<<grid, kTopkThreads, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
    // launched as a programmatic dependent of the top-k grid: only its launch overlaps it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.B));
    cfg.blockDim = dim3(kSelectThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, draft_select_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_rerank(const RerankParams& p, cudaStream_t s) {
    rerank_kernel<<<unsigned(p.B), kRerankThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace treespec
