// Tree prologue: parent array -> ancestor-or-self sets, plus validation.
//
// "Tech Radar: SGLang EAGLE-2", section 2: node i may attend to node j iff j is an
// ancestor of i or j == i; section 5 item 1: with at most 64 nodes the relation is
// one 64-bit word per node and the test is (word_i >> j) & 1.  Trees of up to 128 nodes
// ("EAGLE-2 & Lookahead Decoding", section 6: the tree grows when the load is light) use
// two words per node, word w holding nodes 64w .. 64w+63.  The set of node i is its own
// bit OR the bits of every node on its parent chain.
//
// A batch may hold trees of different sizes ("EAGLE-2 & Lookahead Decoding", section 6,
// batched dynamic tree slicing): a row of the parent array is padded with kAbsent after
// its tree's N_b nodes.  The prologue records N_b; padding slots get no ancestry bits and
// the sequence is S + N_b tokens long.
#include "common.cuh"

namespace treespec {

__global__ void __launch_bounds__(kMaxNodes) tree_prologue_kernel(AttnParams p) {
    __shared__ int par[kMaxNodes];
    __shared__ int bad, first_pad;
    grid_dep_release();                   // the attention kernel may launch; it waits for this grid
    const int b = blockIdx.x, i = threadIdx.x, N = p.N;
    if (i == 0) {
        bad = 0;
        first_pad = N;
    }
    __syncthreads();
    int pi = 0;
    if (i < N) {
        pi = p.parents[(size_t)b * N + i];
        if (pi == kAbsent) atomicMin(&first_pad, i);
    }
    __syncthreads();
    const int nb = max(first_pad, 1);     // the root is always a node
    if (i < N) {
        // a node's parent is an earlier node; every slot after the first padding slot pads too
        const bool ok = i >= nb ? pi == kAbsent : (i == 0) ? (pi == -1) : (pi >= 0 && pi < i);
        if (!ok) {
            bad = 1;
            pi = (i == 0) ? -1 : 0;       // keep the walk finite: attach to the root
        }
        par[i] = pi;
    }
    __syncthreads();
    if (i < N) {
        static_assert(kAncWords == 2, "two words per node");
        uint64_t w0 = 0, w1 = 0;                                  // nodes 0..63, 64..127
        if (i < nb) {
            for (int j = i; j >= 0; j = par[j]) {                 // i, then its parent chain (par[j] < j)
                if (j < 64) w0 |= 1ull << j;
                else w1 |= 1ull << (j - 64);
            }
        }
        p.anc[((size_t)b * N + i) * kAncWords] = w0;
        p.anc[((size_t)b * N + i) * kAncWords + 1] = w1;
    }
    if (p.stream_flags && b == 0)         // the persistent kernel's piece flags
        for (int e = i; e < 2 * p.stream_ctas * 2; e += kMaxNodes) p.stream_flags[e] = 0;
    if (i == 0) {
        p.nn[b] = nb;
        int S = p.prefix_lens[b];
        long long need = (long long)S + nb;
        bool ok = S >= 0 && need <= (long long)p.max_pages * p.ps;
        p.lens[b] = ok ? S : -1;
        uint32_t st = (bad ? TREESPEC_STATUS_BAD_PARENT : 0u) | (ok ? 0u : TREESPEC_STATUS_BAD_LENGTH);
        if (st) atomicOr(p.status, st);
    }
}

cudaError_t launch_tree_prologue(const AttnParams& p, cudaStream_t s) {
    tree_prologue_kernel<<<p.B, kMaxNodes, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace treespec
