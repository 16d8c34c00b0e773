// Tree prologue: parent array -> 64-bit ancestor-or-self words, plus validation.
//
// "Tech Radar: SGLang EAGLE-2", section 2: node i may attend to node j iff j is an
// ancestor of i or j == i; section 5 item 1: with at most 64 nodes the relation is
// one 64-bit word per node and the test is (word_i >> j) & 1.  The word of node i is
// its own bit OR the bits of every node on its parent chain.
#include "common.cuh"

namespace treespec {

__global__ void __launch_bounds__(64) tree_prologue_kernel(AttnParams p) {
    __shared__ int par[kMaxNodes];
    __shared__ int bad;
    const int b = blockIdx.x, i = threadIdx.x, N = p.N;
    if (i == 0) bad = 0;
    __syncthreads();
    if (i < N) {
        int pi = p.parents[(size_t)b * N + i];
        bool ok = (i == 0) ? (pi == -1) : (pi >= 0 && pi < i);
        if (!ok) {
            bad = 1;
            pi = (i == 0) ? -1 : 0;       // keep the walk finite: attach to the root
        }
        par[i] = pi;
    }
    __syncthreads();
    if (i < N) {
        uint64_t w = 1ull << i;
        for (int j = par[i]; j >= 0; j = par[j]) w |= 1ull << j;   // par[j] < j: at most i steps
        p.anc[(size_t)b * N + i] = w;
    }
    if (i == 0) {
        int S = p.prefix_lens[b];
        long long need = (long long)S + N;
        bool ok = S >= 0 && need <= (long long)p.max_pages * p.ps;
        p.lens[b] = ok ? S : -1;
        uint32_t st = (bad ? TREESPEC_STATUS_BAD_PARENT : 0u) | (ok ? 0u : TREESPEC_STATUS_BAD_LENGTH);
        if (st) atomicOr(p.status, st);
    }
}

cudaError_t launch_tree_prologue(const AttnParams& p, cudaStream_t s) {
    tree_prologue_kernel<<<p.B, 64, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace treespec
