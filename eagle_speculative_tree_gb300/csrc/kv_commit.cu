// tree_kv_commit: move the accepted path's K/V rows next to the prefix, in place.
//
// One CTA per (sequence, kv head).  Thread 0 checks the sequence's path and that every
// position the commit touches (S .. S + max(path)) lies in its page table; every thread
// checks the page ids of the rows it moves.  The CTA then reads all
// source rows of K into shared memory, waits, writes them to their destinations, and
// does the same for V -- so a destination that is also a later source is never
// overwritten before it is read.  Rows move as 16-byte words.
#include "common.cuh"

namespace treespec {

namespace {

constexpr int kCommitThreads = 256;
constexpr int kMaxRowWords = 128 * 4 / 16;              // a float32 row of head dim 128
// staging for up to N - 1 accepted rows of one kv head (dynamic shared memory)
constexpr int kMaxStageBytes = (kMaxNodes - 1) * kMaxRowWords * 16;

__global__ void __launch_bounds__(kCommitThreads) kv_commit_kernel(const CommitParams p) {
    extern __shared__ uint4 buf[];                        // [N - 1][words]: the accepted rows of one kv head
    __shared__ int s_ok, s_len, s_S, s_badpage;
    const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int* path = p.path + size_t(b) * p.N;
    const int* ptab = p.page_table + size_t(b) * p.max_pages;
    if (tid == 0) {
        const int S = p.prefix_lens[b], n = p.len[b];
        uint32_t bad = 0;
        int top = 0;                                     // deepest node moved: positions S .. S + top are touched
        if (n < 0 || n > p.N - 1) {
            bad |= TREESPEC_STATUS_BAD_PATH;
        } else {
            int prev = 0;
            for (int k = 0; k < n; ++k) {
                const int x = path[k];
                if (x <= prev || x >= p.N) { bad |= TREESPEC_STATUS_BAD_PATH; break; }
                prev = x;
            }
            if (!bad) top = prev;
        }
        // the bound is what the moves touch, not the tree size: a tree padded after its own
        // last node commits whenever its accepted path fits the page table
        if (S < 0 || (long long)S + 1 + top > (long long)p.max_pages * p.ps) bad |= TREESPEC_STATUS_BAD_LENGTH;
        s_ok = bad == 0;
        s_len = bad ? 0 : n;
        s_S = S;
        s_badpage = 0;
        if (bad && h == 0) atomicOr(p.status, bad);
    }
    __syncthreads();
    const int n = s_len, S = s_S;
    const int words = p.D * p.elem / 16;                 // 16-byte words per row
    // every page a move touches must lie in the pool
    if (s_ok) {
        for (int k = tid; k < n; k += kCommitThreads) {
            const int src = S + path[k], dst = S + 1 + k;
            const int pgs = ptab[src / p.ps], pgd = ptab[dst / p.ps];
            if (pgs < 0 || pgs >= p.num_pool_pages || pgd < 0 || pgd >= p.num_pool_pages) s_badpage = 1;
        }
    }
    __syncthreads();
    if (!s_ok || s_badpage) {                            // this sequence stays as it was
        if (tid == 0 && h == 0) {
            if (s_badpage) atomicOr(p.status, TREESPEC_STATUS_BAD_PAGE);
            p.new_lens[b] = -1;
        }
        return;
    }
    auto row_word = [&](void* base, int pos, int w) -> uint4* {
        const int page = ptab[pos / p.ps];
        const size_t row = (size_t(page) * p.ps + (pos % p.ps)) * p.Hkv + h;
        return reinterpret_cast<uint4*>(static_cast<unsigned char*>(base) + row * size_t(p.D) * p.elem) + w;
    };
    for (int t = 0; t < 2; ++t) {
        void* base = t == 0 ? p.k : p.v;
        for (int e = tid; e < n * words; e += kCommitThreads) {
            const int k = e / words, w = e % words;
            buf[k * words + w] = *row_word(base, S + path[k], w);
        }
        __syncthreads();
        for (int e = tid; e < n * words; e += kCommitThreads) {
            const int k = e / words, w = e % words;
            *row_word(base, S + 1 + k, w) = buf[k * words + w];
        }
        __syncthreads();
    }
    if (tid == 0 && h == 0) p.new_lens[b] = S + 1 + n;
}

}  // namespace

cudaError_t launch_kv_commit(const CommitParams& p, cudaStream_t s) {
    const int smem = max(16, (p.N - 1) * (p.D * p.elem / 16) * 16);
    if (smem > kMaxStageBytes) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kv_commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxStageBytes);
    if (e != cudaSuccess) return e;
    kv_commit_kernel<<<dim3(unsigned(p.B), unsigned(p.Hkv)), kCommitThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace treespec
