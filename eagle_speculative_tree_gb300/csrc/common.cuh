// Shared device helpers and launch parameter blocks of libtreespec.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "treespec.h"

namespace treespec {

// Tree nodes per sequence.  A node's ancestor-or-self set is kAncWords 64-bit words
// (word w holds nodes 64w .. 64w+63): one word covers the 64-node trees of the radar
// page's single-word mask, two cover trees of up to 128 nodes.
constexpr int kMaxNodes = 128;
constexpr int kStreamMaxBatch = 256;   // persistent two-tile attention: sequences per call
constexpr int kStreamMaxCtas = 1024;   // persistent two-tile attention: CTAs (one per SM)
constexpr int kAncWords = 2;
constexpr int kAbsent = TREESPEC_ABSENT;   // parent entry of a padding slot past the end of a smaller tree
constexpr size_t kWsAlign = 256;
// Every wait inside a kernel gives up after this long (nanoseconds), sets
// TREESPEC_STATUS_TIMEOUT and winds the CTA down.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Programmatic dependent launch between the tree prologue and the attention kernel that
// follows it on the stream.  The prologue lets the next grid launch at once; the
// attention kernel, launched with the programmatic-serialisation attribute, waits at its
// first instruction until the prologue has finished and its writes are visible, so only
// the launch and the CTAs' start overlap the prologue.  Launched without the attribute,
// the wait returns at once.
__device__ __forceinline__ void grid_dep_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// bf16 <-> f32 on raw bit patterns (bf16 is the high half of an f32).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return uint16_t((u >> 16) | 0x40u);   // NaN stays NaN
    u += 0x7fffu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

// Bits sh .. sh+31 of a 128-bit ancestor set {a0, a1} (bit j of the set = node j), as one
// 32-bit word; positions outside 0..127 read as 0.  sh may be negative (down to -31).
__device__ __forceinline__ uint32_t anc_bits32(uint64_t a0, uint64_t a1, int sh) {
    if (sh <= -32 || sh >= 128) return 0u;
    if (sh < 0) return uint32_t(a0 << (-sh));
    if (sh >= 64) return uint32_t(a1 >> (sh - 64));
    uint64_t w = a0 >> sh;
    if (sh > 32) w |= a1 << (64 - sh);
    return uint32_t(w);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ attention

// Workspace of tree_attn_verify (offsets in bytes from the workspace base).
struct AttnLayout {
    size_t status, anc, lens, nn, ml, acc, flags, total;
};

struct AttnPlan {
    int kernel;          // TREESPEC_KERNEL_SIMT / _TC / _TC_PAIR / _TC_2SM / _TC_STREAM
    int num_splits;
    int split_tokens;
    int rows_per_block;
    int row_blocks;
    int merge;
    int stream_ctas;     // _TC_STREAM: persistent CTAs (one per SM)
};

struct AttnParams {
    const void* q;
    const void* k;
    const void* v;
    const int32_t* page_table;
    const int32_t* prefix_lens;   // caller's array (read by the prologue only)
    const int32_t* parents;       // caller's array (read by the prologue only)
    void* out;
    uint32_t* status;
    uint64_t* anc;                // [B][N][kAncWords] ancestor-or-self sets
    int32_t* lens;                // [B] validated prefix lengths, -1 = invalid sequence
    int32_t* nn;                  // [B] nodes of each tree: parent entries before the first kAbsent
    float* part_ml;               // [B][Hkv][splits][R][2]  (m in log2 units, l)
    float* part_acc;              // [B][Hkv][splits][R][D]
    int B, N, Hq, Hkv, G, R, D, ps, max_pages, num_pool_pages;
    int num_splits, split_tokens, rows_per_block, row_blocks, merge;
    float scale_log2;             // log2(e) / sqrt(D)
    int stream_ctas;              // persistent two-tile kernel: CTAs (one per SM)
    int32_t* stream_flags;        // persistent two-tile kernel: [2 * CTAs][2] a piece's partial is written
                                  // (slot, query tile); zeroed by the prologue
    uint64_t wait_ns;             // bound of the tensor-core kernels' pipeline waits (kDefaultWaitNs unless a test shortens it)
};

// ------------------------------------------------------------------ accept

struct AcceptLayout {
    size_t status, amax, stats, izs, total;
};

struct AcceptParams {
    const float* logits;
    const int32_t* tokens;
    const float* probs;
    const int32_t* parents;
    const float* uniforms;
    int32_t* path;
    int32_t* len;
    int32_t* bonus;
    uint32_t* status;
    int32_t* amax;    // [B][N]   lowest argmax of each target row
    float* stats;     // [B][N][2] (M2, S): max of logits*c and sum of 2^(logits*c - M2)
    float* izs;       // [B][N][64] 1/Z_1.. of the sibling residual chain of each row (0: Z = 0)
    int B, N, V;
    float temperature;
    float c;          // log2(e) / temperature
    int sms;          // SMs of the device (the cluster size of the walk depends on B / sms)
    int probs_on_host;  // draft_probs is host memory read over the CPU-GPU link: fetch a draft
                        // row only where a child is rejected, never ahead
};

// Kernel launchers (each returns cudaGetLastError() of its launch).
cudaError_t launch_tree_prologue(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_simt(const AttnParams& p, int dtype, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_tc_2sm(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_tc_pair(const AttnParams& p, cudaStream_t s);
cudaError_t launch_attn_tc_stream(const AttnParams& p, cudaStream_t s);
bool attn_tc_supported(int dtype, int D);
// TMA map of a K or V page pool [P][16][Hkv][128] bf16, one page x 64 head dims per box
bool make_pool_map(CUtensorMap* map, const void* base, int Hkv, long long pool_tokens);
cudaError_t launch_attn_merge(const AttnParams& p, int dtype, cudaStream_t s);
cudaError_t launch_accept(const AcceptParams& p, int mode, cudaStream_t s, int* kernels);

// KV commit (tree_kv_commit)
struct CommitParams {
    void* k;
    void* v;
    const int32_t* page_table;
    const int32_t* prefix_lens;
    const int32_t* path;
    const int32_t* len;
    int32_t* new_lens;
    uint32_t* status;
    int B, N, Hkv, D, ps, max_pages, num_pool_pages, elem;   // elem: bytes per element
};
cudaError_t launch_kv_commit(const CommitParams& p, cudaStream_t s);

// Draft-tree construction (tree_draft_step, tree_rerank)
constexpr int kMaxTopk = 16;          // branching per step
constexpr int kMaxFrontier = 16;      // frontier rows per step (1 or topk)
constexpr int kMaxDraftNodes = 1024;  // node arrays of a sequence (root + steps * topk)
constexpr int kMaxDraftSplits = 16;   // CTAs that share one frontier row's vocabulary
struct DraftParams {
    const float* logprobs;            // [B][F][V]
    const int32_t* frontier_in;       // [B][F] node ids (unused at step 0)
    int32_t* frontier_out;            // [B][k]
    int32_t* node_parent;             // [B][M]
    int32_t* node_token;
    float* node_score;
    int32_t* tk_tok;                  // workspace: [B][F][S][k] top-k of each part of a row
    float* tk_lp;
    uint32_t* status;
    int B, F, V, k, step, M;
    int S, chunk;                     // a row's vocabulary in S parts of `chunk` tokens (one CTA each)
};
struct RerankParams {
    const int32_t* node_parent;
    const int32_t* node_token;
    const float* node_score;
    const int32_t* pool;              // [B][P] eligible node ids, or NULL: every node
    int P;
    int32_t* parents;                 // [B][N]
    int32_t* tokens;
    uint32_t* status;
    int B, M, N;
};
cudaError_t launch_draft_step(const DraftParams& p, cudaStream_t s);
cudaError_t launch_rerank(const RerankParams& p, cudaStream_t s);
size_t attn_simt_smem_bytes(int dtype, int D, int R_block);

}  // namespace treespec
