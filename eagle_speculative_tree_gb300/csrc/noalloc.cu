// tree_attn_verify_noalloc: the tree-attention pass for callers that cannot hand the
// library any device memory of their own.
//
// Some callers can't call cudaMalloc (or any allocator) at the point where they verify
// a tree: an application that reserves nearly all device memory up front for its own
// pools (a serving engine that gives the rest of HBM to its KV-cache allocator and
// forbids ad-hoc allocations), or a latency-critical decode loop where an allocation's
// implicit device synchronisation is not acceptable.  For them the scratch space that
// tree_attn_verify normally takes as `workspace` (status word, ancestor words, checked
// lengths, split partials) lives instead in one fixed device array defined in this
// file.  The array exists on every GPU that loads this library, for the life of the
// process, whether or not this entry point is used.
//
// Set-up: the first call on a device looks up that device's address of the array with
// cudaGetSymbolAddress (with that device current) and caches it; make that first call
// before any stream capture.  Nothing is allocated, here or later.
//
// Sharing: every call on a device uses the same array and leaves its contents behind.
// Nothing in it has to start at zero -- each call clears its status word and writes
// every other byte it reads before reading it -- but two calls whose work overlaps on
// the GPU (different streams, or host threads racing) corrupt each other's scratch.
// Serialise the calls, e.g. issue them all on one stream.
#include <mutex>

#include "common.cuh"

namespace {

// Largest workspace this entry point can serve (treespec_attn_workspace_bytes of the
// shape must not exceed it).  32 MiB covers a single split for thousands of
// (sequence, kv head) pairs, or split partials for the moderate batches.
constexpr size_t kScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

int scratch_of_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return TREESPEC_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_scratch) != cudaSuccess || !addr) {
            cudaGetLastError();
            return TREESPEC_ERR_DEVICE;
        }
        g_scratch_addr[dev] = addr;
    }
    *out = g_scratch_addr[dev];
    return TREESPEC_OK;
}

}  // namespace

extern "C" int tree_attn_verify_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                        const int32_t* page_table, const int32_t* prefix_lens,
                                        const int32_t* tree_parents, void* out,
                                        const treespec_attn_shape* shape, treespec_stream_t stream) {
    treespec_attn_plan plan;
    const int rc = treespec_attn_plan_for(shape, &plan);
    if (rc != TREESPEC_OK) return rc;
    treespec_attn_shape sh = *shape;
    // The persistent two-tile kernel's partial slots (about 40 MB on 152 SMs) do not fit the
    // array: an automatic plan that picks it runs the two-tile kernel one range per CTA.
    if (sh.kernel == TREESPEC_KERNEL_AUTO && plan.kernel == TREESPEC_KERNEL_TC_STREAM &&
        treespec_attn_workspace_bytes(&sh) > kScratchBytes)
        sh.kernel = TREESPEC_KERNEL_TC_PAIR;
    if (treespec_attn_workspace_bytes(&sh) > kScratchBytes) return TREESPEC_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int dev_rc = scratch_of_current_device(&scratch);
    if (dev_rc != TREESPEC_OK) return dev_rc;
    return tree_attn_verify(q, k_pages, v_pages, page_table, prefix_lens, tree_parents, out, &sh, scratch,
                            kScratchBytes, stream);
}

// The device status word of the last tree_attn_verify_noalloc call on the current device
// (the first word of the fixed array, where the workspace layout keeps it).  Waits for
// `stream` first.  Callers of the no-allocation entry point have no workspace pointer
// to hand treespec_read_status, so this is their only view of the bad-index and
// timeout bits the kernels set.
extern "C" int treespec_noalloc_read_status(uint32_t* status, treespec_stream_t stream) {
    if (!status) return TREESPEC_ERR_NULL_POINTER;
    void* scratch = nullptr;
    const int rc = scratch_of_current_device(&scratch);
    if (rc != TREESPEC_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    if (cudaMemcpy(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TREESPEC_ERR_LAUNCH;
    return TREESPEC_OK;
}
