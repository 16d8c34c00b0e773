// Host side of libtreespec: argument checks, the split planner, workspace layout and
// launches.  Every exported symbol is declared in include/treespec.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace treespec {
namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};     // see treespec_set_wait_limit_ns
std::atomic<int> g_launch_error{0};                 // cudaError_t of the last rejected launch

// TREESPEC_ERR_LAUNCH for a launch the runtime rejected, keeping the runtime's code
int launch_failed(cudaError_t e) {
    g_launch_error.store(int(e));
    return TREESPEC_ERR_LAUNCH;
}

constexpr int kDefaultSms = 152;
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
};

// Per-device attributes, read once.  Returns false when no device is usable.
bool device_info(DeviceInfo* out) {
    static DeviceInfo cache[kMaxDevices];
    static std::mutex mu;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        cache[dev] = d;
    }
    *out = cache[dev];
    return true;
}

int sm_count_or_default() {
    DeviceInfo d;
    return device_info(&d) ? d.sms : kDefaultSms;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The persistent two-tile kernel keeps the batch's 64-token tile offsets in shared memory
// and its tile positions (over row-block pairs, sequences and kv heads) as int32: at most
// kStreamMaxBatch sequences and fewer than 2^31 positions.
bool stream_fits(const treespec_attn_shape& s) {
    const long long tiles = ((long long)s.max_pages_per_seq * s.page_size + 63) / 64 + 3;   // + tree nodes
    const long long G = s.num_q_heads / s.num_kv_heads;
    const long long pairs = ((long long)s.num_nodes * G + 255) / 256;
    return s.batch <= kStreamMaxBatch && pairs * s.num_kv_heads * s.batch * tiles < (1ll << 31);
}

int check_attn_shape(const treespec_attn_shape* s) {
    if (!s) return TREESPEC_ERR_NULL_POINTER;
    if (s->dtype != TREESPEC_DTYPE_F32 && s->dtype != TREESPEC_DTYPE_BF16) return TREESPEC_ERR_DTYPE;
    if (s->batch < 1 || s->batch > 65535) return TREESPEC_ERR_SHAPE;
    if (s->num_nodes < 1 || s->num_nodes > kMaxNodes) return TREESPEC_ERR_SHAPE;
    if (s->num_kv_heads < 1 || s->num_q_heads < 1 || s->num_q_heads % s->num_kv_heads) return TREESPEC_ERR_SHAPE;
    if (s->head_dim != 64 && s->head_dim != 128) return TREESPEC_ERR_SHAPE;
    if (s->page_size != 16) return TREESPEC_ERR_SHAPE;
    if (s->max_pages_per_seq < 1 || s->num_pool_pages < 1) return TREESPEC_ERR_SHAPE;
    if ((long long)s->max_pages_per_seq * s->page_size > (1ll << 30)) return TREESPEC_ERR_SHAPE;
    const long long R = (long long)s->num_nodes * (s->num_q_heads / s->num_kv_heads);
    if (R > 4096 || (long long)s->num_kv_heads * ((R + 63) / 64) > 65535) return TREESPEC_ERR_SHAPE;
    if (s->kernel < TREESPEC_KERNEL_AUTO || s->kernel > TREESPEC_KERNEL_TC_STREAM) return TREESPEC_ERR_SHAPE;
    if (s->num_splits < 0) return TREESPEC_ERR_SHAPE;
    if (s->kernel >= TREESPEC_KERNEL_TC) {
        if (!attn_tc_supported(s->dtype, s->head_dim)) return TREESPEC_ERR_DTYPE;
        if ((long long)s->num_pool_pages * s->page_size >= (1ll << 31)) return TREESPEC_ERR_SHAPE;
    }
    if (s->kernel >= TREESPEC_KERNEL_TC_PAIR && ((R + 127) / 128) % 2 != 0) return TREESPEC_ERR_SHAPE;
    if (s->kernel == TREESPEC_KERNEL_TC_STREAM && !stream_fits(*s)) return TREESPEC_ERR_SHAPE;
    return TREESPEC_OK;
}

AttnPlan make_plan(const treespec_attn_shape& s, int sms) {
    AttnPlan p{};
    const int G = s.num_q_heads / s.num_kv_heads;
    const int R = s.num_nodes * G;
    const bool tc_ok = attn_tc_supported(s.dtype, s.head_dim) &&
                       (long long)s.num_pool_pages * s.page_size < (1ll << 31);
    // Tensor cores for every bf16 / head_dim 128 shape: measured faster than the CUDA-core
    // kernel from 16 rows per kv head up (rows are padded to the 128-row MMA tile).
    // Where the row blocks of a kv head pair up, a K/V tile should serve 256 rows: the
    // one-tile kernel's L2 reads bind first otherwise.  Of the two kernels that do that, the
    // CTA-pair kernel (256-row MMAs across two SMs) when the two-tile kernel's CTAs would
    // not fill the SMs once, the two-tile kernel (two 128-row tiles in one CTA) otherwise.
    // Measured at 64 q / 8 kv heads, 64 nodes, 8192-token prefixes (ms, CTA pair / two-tile /
    // one-tile): batch 2 0.080 / 0.088 / -, batch 8 0.149 / 0.169 / 0.169, batch 16
    // 0.279 / 0.243 / 0.315, batch 32 0.491 / 0.474 / 0.543.
    if (s.kernel >= TREESPEC_KERNEL_TC || (s.kernel == TREESPEC_KERNEL_AUTO && tc_ok)) {
        const long long rbs = (R + 127) / 128;
        const bool paired = rbs % 2 == 0;
        const long long pair_units = (long long)s.batch * s.num_kv_heads * (rbs / 2);
        const bool small = pair_units < sms;
        // the persistent form pays a merge of the cut units and a few us per unit change,
        // which two waves of two-tile CTAs or more amortise (measured: batch 32 0.460 ms
        // against 0.473, batch 16 0.255 against 0.250)
        const bool many = pair_units >= 2ll * sms;
        p.kernel = s.kernel != TREESPEC_KERNEL_AUTO ? s.kernel
                   : !paired                        ? TREESPEC_KERNEL_TC
                   : small                          ? TREESPEC_KERNEL_TC_2SM
                   : (many && stream_fits(s))       ? TREESPEC_KERNEL_TC_STREAM
                                                    : TREESPEC_KERNEL_TC_PAIR;
        p.rows_per_block = 128;
    } else {
        p.kernel = TREESPEC_KERNEL_SIMT;
        p.rows_per_block = R < 64 ? R : 64;
    }
    p.row_blocks = (R + p.rows_per_block - 1) / p.rows_per_block;
    const long long max_tokens = (long long)s.max_pages_per_seq * s.page_size;
    const int tile = 128;                       // split sizes are multiples of every tile size
    const bool tc = p.kernel != TREESPEC_KERNEL_SIMT;
    const long long units = (long long)s.batch * s.num_kv_heads *
                            (p.kernel == TREESPEC_KERNEL_TC_PAIR ? p.row_blocks / 2 : p.row_blocks);
    long long splits;
    if (s.num_splits > 0) {
        splits = s.num_splits;
    } else if (tc) {
        // One CTA fits an SM.  Split a sequence only as far as one wave of CTAs holds
        // (rounded down: a few CTAs past the SM count would run as a second wave), keep a
        // CTA's run at most 66 tiles (a ragged batch's longest sequences split into several
        // CTAs; an 8256-token one stays whole), and no chunk below two tiles: each split
        // costs a pipeline fill and its partials.  Measured against earlier rules: about two
        // CTAs per SM gave 32 x 8192 tokens at batch 8 0.192 ms against 0.147, 8 x 4096
        // tokens (32 kv heads) 0.131 against 0.116, 64 ragged sequences up to 32768 tokens
        // 0.774 against 0.751; rounding up gave the 64 q / 8 kv-head, 64-node shape 0.056 ms
        // at batch 1 (160 CTA-pair CTAs) against 0.044 (128) and 0.077 at batch 2 against 0.058.
        splits = units >= sms ? 1 : sms / units;
        const long long cap = 66ll * tile;
        splits = std::max(splits, (max_tokens + cap - 1) / cap);
        splits = std::min(splits, std::max(1ll, (max_tokens + 2 * tile - 1) / (2 * tile)));
        if (splits < 1) splits = 1;
    } else {
        const long long target = 2ll * sms;      // two waves of CTAs, then merge
        splits = (target + units - 1) / units;
        if (splits < 1) splits = 1;
    }
    long long chunk = (max_tokens + splits - 1) / splits;
    chunk = (chunk + tile - 1) / tile * tile;
    if (s.num_splits == 0 && !tc && chunk > 16384) chunk = 16384;   // bounded CTA length
    if (chunk < tile) chunk = tile;
    p.split_tokens = int(chunk);
    p.num_splits = int((max_tokens + chunk - 1) / chunk);
    if (p.num_splits > 65535) {
        p.num_splits = 65535;
        p.split_tokens = int((max_tokens + 65534) / 65535);
        p.split_tokens = (p.split_tokens + tile - 1) / tile * tile;
    }
    p.merge = p.num_splits > 1;
    if (p.kernel == TREESPEC_KERNEL_TC_STREAM) {   // no splits: the SMs share the tiles evenly
        p.num_splits = 1;
        p.split_tokens = int(std::min<long long>(max_tokens + 128, 1ll << 30));
        p.merge = 0;
        p.stream_ctas = std::min(sms, kStreamMaxCtas);
    }
    return p;
}

AttnLayout attn_layout(const treespec_attn_shape& s, const AttnPlan& p) {
    AttnLayout L{};
    const size_t R = size_t(s.num_nodes) * (s.num_q_heads / s.num_kv_heads);
    size_t off = 0;
    L.status = off;
    off += kWsAlign;
    L.anc = off;
    off = align_up(off + size_t(s.batch) * s.num_nodes * kAncWords * 8, kWsAlign);
    L.lens = off;
    off = align_up(off + size_t(s.batch) * 4, kWsAlign);
    L.nn = off;
    off = align_up(off + size_t(s.batch) * 4, kWsAlign);
    const size_t parts = p.merge ? size_t(s.batch) * s.num_kv_heads * p.num_splits * R : 0;
    L.ml = off;
    off = align_up(off + parts * 2 * 4, kWsAlign);
    L.acc = off;
    off = align_up(off + parts * s.head_dim * 4, kWsAlign);
    if (p.kernel == TREESPEC_KERNEL_TC_STREAM) {
        // two partial slots of 2 x 128 rows per CTA for the pieces of cut units, and their
        // ready flags
        const size_t rows = size_t(2) * p.stream_ctas * 256;
        L.ml = off;
        off = align_up(off + rows * 2 * 4, kWsAlign);
        L.acc = off;
        off = align_up(off + rows * s.head_dim * 4, kWsAlign);
        L.flags = off;
        off = align_up(off + size_t(2) * p.stream_ctas * 2 * 4, kWsAlign);
    }
    L.total = off;
    return L;
}

AcceptLayout accept_layout(int B, int N) {
    AcceptLayout L{};
    size_t off = 0;
    L.status = off;
    off += kWsAlign;
    L.amax = off;
    off = align_up(off + size_t(B) * N * 4, kWsAlign);
    L.stats = off;
    off = align_up(off + size_t(B) * N * 8, kWsAlign);
    L.izs = off;
    off = align_up(off + size_t(B) * N * kMaxNodes * 4, kWsAlign);
    L.total = off;
    return L;
}

int check_device() {
    DeviceInfo d;
    if (!device_info(&d)) return TREESPEC_ERR_DEVICE;
    if (d.cc_major != 10 || d.cc_minor != 3) return TREESPEC_ERR_DEVICE;
    return TREESPEC_OK;
}

}  // namespace
}  // namespace treespec

using namespace treespec;

extern "C" size_t treespec_attn_workspace_bytes(const treespec_attn_shape* shape) {
    if (check_attn_shape(shape) != TREESPEC_OK) return 0;
    return attn_layout(*shape, make_plan(*shape, sm_count_or_default())).total;
}

extern "C" int treespec_attn_plan_for(const treespec_attn_shape* shape, treespec_attn_plan* plan) {
    const int rc = check_attn_shape(shape);
    if (rc != TREESPEC_OK) return rc;
    if (!plan) return TREESPEC_ERR_NULL_POINTER;
    const AttnPlan p = make_plan(*shape, sm_count_or_default());
    plan->kernel = p.kernel;
    plan->num_splits = p.num_splits;
    plan->split_tokens = p.split_tokens;
    plan->rows_per_block = p.rows_per_block;
    plan->row_blocks = p.row_blocks;
    plan->merge = p.merge;
    return TREESPEC_OK;
}

extern "C" int tree_attn_verify(const void* q, const void* k_pages, const void* v_pages,
                                const int32_t* page_table, const int32_t* prefix_lens,
                                const int32_t* tree_parents, void* out,
                                const treespec_attn_shape* shape, void* workspace,
                                size_t workspace_bytes, treespec_stream_t stream) {
    int rc = check_attn_shape(shape);
    if (rc != TREESPEC_OK) return rc;
    if (!q || !k_pages || !v_pages || !page_table || !prefix_lens || !tree_parents || !out)
        return TREESPEC_ERR_NULL_POINTER;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
        return TREESPEC_ERR_ALIGNMENT;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)) return TREESPEC_ERR_WORKSPACE;
    rc = check_device();
    if (rc != TREESPEC_OK) return rc;
    const treespec_attn_shape& s = *shape;
    const AttnPlan plan = make_plan(s, sm_count_or_default());
    const AttnLayout lay = attn_layout(s, plan);
    if (workspace_bytes < lay.total) return TREESPEC_ERR_WORKSPACE;

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    AttnParams p{};
    p.q = q;
    p.k = k_pages;
    p.v = v_pages;
    p.page_table = page_table;
    p.prefix_lens = prefix_lens;
    p.parents = tree_parents;
    p.out = out;
    p.status = reinterpret_cast<uint32_t*>(ws + lay.status);
    p.anc = reinterpret_cast<uint64_t*>(ws + lay.anc);
    p.lens = reinterpret_cast<int32_t*>(ws + lay.lens);
    p.nn = reinterpret_cast<int32_t*>(ws + lay.nn);
    p.part_ml = reinterpret_cast<float*>(ws + lay.ml);
    p.part_acc = reinterpret_cast<float*>(ws + lay.acc);
    p.B = s.batch;
    p.N = s.num_nodes;
    p.Hq = s.num_q_heads;
    p.Hkv = s.num_kv_heads;
    p.G = s.num_q_heads / s.num_kv_heads;
    p.R = p.N * p.G;
    p.D = s.head_dim;
    p.ps = s.page_size;
    p.max_pages = s.max_pages_per_seq;
    p.num_pool_pages = s.num_pool_pages;
    p.num_splits = plan.num_splits;
    p.split_tokens = plan.split_tokens;
    p.rows_per_block = plan.rows_per_block;
    p.row_blocks = plan.row_blocks;
    p.merge = plan.merge;
    p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(s.head_dim)));
    p.wait_ns = g_wait_ns.load();
    p.stream_ctas = plan.stream_ctas;
    p.stream_flags = plan.kernel == TREESPEC_KERNEL_TC_STREAM ? reinterpret_cast<int32_t*>(ws + lay.flags) : nullptr;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    if (launch_tree_prologue(p, st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    g_launches++;
    const cudaError_t e = plan.kernel == TREESPEC_KERNEL_TC_STREAM ? launch_attn_tc_stream(p, st)
                          : plan.kernel == TREESPEC_KERNEL_TC_PAIR ? launch_attn_tc_pair(p, st)
                          : plan.kernel == TREESPEC_KERNEL_TC_2SM ? launch_attn_tc_2sm(p, st)
                          : plan.kernel == TREESPEC_KERNEL_TC    ? launch_attn_tc(p, st)
                                                                 : launch_attn_simt(p, s.dtype, st);
    if (e != cudaSuccess) return launch_failed(e);
    g_launches++;
    if (plan.merge) {
        if (launch_attn_merge(p, s.dtype, st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
        g_launches++;
    }
    return TREESPEC_OK;
}

extern "C" size_t treespec_accept_workspace_bytes(int32_t batch, int32_t num_nodes, int32_t vocab) {
    if (batch < 1 || num_nodes < 1 || num_nodes > kMaxNodes || vocab < 1 || vocab > (1 << 30)) return 0;
    return accept_layout(batch, num_nodes).total;
}

extern "C" int tree_accept_with_mode(const float* target_logits, const int32_t* draft_tokens,
                                     const float* draft_probs, const int32_t* tree_parents,
                                     const float* uniforms, float temperature, int32_t* accept_path,
                                     int32_t* accept_len, int32_t* bonus_token, int32_t batch,
                                     int32_t num_nodes, int32_t vocab, int32_t mode, void* workspace,
                                     size_t workspace_bytes, treespec_stream_t stream) {
    if (batch < 1 || num_nodes < 1 || num_nodes > kMaxNodes || vocab < 1 || vocab > (1 << 30))
        return TREESPEC_ERR_SHAPE;
    if ((long long)batch * num_nodes > 0x7fffffffll) return TREESPEC_ERR_SHAPE;
    if (mode < TREESPEC_ACCEPT_AUTO || mode > TREESPEC_ACCEPT_PATH_ONLY) return TREESPEC_ERR_SHAPE;
    if (!target_logits || !draft_tokens || !tree_parents || !accept_path || !accept_len || !bonus_token)
        return TREESPEC_ERR_NULL_POINTER;
    if (!(temperature >= 0.f) || std::isinf(temperature)) return TREESPEC_ERR_SAMPLING;
    const bool stoch = temperature > 0.f;
    if (stoch && (!draft_probs || !uniforms)) return TREESPEC_ERR_SAMPLING;
    if (!aligned16(target_logits) || (stoch && !aligned16(draft_probs))) return TREESPEC_ERR_ALIGNMENT;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign)) return TREESPEC_ERR_WORKSPACE;
    const AcceptLayout lay = accept_layout(batch, num_nodes);
    if (workspace_bytes < lay.total) return TREESPEC_ERR_WORKSPACE;
    const int rc = check_device();
    if (rc != TREESPEC_OK) return rc;
    if (mode == TREESPEC_ACCEPT_AUTO) mode = TREESPEC_ACCEPT_PATH_ONLY;   // measured faster on every workload

    unsigned char* ws = static_cast<unsigned char*>(workspace);
    AcceptParams p{};
    p.logits = target_logits;
    p.tokens = draft_tokens;
    p.probs = draft_probs;
    p.parents = tree_parents;
    p.uniforms = uniforms;
    p.path = accept_path;
    p.len = accept_len;
    p.bonus = bonus_token;
    p.status = reinterpret_cast<uint32_t*>(ws + lay.status);
    p.amax = reinterpret_cast<int32_t*>(ws + lay.amax);
    p.stats = reinterpret_cast<float*>(ws + lay.stats);
    p.izs = reinterpret_cast<float*>(ws + lay.izs);
    p.B = batch;
    p.N = num_nodes;
    p.V = vocab;
    p.temperature = temperature;
    p.c = stoch ? float(1.4426950408889634 / double(temperature)) : 0.f;
    p.sms = sm_count_or_default();
    if (stoch) {
        cudaPointerAttributes at{};
        if (cudaPointerGetAttributes(&at, draft_probs) == cudaSuccess) p.probs_on_host = at.type == cudaMemoryTypeHost;
        else cudaGetLastError();                         // not a pointer CUDA knows: treat as device memory
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    int kernels = 0;
    if (launch_accept(p, mode, st, &kernels) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    g_launches += kernels;
    return TREESPEC_OK;
}

extern "C" int tree_accept(const float* target_logits, const int32_t* draft_tokens,
                           const float* draft_probs, const int32_t* tree_parents,
                           const float* uniforms, float temperature, int32_t* accept_path,
                           int32_t* accept_len, int32_t* bonus_token, int32_t batch,
                           int32_t num_nodes, int32_t vocab, void* workspace,
                           size_t workspace_bytes, treespec_stream_t stream) {
    return tree_accept_with_mode(target_logits, draft_tokens, draft_probs, tree_parents, uniforms, temperature,
                                 accept_path, accept_len, bonus_token, batch, num_nodes, vocab,
                                 TREESPEC_ACCEPT_AUTO, workspace, workspace_bytes, stream);
}

extern "C" size_t treespec_commit_workspace_bytes(void) { return kWsAlign; }

extern "C" int tree_kv_commit(void* k_pages, void* v_pages, const int32_t* page_table,
                              const int32_t* prefix_lens, const int32_t* accept_path,
                              const int32_t* accept_len, int32_t* new_prefix_lens,
                              const treespec_attn_shape* shape, void* workspace, size_t workspace_bytes,
                              treespec_stream_t stream) {
    int rc = check_attn_shape(shape);
    if (rc != TREESPEC_OK) return rc;
    if (!k_pages || !v_pages || !page_table || !prefix_lens || !accept_path || !accept_len || !new_prefix_lens)
        return TREESPEC_ERR_NULL_POINTER;
    if (!aligned16(k_pages) || !aligned16(v_pages)) return TREESPEC_ERR_ALIGNMENT;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) ||
        workspace_bytes < treespec_commit_workspace_bytes())
        return TREESPEC_ERR_WORKSPACE;
    rc = check_device();
    if (rc != TREESPEC_OK) return rc;
    const treespec_attn_shape& s = *shape;
    CommitParams p{};
    p.k = k_pages;
    p.v = v_pages;
    p.page_table = page_table;
    p.prefix_lens = prefix_lens;
    p.path = accept_path;
    p.len = accept_len;
    p.new_lens = new_prefix_lens;
    p.status = static_cast<uint32_t*>(workspace);
    p.B = s.batch;
    p.N = s.num_nodes;
    p.Hkv = s.num_kv_heads;
    p.D = s.head_dim;
    p.ps = s.page_size;
    p.max_pages = s.max_pages_per_seq;
    p.num_pool_pages = s.num_pool_pages;
    p.elem = s.dtype == TREESPEC_DTYPE_BF16 ? 2 : 4;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    if (launch_kv_commit(p, st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    g_launches++;
    return TREESPEC_OK;
}

extern "C" size_t treespec_draft_workspace_bytes(int32_t batch, int32_t frontier, int32_t topk) {
    if (batch < 1 || batch > 65535 || frontier < 1 || frontier > kMaxFrontier || topk < 1 || topk > kMaxTopk)
        return 0;
    const size_t per = size_t(batch) * frontier * kMaxDraftSplits * topk;
    return kWsAlign + align_up(per * 4, kWsAlign) * 2;
}

extern "C" int tree_draft_step(const float* logprobs, int32_t batch, int32_t frontier, int32_t vocab,
                               int32_t topk, int32_t step, const int32_t* frontier_in, int32_t* node_parent,
                               int32_t* node_token, float* node_score, int32_t max_nodes, int32_t* frontier_out,
                               void* workspace, size_t workspace_bytes, treespec_stream_t stream) {
    if (batch < 1 || batch > 65535 || topk < 1 || topk > kMaxTopk || step < 0) return TREESPEC_ERR_SHAPE;
    if (frontier != (step == 0 ? 1 : topk)) return TREESPEC_ERR_SHAPE;
    if (vocab < topk || vocab > (1 << 30)) return TREESPEC_ERR_SHAPE;
    const long long base = step == 0 ? 1 : 1 + topk + (long long)(step - 1) * topk * topk;
    if (max_nodes > kMaxDraftNodes || base + (long long)frontier * topk > max_nodes) return TREESPEC_ERR_SHAPE;
    if ((long long)batch * frontier * vocab > (1ll << 40)) return TREESPEC_ERR_SHAPE;
    if (!logprobs || !node_parent || !node_token || !node_score || !frontier_out || (step > 0 && !frontier_in))
        return TREESPEC_ERR_NULL_POINTER;
    if (vocab % 4 == 0 && !aligned16(logprobs)) return TREESPEC_ERR_ALIGNMENT;
    const size_t need = treespec_draft_workspace_bytes(batch, frontier, topk);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) || workspace_bytes < need)
        return TREESPEC_ERR_WORKSPACE;
    int rc = check_device();
    if (rc != TREESPEC_OK) return rc;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const size_t per = size_t(batch) * frontier * kMaxDraftSplits * topk;
    DraftParams p{};
    p.logprobs = logprobs;
    p.frontier_in = frontier_in;
    p.frontier_out = frontier_out;
    p.node_parent = node_parent;
    p.node_token = node_token;
    p.node_score = node_score;
    p.status = reinterpret_cast<uint32_t*>(ws);
    p.tk_tok = reinterpret_cast<int32_t*>(ws + kWsAlign);
    p.tk_lp = reinterpret_cast<float*>(ws + kWsAlign + align_up(per * 4, kWsAlign));
    p.B = batch;
    p.F = frontier;
    p.V = vocab;
    p.k = topk;
    p.step = step;
    p.M = max_nodes;
    // A row's vocabulary is cut into S parts (one CTA each) only where the rows alone would
    // leave SMs idle: a CTA's lists filter best over a long stream (the floor rises and
    // fewer groups pass the vote), so parts cost more than they save once every SM has a
    // row (measured per step over 128256 tokens: 256 rows 36 us in one part, 41 in two;
    // 64 rows 23 us in one, 19 in two, 21 in four).  No part below 8192 tokens, parts a
    // multiple of 1024 tokens.
    {
        const long long rows = (long long)batch * frontier;
        long long S = sm_count_or_default() / rows;
        S = std::min<long long>(S, std::max<long long>(1, vocab / 8192));
        S = std::max<long long>(1, std::min<long long>(S, kMaxDraftSplits));
        long long chunk = (vocab + S - 1) / S;
        chunk = (chunk + 1023) / 1024 * 1024;
        p.S = int((vocab + chunk - 1) / chunk);
        p.chunk = int(chunk);
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the top-k kernel clears the status word (no memset: one stream operation fewer a step)
    if (launch_draft_step(p, st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    g_launches += 2;
    return TREESPEC_OK;
}

extern "C" int tree_rerank(const int32_t* node_parent, const int32_t* node_token, const float* node_score,
                           int32_t batch, int32_t max_nodes, int32_t num_nodes, int32_t* tree_parents,
                           int32_t* draft_tokens, void* workspace, size_t workspace_bytes,
                           treespec_stream_t stream) {
    return tree_rerank_pool(node_parent, node_token, node_score, nullptr, 0, batch, max_nodes, num_nodes,
                            tree_parents, draft_tokens, workspace, workspace_bytes, stream);
}

extern "C" int tree_rerank_pool(const int32_t* node_parent, const int32_t* node_token, const float* node_score,
                                const int32_t* pool, int32_t pool_size, int32_t batch, int32_t max_nodes,
                                int32_t num_nodes, int32_t* tree_parents, int32_t* draft_tokens, void* workspace,
                                size_t workspace_bytes, treespec_stream_t stream) {
    if (batch < 1 || batch > 65535 || max_nodes < 1 || max_nodes > kMaxDraftNodes) return TREESPEC_ERR_SHAPE;
    if (pool ? (pool_size < 1 || pool_size > kMaxDraftNodes) : pool_size != 0) return TREESPEC_ERR_SHAPE;
    if (num_nodes < 1 || num_nodes > kMaxNodes || num_nodes > max_nodes) return TREESPEC_ERR_SHAPE;
    if (!node_parent || !node_token || !node_score || !tree_parents || !draft_tokens)
        return TREESPEC_ERR_NULL_POINTER;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) || workspace_bytes < kWsAlign)
        return TREESPEC_ERR_WORKSPACE;
    int rc = check_device();
    if (rc != TREESPEC_OK) return rc;
    RerankParams p{};
    p.node_parent = node_parent;
    p.node_token = node_token;
    p.node_score = node_score;
    p.pool = pool;
    p.P = pool_size;
    p.parents = tree_parents;
    p.tokens = draft_tokens;
    p.status = static_cast<uint32_t*>(workspace);
    p.B = batch;
    p.M = max_nodes;
    p.N = num_nodes;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(p.status, 0, sizeof(uint32_t), st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    if (launch_rerank(p, st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    g_launches++;
    return TREESPEC_OK;
}

extern "C" int treespec_read_status(const void* workspace, uint32_t* status, treespec_stream_t stream) {
    if (!workspace || !status) return TREESPEC_ERR_NULL_POINTER;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return TREESPEC_ERR_LAUNCH;
    if (cudaMemcpy(status, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return TREESPEC_ERR_LAUNCH;
    return TREESPEC_OK;
}

extern "C" const char* treespec_error_string(int code) {
    switch (code) {
        case TREESPEC_OK: return "ok";
        case TREESPEC_ERR_NULL_POINTER: return "a required pointer is NULL";
        case TREESPEC_ERR_SHAPE: return "a size is outside the supported range";
        case TREESPEC_ERR_DTYPE: return "unsupported dtype or kernel for this dtype";
        case TREESPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case TREESPEC_ERR_SAMPLING: return "invalid temperature, or sampling inputs missing";
        case TREESPEC_ERR_ALIGNMENT: return "a tensor is not 16-byte aligned";
        case TREESPEC_ERR_DEVICE: return "no usable sm_103 CUDA device";
        case TREESPEC_ERR_LAUNCH: return "the CUDA runtime rejected a launch";
        default: return "unknown error code";
    }
}

extern "C" int treespec_version(void) { return 100; }

extern "C" uint64_t treespec_launch_count(void) { return g_launches.load(); }

extern "C" void treespec_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

extern "C" int treespec_last_launch_error(const char** name) {
    const int e = g_launch_error.load();
    if (name) *name = cudaGetErrorName(cudaError_t(e));
    return e;
}
