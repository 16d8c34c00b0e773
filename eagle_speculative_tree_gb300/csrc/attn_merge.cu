// Merge of split-KV partial states into the attention output.
//
// Each split s of a (sequence, kv head, row) holds m_s (running max of the log2-scaled
// scores), l_s = sum 2^(s - m_s) and acc_s = sum 2^(s - m_s) V.  Softmax over the union
// of the splits' tokens is
//     m = max_s m_s,  out = sum_s 2^(m_s - m) acc_s / sum_s 2^(m_s - m) l_s,
// which is the single pass of "Tech Radar: SGLang EAGLE-2", section 2, computed in
// pieces.  Splits beyond the sequence's own length were never run and are not read.
#include "common.cuh"

namespace treespec {

namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(AttnParams p) {
    constexpr int DS = D / 32;
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long total = (long long)p.B * p.Hkv * p.R;
    if (gw >= total) return;
    const int row = int(gw % p.R);
    const int bh = int(gw / p.R);
    const int h = bh % p.Hkv, b = bh / p.Hkv;
    const int i = row / p.G, hq = h * p.G + row % p.G;
    const size_t out_base = ((size_t(b) * p.N + i) * p.Hq + hq) * D + lane * DS;
    const int S = p.lens[b];
    float acc[DS];
#pragma unroll
    for (int e = 0; e < DS; ++e) acc[e] = 0.f;
    const int nb = p.nn[b];
    if (S >= 0 && i < nb) {                // padding rows (nodes nb..) are zero
        const int L = S + nb;
        const int nvalid = min(p.num_splits, (L + p.split_tokens - 1) / p.split_tokens);
        const size_t base = size_t(bh) * p.num_splits * p.R + row;   // + s * R
        float mm = -INFINITY;
        for (int s = 0; s < nvalid; ++s) mm = fmaxf(mm, p.part_ml[(base + size_t(s) * p.R) * 2]);
        float lsum = 0.f;
        for (int s = 0; s < nvalid; ++s) {
            const size_t pr = base + size_t(s) * p.R;
            const float ms = p.part_ml[pr * 2];
            if (ms == -INFINITY) continue;
            const float f = exp2f(ms - mm);
            lsum = fmaf(p.part_ml[pr * 2 + 1], f, lsum);
            const float* src = p.part_acc + pr * D + lane * DS;
#pragma unroll
            for (int e = 0; e < DS; ++e) acc[e] = fmaf(src[e], f, acc[e]);
        }
        const float inv = 1.f / lsum;
#pragma unroll
        for (int e = 0; e < DS; ++e) acc[e] *= inv;
    }
#pragma unroll
    for (int e = 0; e < DS; ++e) {
        if constexpr (sizeof(T) == 4) reinterpret_cast<float*>(p.out)[out_base + e] = acc[e];
        else reinterpret_cast<uint16_t*>(p.out)[out_base + e] = f32_to_bf16_rne(acc[e]);
    }
}

template <typename T, int D>
cudaError_t launch_typed(const AttnParams& p, cudaStream_t s) {
    const long long warps = (long long)p.B * p.Hkv * p.R;
    const long long blocks = (warps * 32 + 255) / 256;
    attn_merge_kernel<T, D><<<unsigned(blocks), 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_merge(const AttnParams& p, int dtype, cudaStream_t s) {
    if (dtype == TREESPEC_DTYPE_F32)
        return p.D == 64 ? launch_typed<float, 64>(p, s) : launch_typed<float, 128>(p, s);
    return p.D == 64 ? launch_typed<uint16_t, 64>(p, s) : launch_typed<uint16_t, 128>(p, s);
}

}  // namespace treespec
