// Split-KV paged tree attention on CUDA cores (any dtype; the path for fewer than
// 64 query rows per kv head and for float32).
//
// What one CTA computes: for sequence b, kv head h, a block of up to 64 query rows
// (row r = node i * G + g, i.e. query head h*G + g of node i) and one contiguous
// range of logical tokens (a "split"), the flash-style partial state
//     m_r = max_t s_rt,  l_r = sum_t 2^(s_rt - m_r),  acc_r = sum_t 2^(s_rt - m_r) V_t
// with s_rt = log2(e)/sqrt(D) * q_r . K_t over the tokens row r may see: every
// prefix token, and tree token S + j only if node i's ancestor-or-self set holds j
// ("Tech Radar: SGLang EAGLE-2", section 2 mask M; section 5 item 1 bitmask test).
// The kernel streams each K/V page of its split once through shared memory for all
// of its rows (the siblings' shared prefix is read once, section 5 item 3), in
// 32*TS-token tiles with a two-stage cp.async pipeline.
//
// Warp layout: RW row-warps (8 rows each) x TS token-slices (32 tokens each).
//   QK^T: lane = token, the 8 scores of its rows accumulate over D.
//   softmax: per-row max by warp shuffles, exp2, running (m, l) per row.
//   PV:   lane = D/32-wide slice of the head dimension, probabilities broadcast from
//         shared memory, 8 x D/32 accumulators per lane.
// Token-slices of one CTA are merged in shared memory at the end.
#include "common.cuh"

namespace treespec {

namespace {

template <typename T, int D>
struct SimtCfg {
    static constexpr int EB = int(sizeof(T));
    static constexpr int EPV = 16 / EB;          // elements per 16-byte vector
    static constexpr int VPR = D * EB / 16;      // 16-byte vectors per K/V row
    static constexpr int ROWB = D * EB + 16;     // padded shared-memory row (bank spread)
    static constexpr int DS = D / 32;            // head-dim elements per lane in PV
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, int src_bytes) {
    unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(gsrc),
                 "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

template <typename T>
__device__ __forceinline__ void vec_to_f32(const uint4& v, float* f);
template <>
__device__ __forceinline__ void vec_to_f32<float>(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void vec_to_f32<uint16_t>(const uint4& v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// DS consecutive elements of one V row -> floats.
template <typename T, int DS>
__device__ __forceinline__ void load_slice(const unsigned char* src, float* f) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (DS == 4) {
            float4 v = *reinterpret_cast<const float4*>(src);
            f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
        } else {
            float2 v = *reinterpret_cast<const float2*>(src);
            f[0] = v.x; f[1] = v.y;
        }
    } else {
        if constexpr (DS == 4) {
            uint2 v = *reinterpret_cast<const uint2*>(src);
            f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        } else {
            uint32_t v = *reinterpret_cast<const uint32_t*>(src);
            f[0] = bf16_lo(v); f[1] = bf16_hi(v);
        }
    }
}

template <typename T>
__device__ __forceinline__ float load_q(const void* q, size_t idx) {
    if constexpr (sizeof(T) == 4) return reinterpret_cast<const float*>(q)[idx];
    else return bf16_to_f32(reinterpret_cast<const uint16_t*>(q)[idx]);
}
template <typename T>
__device__ __forceinline__ void store_out(void* out, size_t idx, float v) {
    if constexpr (sizeof(T) == 4) reinterpret_cast<float*>(out)[idx] = v;
    else reinterpret_cast<uint16_t*>(out)[idx] = f32_to_bf16_rne(v);
}

struct SimtShape {
    int RW, TS, nwarps, TT;
    size_t qs_bytes, stage_bytes, kv_bytes, pt_bytes, smem;
};

template <typename T, int D>
__host__ __device__ inline SimtShape simt_shape(int rows_block) {
    using C = SimtCfg<T, D>;
    SimtShape s;
    s.RW = rows_block <= 8 ? 1 : rows_block <= 16 ? 2 : rows_block <= 32 ? 4 : 8;
    int ts_budget = int((160u * 1024u) / (4u * 32u * C::ROWB));   // two stages of K and V
    int ts = 8 / s.RW;
    if (ts > 4) ts = 4;
    if (ts > ts_budget) ts = ts_budget < 1 ? 1 : ts_budget;
    s.TS = ts;
    s.nwarps = s.RW * s.TS;
    s.TT = 32 * s.TS;
    s.qs_bytes = size_t(s.RW) * 8 * D * 4;
    s.stage_bytes = size_t(2) * s.TT * C::ROWB;
    size_t scratch = size_t(s.nwarps) * 8 * (D + 2) * 4;
    s.kv_bytes = 2 * s.stage_bytes > scratch ? 2 * s.stage_bytes : scratch;
    s.pt_bytes = size_t(s.nwarps) * 32 * 8 * 4;
    s.smem = s.qs_bytes + s.kv_bytes + s.pt_bytes + kMaxNodes * kAncWords * 8;
    return s;
}

template <typename T, int D>
__global__ void __launch_bounds__(256) attn_simt_kernel(AttnParams p) {
    using C = SimtCfg<T, D>;
    constexpr int DS = C::DS;
    extern __shared__ __align__(16) unsigned char smem[];
    const SimtShape sh = simt_shape<T, D>(p.rows_per_block);
    const int RW = sh.RW, TS = sh.TS, TT = sh.TT, nthr = sh.nwarps * 32;
    float* Qs = reinterpret_cast<float*>(smem);
    unsigned char* kv = smem + sh.qs_bytes;
    float* Pt = reinterpret_cast<float*>(kv + sh.kv_bytes);
    uint64_t* anc_s = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(Pt) + sh.pt_bytes);

    const int split = blockIdx.x;
    const int h = blockIdx.y / p.row_blocks, rb = blockIdx.y % p.row_blocks;
    const int b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rw = warp % RW, ts = warp / RW;
    const int r0 = rb * p.rows_per_block;
    const int rows = min(p.rows_per_block, p.R - r0);
    const int S = p.lens[b];

    if (S < 0) {                           // invalid sequence: zeros (the merge does it otherwise)
        if (!p.merge && split == 0) {
            for (int e = tid; e < rows * D; e += nthr) {
                int row = r0 + e / D, d = e % D;
                int i = row / p.G, hq = h * p.G + row % p.G;
                store_out<T>(p.out, ((size_t(b) * p.N + i) * p.Hq + hq) * D + d, 0.f);
            }
        }
        return;
    }
    const int nb = p.nn[b];               // rows of nodes nb.. are padding: zero output
    const int L = S + nb;
    const int t0 = split * p.split_tokens;
    const int t1 = min(L, t0 + p.split_tokens);
    if (t0 >= t1) return;

    for (int e = tid; e < RW * 8 * D; e += nthr) {
        int lr = e / D, d = e % D;
        float v = 0.f;
        if (lr < rows) {
            int row = r0 + lr;
            int i = row / p.G, hq = h * p.G + row % p.G;
            if (i < nb) v = load_q<T>(p.q, ((size_t(b) * p.N + i) * p.Hq + hq) * D + d) * p.scale_log2;
        }
        Qs[e] = v;
    }
    for (int e = tid; e < p.N * kAncWords; e += nthr) anc_s[e] = p.anc[size_t(b) * p.N * kAncWords + e];

    const int* ptab = p.page_table + size_t(b) * p.max_pages;
    auto issue = [&](int tile, int stage) {
        const int base = t0 + tile * TT;
        unsigned char* Kd = kv + stage * sh.stage_bytes;
        unsigned char* Vd = Kd + size_t(TT) * C::ROWB;
        for (int e = tid; e < TT * C::VPR; e += nthr) {
            const int tt = e / C::VPR, vi = e % C::VPR;
            const int pos = base + tt;
            const unsigned char* ks = static_cast<const unsigned char*>(p.k);
            const unsigned char* vs = static_cast<const unsigned char*>(p.v);
            int bytes = 0;
            if (pos < t1) {
                const int page = ptab[pos / p.ps];
                if (page >= 0 && page < p.num_pool_pages) {
                    size_t off = ((size_t(page) * p.ps + pos % p.ps) * p.Hkv + h) * (size_t(D) * C::EB) +
                                 size_t(vi) * 16;
                    ks += off;
                    vs += off;
                    bytes = 16;
                } else if (vi == 0) {
                    atomicOr(p.status, TREESPEC_STATUS_BAD_PAGE);
                }
            }
            cp_async16(Kd + tt * C::ROWB + vi * 16, ks, bytes);
            cp_async16(Vd + tt * C::ROWB + vi * 16, vs, bytes);
        }
    };

    float m[8], l[8], acc[8][DS];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < DS; ++e) acc[r][e] = 0.f;
    }
    const bool has_rows = rw * 8 < rows;
    const int ntiles = (t1 - t0 + TT - 1) / TT;
    float* pt_w = Pt + warp * 256;

    issue(0, 0);
    cp_async_commit();
    for (int tile = 0; tile < ntiles; ++tile) {
        if (tile + 1 < ntiles) issue(tile + 1, (tile + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (has_rows) {
            const unsigned char* Kd = kv + (tile & 1) * sh.stage_bytes;
            const unsigned char* Vd = Kd + size_t(TT) * C::ROWB;
            const int tt = ts * 32 + lane;
            const int pos = t0 + tile * TT + tt;
            // ---- scores for 8 rows x this lane's token
            float s[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) s[r] = 0.f;
            const unsigned char* krow = Kd + tt * C::ROWB;
            const float* qbase = Qs + rw * 8 * D;
#pragma unroll 4
            for (int d = 0; d < D; d += C::EPV) {
                float kf[C::EPV];
                vec_to_f32<T>(*reinterpret_cast<const uint4*>(krow + d * C::EB), kf);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float* qr = qbase + r * D + d;
#pragma unroll
                    for (int e = 0; e < C::EPV; e += 4) {
                        float4 qv = *reinterpret_cast<const float4*>(qr + e);
                        s[r] = fmaf(qv.x, kf[e], s[r]);
                        s[r] = fmaf(qv.y, kf[e + 1], s[r]);
                        s[r] = fmaf(qv.z, kf[e + 2], s[r]);
                        s[r] = fmaf(qv.w, kf[e + 3], s[r]);
                    }
                }
            }
            // ---- tree mask + online softmax
            const bool tok_ok = pos < t1;
            const int j = pos - S;                 // tree node index when >= 0 (then < N)
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int lr = rw * 8 + r;
                bool ok = tok_ok && lr < rows;
                if (ok && j >= 0) ok = (anc_s[(r0 + lr) / p.G * kAncWords + (j >> 6)] >> (j & 63)) & 1ull;
                const float sv = ok ? s[r] : -INFINITY;
                const float mnew = fmaxf(m[r], warp_max(sv));
                const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m[r] - mnew);
                const float pv = ok ? exp2f(sv - mnew) : 0.f;
                l[r] = fmaf(l[r], alpha, pv);
                m[r] = mnew;
#pragma unroll
                for (int e = 0; e < DS; ++e) acc[r][e] *= alpha;
                pt_w[lane * 8 + r] = pv;
            }
            __syncwarp();
            // ---- P V over the warp's 32 tokens
            const unsigned char* vrow = Vd + size_t(ts * 32) * C::ROWB + lane * DS * C::EB;
#pragma unroll 4
            for (int t = 0; t < 32; ++t) {
                float vf[DS];
                load_slice<T, DS>(vrow + t * C::ROWB, vf);
                const float4 pa = *reinterpret_cast<const float4*>(pt_w + t * 8);
                const float4 pb = *reinterpret_cast<const float4*>(pt_w + t * 8 + 4);
                const float pr[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int e = 0; e < DS; ++e) acc[r][e] = fmaf(pr[r], vf[e], acc[r][e]);
            }
            __syncwarp();
        }
        __syncthreads();
    }
    cp_async_wait<0>();

#pragma unroll
    for (int r = 0; r < 8; ++r) l[r] = warp_sum(l[r]);
    __syncthreads();
    float* scr = reinterpret_cast<float*>(kv);          // [nwarps][8][D + 2]
    if (has_rows) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            float* dst = scr + size_t(warp * 8 + r) * (D + 2);
#pragma unroll
            for (int e = 0; e < DS; ++e) dst[lane * DS + e] = acc[r][e];
            if (lane == 0) {
                dst[D] = m[r];
                dst[D + 1] = l[r];
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < rows * D; e += nthr) {
        const int lr = e / D, d = e % D, rwi = lr / 8, r = lr % 8;
        float mm = -INFINITY;
        for (int t = 0; t < TS; ++t) mm = fmaxf(mm, scr[size_t((t * RW + rwi) * 8 + r) * (D + 2) + D]);
        float lsum = 0.f, a = 0.f;
        if (mm != -INFINITY) {
            for (int t = 0; t < TS; ++t) {
                const float* src = scr + size_t((t * RW + rwi) * 8 + r) * (D + 2);
                if (src[D] == -INFINITY) continue;
                const float f = exp2f(src[D] - mm);
                lsum = fmaf(src[D + 1], f, lsum);
                a = fmaf(src[d], f, a);
            }
        }
        const int row = r0 + lr;
        if (!p.merge) {
            const int i = row / p.G, hq = h * p.G + row % p.G;
            const bool present = i < *static_cast<volatile const int32_t*>(p.nn + b);   // re-read: not kept live
            store_out<T>(p.out, ((size_t(b) * p.N + i) * p.Hq + hq) * D + d, present ? a / lsum : 0.f);
        } else {
            const size_t pr = (size_t(b * p.Hkv + h) * p.num_splits + split) * p.R + row;
            p.part_acc[pr * D + d] = a;
            if (d == 0) {
                p.part_ml[pr * 2] = mm;
                p.part_ml[pr * 2 + 1] = lsum;
            }
        }
    }
}

template <typename T, int D>
cudaError_t launch_typed(const AttnParams& p, cudaStream_t s) {
    const SimtShape sh = simt_shape<T, D>(p.rows_per_block);
    auto kern = attn_simt_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sh.smem));
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.Hkv * p.row_blocks, p.B);
    kern<<<grid, sh.nwarps * 32, sh.smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t attn_simt_smem_bytes(int dtype, int D, int R_block) {
    if (dtype == TREESPEC_DTYPE_F32)
        return D == 64 ? simt_shape<float, 64>(R_block).smem : simt_shape<float, 128>(R_block).smem;
    return D == 64 ? simt_shape<uint16_t, 64>(R_block).smem : simt_shape<uint16_t, 128>(R_block).smem;
}

cudaError_t launch_attn_simt(const AttnParams& p, int dtype, cudaStream_t s) {
    if (dtype == TREESPEC_DTYPE_F32)
        return p.D == 64 ? launch_typed<float, 64>(p, s) : launch_typed<float, 128>(p, s);
    return p.D == 64 ? launch_typed<uint16_t, 64>(p, s) : launch_typed<uint16_t, 128>(p, s);
}

}  // namespace treespec
