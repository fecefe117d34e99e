// attn_simt.cu -- tree-masked GQA attention on CUDA cores (fp32 arithmetic), any supported dtype.
//
// Serves shapes outside the tensor-core kernel's envelope (float32 inputs, D other than 64/128, small
// problems) and is the fp32 cross-check of that kernel.  One CTA per (tree node, kv head, request) runs
// the G query heads of the group together over the node's allowed positions: the prefix [0, L) and the
// cache slots L + a of the node's ancestors a ("Aurora" post, section 2: the tree-attention mask follows
// the speculative tree's causal structure).  Online softmax in the log2 domain, 32 positions per step.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kThreads = 128;
constexpr int kTile = 32;

template <int QDT, int KVDT>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(AttnArgs a, float scale_log2) {
    using QE = Elem<QDT>;
    using KE = Elem<KVDT>;
    extern __shared__ float smem[];
    const int G = a.Hq / a.Hkv, D = a.D;
    const int t = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    float* qs = smem;                       // [G][D]
    float* os = qs + G * D;                 // [G][D]
    float* ks = os + G * D;                 // [kTile][D+1]
    float* vs = ks + kTile * (D + 1);       // [kTile][D]
    float* ms = vs + kTile * D;             // [G]
    float* ls = ms + G;                     // [G]
    __shared__ int32_t s_par[SV_MAX_T];
    __shared__ int32_t s_anc[SV_MAX_T];
    __shared__ int s_nanc;

    const int T = a.T;
    for (int i = tid; i < T; i += kThreads) s_par[i] = a.parent[(size_t)b * T + i];
    __syncthreads();
    const int L = a.kv_len[b];
    int st = block_tree_check(s_par, T);
    if (st == SV_OK && (L < 0 || L + T > a.kv_cap)) st = SV_ERR_INVALID_ARG;
    const int32_t* pt = a.page_table ? a.page_table + (size_t)b * a.max_pages : nullptr;
    if (pt && st == SV_OK) {   // every page the request reads must name a page of the pool
        int bad = 0;
        for (int i = tid; i < ((L + T - 1) >> a.page_shift) + 1; i += kThreads) bad |= pt[i] < 0 || pt[i] >= a.num_pages;
        if (__syncthreads_or(bad)) st = SV_ERR_INVALID_ARG;
    }

    const size_t out_row0 = ((size_t)b * T + t) * a.Hq + (size_t)hk * G;
    if (st != SV_OK) {
        for (int i = tid; i < G * D; i += kThreads) {
            if (QDT == SV_F32) ((float*)a.out)[out_row0 * D + i] = 0.f;
            else ((uint16_t*)a.out)[out_row0 * D + i] = 0;
        }
        if (a.lse) for (int g = tid; g < G; g += kThreads) a.lse[out_row0 + g] = 0.f;
        if (a.status && t == 0 && hk == 0 && tid == 0) a.status[b] = st;
        return;
    }
    if (a.status && t == 0 && hk == 0 && tid == 0) a.status[b] = SV_OK;

    if (tid == 0) {   // ancestors of node t (itself and the root included), as cache positions
        int n = 0;
        for (int x = t; x >= 0; x = s_par[x]) s_anc[n++] = L + x;
        s_nanc = n;
    }
    const typename QE::T* q = (const typename QE::T*)a.q;
    for (int i = tid; i < G * D; i += kThreads) {
        qs[i] = QE::get(q, out_row0 * D + i);
        os[i] = 0.f;
    }
    for (int g = tid; g < G; g += kThreads) { ms[g] = -INFINITY; ls[g] = 0.f; }
    __syncthreads();

    const float ksc = (KVDT == SV_E4M3) ? a.k_scale[hk] : 1.f;
    const float vsc = (KVDT == SV_E4M3) ? a.v_scale[hk] : 1.f;
    // contiguous caches: the (request, kv head) block; paged caches: the pool, rows found through pt
    const size_t blk = pt ? 0 : ((size_t)b * a.Hkv + hk) * (size_t)a.kv_cap * D;
    const typename KE::T* kp = (const typename KE::T*)a.k + blk;
    const typename KE::T* vp = (const typename KE::T*)a.v + blk;
    const int pmask = (1 << a.page_shift) - 1;
    auto cache_row = [&](int pos) -> size_t {
        if (!pt) return (size_t)pos;
        return ((size_t)__ldg(pt + (pos >> a.page_shift)) * a.Hkv + hk) * (size_t)(pmask + 1) + (pos & pmask);
    };
    const int npos = L + s_nanc;

    for (int start = 0; start < npos; start += kTile) {
        // all loads of a batch are issued before any is used, so a tile costs one memory round trip
        constexpr int kBatch = 16;
        for (int base = 0; base < kTile * D; base += kThreads * kBatch) {
            float kv[kBatch], vv[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kThreads + tid;
                const int r = i / D, d = i - r * D;
                const int j = start + r;
                kv[u] = 0.f;
                vv[u] = 0.f;
                if (i < kTile * D && j < npos) {
                    const size_t row = cache_row(j < L ? j : s_anc[j - L]);
                    kv[u] = KE::get(kp, row * D + d);
                    vv[u] = KE::get(vp, row * D + d);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kThreads + tid;
                if (i < kTile * D) {
                    const int r = i / D, d = i - r * D;
                    ks[r * (D + 1) + d] = kv[u] * ksc;
                    vs[r * D + d] = vv[u] * vsc;
                }
            }
        }
        __syncthreads();
        for (int g = warp; g < G; g += kThreads / 32) {
            float s = -INFINITY;
            if (start + lane < npos) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};   // four independent chains
                const float* qr = qs + g * D;
                const float* kr = ks + lane * (D + 1);
                const int D4 = D & ~3;
                for (int d = 0; d < D4; d += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc[u] = fmaf(qr[d + u], kr[d + u], acc[u]);
                }
                for (int d = D4; d < D; ++d) acc[0] = fmaf(qr[d], kr[d], acc[0]);
                s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * scale_log2;
            }
            float m_old = ms[g];
            float m_new = fmaxf(m_old, warp_max(s));
            float p = (s == -INFINITY) ? 0.f : exp2f(s - m_new);
            float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
            float psum = warp_sum(p);
            for (int d = lane; d < D; d += 32) {
                float acc[4] = {os[g * D + d] * alpha, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < kTile; j += 4) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        acc[u] = fmaf(__shfl_sync(0xffffffffu, p, j + u), vs[(j + u) * D + d], acc[u]);
                }
                os[g * D + d] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            }
            __syncwarp();
            if (lane == 0) { ls[g] = ls[g] * alpha + psum; ms[g] = m_new; }
            __syncwarp();
        }
        __syncthreads();
    }

    for (int i = tid; i < G * D; i += kThreads) {
        int g = i / D;
        float o = os[i] / ls[g];
        if (QDT == SV_F32) ((float*)a.out)[out_row0 * D + i] = o;
        else ((uint16_t*)a.out)[out_row0 * D + i] = float_to_bf16_bits(o);
    }
    if (a.lse)
        for (int g = tid; g < G; g += kThreads) a.lse[out_row0 + g] = (ms[g] + log2f(ls[g])) * 0.69314718055994531f;
}

template <int QDT, int KVDT>
cudaError_t launch_typed(const AttnArgs& a, cudaStream_t s) {
    const int G = a.Hq / a.Hkv;
    size_t smem = sizeof(float) * ((size_t)2 * G * a.D + (size_t)kTile * (a.D + 1) + (size_t)kTile * a.D + 2 * G);
    auto kern = attn_simt_kernel<QDT, KVDT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    dim3 grid(a.T, a.Hkv, a.B);
    kern<<<grid, kThreads, smem, s>>>(a, scale * 1.4426950408889634f);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    if (a.q_dt == SV_F32) {
        if (a.kv_dt == SV_F32) return launch_typed<SV_F32, SV_F32>(a, s);
        if (a.kv_dt == SV_BF16) return launch_typed<SV_F32, SV_BF16>(a, s);
        return launch_typed<SV_F32, SV_E4M3>(a, s);
    }
    if (a.kv_dt == SV_F32) return launch_typed<SV_BF16, SV_F32>(a, s);
    if (a.kv_dt == SV_BF16) return launch_typed<SV_BF16, SV_BF16>(a, s);
    return launch_typed<SV_BF16, SV_E4M3>(a, s);
}

}  // namespace sv
