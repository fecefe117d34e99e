// attn_bwd.cu -- backward of the tree-masked GQA attention on CUDA cores (fp32 arithmetic).
//
// The draft is trained on every accepted and rejected branch of its trees in one batched forward and
// backward pass ("Aurora" post, section 2), so the tree attention of that pass needs its gradient under the
// same ancestor mask.  With P recomputed from the forward's log-sum-exp (p_j = exp(s_j - lse)), the upstream
// gradient dO and delta = <dO, O> per query row:
//     dp_j = <dO, v_j>,  ds_j = p_j (dp_j - delta),  dq = scale sum_j ds_j k_j,
//     dk_j = scale sum_rows ds_j q,  dv_j = sum_rows p_j dO.
// Kernel 1 (dq): one CTA per (tree node, kv head, request) over the node's allowed positions, 32 per step,
//   like the CUDA-core forward; it also writes delta of its rows for kernel 2.
// Kernel 2 (dk, dv): one CTA per 16 consecutive cache positions of a (request, kv head); its four warps
//   split the query rows that can see those positions and keep 16 x D/32 accumulators per lane; the 16 dot
//   products of a row are reduced across the warp by recursive halving (16 shuffles per product instead
//   of 80), and the warps' partial sums meet in shared memory at the end.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kThreads = 128;
constexpr int kTileQ = 32;    // positions per step of the dq kernel
constexpr int kTileKV = 16;   // positions per CTA of the dk / dv kernel
constexpr float kLog2e = 1.4426950408889634f;

// The allowed positions of node t: the prefix [0, L) then the cache slots L + a of its ancestors a (itself
// and the root included), root first.  Returns their count; the ancestor slots land in s_anc.
__device__ __forceinline__ int node_positions(const int32_t* s_par, int t, int L, int32_t* s_anc) {
    int n = 0;
    for (int x = t; x >= 0; x = s_par[x]) ++n;
    int k = n;
    for (int x = t; x >= 0; x = s_par[x]) s_anc[--k] = L + x;
    return n;
}

template <int QDT, int KVDT>
__global__ void __launch_bounds__(kThreads) attn_bwd_dq_kernel(AttnBwdArgs a, float scale) {
    using QE = Elem<QDT>;
    using KE = Elem<KVDT>;
    extern __shared__ float smem[];
    const int G = a.Hq / a.Hkv, D = a.D;
    const int t = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    float* qs = smem;                       // [G][D]
    float* gs = qs + G * D;                 // [G][D]  dO
    float* dqs = gs + G * D;                // [G][D]  accumulators
    float* ks = dqs + G * D;                // [kTileQ][D+4]: rows 16-byte aligned for float4 reads
    float* vs = ks + kTileQ * (D + 4);      // [kTileQ][D+4]
    float* lses = vs + kTileQ * (D + 4);    // [G]  lse * log2(e)
    float* dls = lses + G;                  // [G]  delta
    __shared__ int32_t s_par[SV_MAX_T];
    __shared__ int32_t s_anc[SV_MAX_T];
    __shared__ int s_nanc;

    const int T = a.T;
    for (int i = tid; i < T; i += kThreads) s_par[i] = a.parent[(size_t)b * T + i];
    __syncthreads();
    const int L = a.kv_len[b];
    int st = block_tree_check(s_par, T);
    if (st == SV_OK && (L < 0 || L + T > a.kv_cap)) st = SV_ERR_INVALID_ARG;
    const size_t row0 = ((size_t)b * T + t) * a.Hq + (size_t)hk * G;
    if (st != SV_OK) {
        for (int i = tid; i < G * D; i += kThreads) a.dq[row0 * D + i] = 0.f;
        for (int g = tid; g < G; g += kThreads) a.delta[row0 + g] = 0.f;
        if (a.status && t == 0 && hk == 0 && tid == 0) a.status[b] = st;
        return;
    }
    if (a.status && t == 0 && hk == 0 && tid == 0) a.status[b] = SV_OK;
    if (tid == 0) s_nanc = node_positions(s_par, t, L, s_anc);
    const typename QE::T* q = (const typename QE::T*)a.q;
    const typename QE::T* go = (const typename QE::T*)a.dout;
    const typename QE::T* o = (const typename QE::T*)a.out;
    for (int i = tid; i < G * D; i += kThreads) {
        qs[i] = QE::get(q, row0 * D + i);
        gs[i] = QE::get(go, row0 * D + i);
        dqs[i] = 0.f;
    }
    __syncthreads();
    // delta = <dO, O> per query row, one warp per row
    for (int g = warp; g < G; g += kThreads / 32) {
        float acc = 0.f;
        for (int d = lane; d < D; d += 32) acc = fmaf(gs[g * D + d], QE::get(o, (row0 + g) * D + d), acc);
        acc = warp_sum(acc);
        if (lane == 0) {
            dls[g] = acc;
            lses[g] = a.lse[row0 + g] * kLog2e;
            a.delta[row0 + g] = acc;
        }
    }
    __syncthreads();

    const typename KE::T* kp = (const typename KE::T*)a.k + ((size_t)b * a.Hkv + hk) * (size_t)a.kv_cap * D;
    const typename KE::T* vp = (const typename KE::T*)a.v + ((size_t)b * a.Hkv + hk) * (size_t)a.kv_cap * D;
    const int npos = L + s_nanc;
    const float sl2 = scale * kLog2e;
    for (int start = 0; start < npos; start += kTileQ) {
        // all loads of a batch are issued before any is used, so a tile costs one memory round trip
        constexpr int kBatch = 16;
        for (int base = 0; base < kTileQ * D; base += kThreads * kBatch) {
            float kx[kBatch], vx[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kThreads + tid;
                const int r = i / D, d = i - r * D;
                const int j = start + r;
                kx[u] = 0.f;
                vx[u] = 0.f;
                if (i < kTileQ * D && j < npos) {
                    const size_t pos = (size_t)(j < L ? j : s_anc[j - L]);
                    kx[u] = KE::get(kp, pos * D + d);
                    vx[u] = KE::get(vp, pos * D + d);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int i = base + u * kThreads + tid;
                if (i < kTileQ * D) {
                    const int r = i / D, d = i - r * D;
                    ks[r * (D + 4) + d] = kx[u];
                    vs[r * (D + 4) + d] = vx[u];
                }
            }
        }
        __syncthreads();
        for (int g = warp; g < G; g += kThreads / 32) {
            float ds = 0.f;
            if (start + lane < npos) {
                const float* qr = qs + g * D;
                const float* gr = gs + g * D;
                const float* kr = ks + lane * (D + 4);
                const float* vr = vs + lane * (D + 4);
                float s0 = 0.f, s1 = 0.f, p0 = 0.f, p1 = 0.f;
                for (int d = 0; d < D; d += 4) {   // D is a multiple of 32
                    const float4 qa = *reinterpret_cast<const float4*>(qr + d);
                    const float4 ka = *reinterpret_cast<const float4*>(kr + d);
                    const float4 ga = *reinterpret_cast<const float4*>(gr + d);
                    const float4 va = *reinterpret_cast<const float4*>(vr + d);
                    s0 = fmaf(qa.x, ka.x, s0); s1 = fmaf(qa.y, ka.y, s1);
                    s0 = fmaf(qa.z, ka.z, s0); s1 = fmaf(qa.w, ka.w, s1);
                    p0 = fmaf(ga.x, va.x, p0); p1 = fmaf(ga.y, va.y, p1);
                    p0 = fmaf(ga.z, va.z, p0); p1 = fmaf(ga.w, va.w, p1);
                }
                const float p = exp2f(fmaf(s0 + s1, sl2, -lses[g]));
                ds = p * ((p0 + p1) - dls[g]);
            }
            for (int d = lane; d < D; d += 32) {
                float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
                for (int j = 0; j < kTileQ; j += 2) {
                    acc0 = fmaf(__shfl_sync(0xffffffffu, ds, j), ks[j * (D + 4) + d], acc0);
                    acc1 = fmaf(__shfl_sync(0xffffffffu, ds, j + 1), ks[(j + 1) * (D + 4) + d], acc1);
                }
                dqs[g * D + d] += acc0 + acc1;
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < G * D; i += kThreads) a.dq[row0 * D + i] = dqs[i] * scale;
}

// 16 per-lane partial sums -> lane l holds the warp-wide total of value (l >> 1): recursive halving, each
// round trading half of the values with the partner lane
__device__ __forceinline__ float reduce16(float (&v)[kTileKV], int lane) {
#pragma unroll
    for (int half = 8, off = 16; half >= 1; half >>= 1, off >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int m = 0; m < half; ++m) {
            const float send = hi ? v[m] : v[m + half];
            const float keep = hi ? v[m + half] : v[m];
            v[m] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

template <int QDT, int KVDT, int DL>
__global__ void __launch_bounds__(kThreads) attn_bwd_dkv_kernel(AttnBwdArgs a, float scale) {
    using QE = Elem<QDT>;
    using KE = Elem<KVDT>;
    constexpr int D = DL * 32;
    constexpr int NW = kThreads / 32;
    static_assert(NW == 4, "four warps");
    __shared__ float ks[kTileKV][D];
    __shared__ float vs[kTileKV][D];
    __shared__ float red[kTileKV][D];           // the warps' sums, dk then dv
    __shared__ int32_t s_par[SV_MAX_T];
    __shared__ unsigned long long s_anc[SV_MAX_T];
    const int G = a.Hq / a.Hkv, T = a.T;
    const int j0 = blockIdx.x * kTileKV, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.kv_len[b];
    for (int i = tid; i < T; i += kThreads) s_par[i] = a.parent[(size_t)b * T + i];
    __syncthreads();
    int st = block_tree_check(s_par, T);
    if (st != SV_OK || L < 0 || L + T > a.kv_cap || j0 >= L + T) return;   // kernel 1 reports the status
    if (tid == 0)
        for (int i = 0; i < T; ++i) s_anc[i] = (1ull << i) | (i ? s_anc[s_par[i]] : 0ull);
    const size_t kvrow0 = ((size_t)b * a.Hkv + hk) * (size_t)a.kv_cap;
    const typename KE::T* kp = (const typename KE::T*)a.k + kvrow0 * D;
    const typename KE::T* vp = (const typename KE::T*)a.v + kvrow0 * D;
    const int nj = min(kTileKV, L + T - j0);
    for (int i = tid; i < kTileKV * D; i += kThreads) {
        const int r = i / D, d = i - r * D;
        const bool ok = r < nj;
        ks[r][d] = ok ? KE::get(kp, (size_t)(j0 + r) * D + d) : 0.f;
        vs[r][d] = ok ? KE::get(vp, (size_t)(j0 + r) * D + d) : 0.f;
    }
    __syncthreads();
    // tree slots of this tile as a bit mask over node ids; prefix positions are seen by every row
    const bool has_prefix = j0 < L;
    unsigned long long tile_tree = 0;
    for (int r = 0; r < nj; ++r) if (j0 + r >= L) tile_tree |= 1ull << (j0 + r - L);

    float dk[kTileKV][DL], dv[kTileKV][DL];
#pragma unroll
    for (int j = 0; j < kTileKV; ++j)
#pragma unroll
        for (int m = 0; m < DL; ++m) { dk[j][m] = 0.f; dv[j][m] = 0.f; }
    const typename QE::T* q = (const typename QE::T*)a.q;
    const typename QE::T* go = (const typename QE::T*)a.dout;
    const float sl2 = scale * kLog2e;
    // each warp walks its rows with the next row's q, dO, lse and delta already in flight
    const int TG = T * G;
    float qn[DL], gn[DL], lsen = 0.f, dln = 0.f;
    auto fetch = [&](int rr) {
        const int i = rr / G, g = rr - i * G;
        const size_t row = ((size_t)b * T + i) * a.Hq + (size_t)hk * G + g;
#pragma unroll
        for (int m = 0; m < DL; ++m) {
            qn[m] = QE::get(q, row * D + lane + 32 * m);
            gn[m] = QE::get(go, row * D + lane + 32 * m);
        }
        lsen = a.lse[row];
        dln = a.delta[row];
    };
    if (warp < TG) fetch(warp);
    for (int rr = warp; rr < TG; rr += NW) {
        const int i = rr / G;
        float qv[DL], gv[DL];
#pragma unroll
        for (int m = 0; m < DL; ++m) { qv[m] = qn[m]; gv[m] = gn[m]; }
        const float lse_r = lsen, delta_r = dln;
        if (rr + NW < TG) fetch(rr + NW);
        const unsigned long long anc = s_anc[i];
        if (!has_prefix && !(anc & tile_tree)) continue;   // the row sees none of these positions
        float sp[kTileKV], dpp[kTileKV];
#pragma unroll
        for (int j = 0; j < kTileKV; ++j) {
            float s = 0.f, dp = 0.f;
#pragma unroll
            for (int m = 0; m < DL; ++m) {
                s = fmaf(qv[m], ks[j][lane + 32 * m], s);
                dp = fmaf(gv[m], vs[j][lane + 32 * m], dp);
            }
            sp[j] = s;
            dpp[j] = dp;
        }
        const float s_tot = reduce16(sp, lane);     // position lane >> 1 of the tile
        const float dp_tot = reduce16(dpp, lane);
        const int jl = lane >> 1, jabs = j0 + jl;
        const bool allowed = jl < nj && (jabs < L || ((anc >> (jabs - L)) & 1ull));
        const float p = allowed ? exp2f(fmaf(s_tot, sl2, -lse_r * kLog2e)) : 0.f;
        const float ds = p * (dp_tot - delta_r);
#pragma unroll
        for (int j = 0; j < kTileKV; ++j) {
            const float pj = __shfl_sync(0xffffffffu, p, 2 * j);
            const float dsj = __shfl_sync(0xffffffffu, ds, 2 * j);
#pragma unroll
            for (int m = 0; m < DL; ++m) {
                dv[j][m] = fmaf(pj, gv[m], dv[j][m]);
                dk[j][m] = fmaf(dsj, qv[m], dk[j][m]);
            }
        }
    }
    // the warps' partial sums meet in shared memory in warp order (deterministic), dk then dv
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        for (int w = 0; w < NW; ++w) {
            if (warp == w) {
#pragma unroll
                for (int j = 0; j < kTileKV; ++j)
#pragma unroll
                    for (int m = 0; m < DL; ++m) {
                        const float x = pass == 0 ? dk[j][m] : dv[j][m];
                        red[j][lane + 32 * m] = w == 0 ? x : red[j][lane + 32 * m] + x;
                    }
            }
            __syncthreads();
        }
        float* outp = (pass == 0 ? a.dk : a.dv) + (kvrow0 + j0) * D;
        for (int i = tid; i < nj * D; i += kThreads) {
            const int r = i / D, d = i - r * D;
            outp[i] = pass == 0 ? red[r][d] * scale : red[r][d];
        }
        __syncthreads();
    }
}

template <int QDT, int KVDT>
cudaError_t launch_typed(const AttnBwdArgs& a, cudaStream_t s) {
    const int G = a.Hq / a.Hkv;
    const size_t smem = sizeof(float) * ((size_t)3 * G * a.D + (size_t)2 * kTileQ * (a.D + 4) + 2 * G);
    auto k1 = attn_bwd_dq_kernel<QDT, KVDT>;
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    k1<<<dim3(a.T, a.Hkv, a.B), kThreads, smem, s>>>(a, scale);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 g2((a.kv_cap + kTileKV - 1) / kTileKV, a.Hkv, a.B);
    switch (a.D) {
    case 32: attn_bwd_dkv_kernel<QDT, KVDT, 1><<<g2, kThreads, 0, s>>>(a, scale); break;
    case 64: attn_bwd_dkv_kernel<QDT, KVDT, 2><<<g2, kThreads, 0, s>>>(a, scale); break;
    default: attn_bwd_dkv_kernel<QDT, KVDT, 4><<<g2, kThreads, 0, s>>>(a, scale); break;
    }
    return cudaGetLastError();
}

}  // namespace

size_t attn_bwd_workspace_size(int B, int T, int Hq) {
    return ((size_t)B * T * Hq * sizeof(float) + 255) / 256 * 256;
}

// the tensor-core kernels (attn_bwd_tc.cu)
bool attn_bwd_tc_supported(const AttnBwdArgs& a);
cudaError_t launch_attn_bwd_tc(const AttnBwdArgs& a, cudaStream_t s);

cudaError_t launch_attn_bwd(const AttnBwdArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    if (attn_bwd_tc_supported(a)) return launch_attn_bwd_tc(a, s);   // bf16, D = 128: tensor cores
    if (a.q_dt == SV_F32) return a.kv_dt == SV_F32 ? launch_typed<SV_F32, SV_F32>(a, s) : launch_typed<SV_F32, SV_BF16>(a, s);
    return a.kv_dt == SV_F32 ? launch_typed<SV_BF16, SV_F32>(a, s) : launch_typed<SV_BF16, SV_BF16>(a, s);
}

}  // namespace sv
