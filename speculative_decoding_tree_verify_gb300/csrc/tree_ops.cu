// tree_ops.cu -- the steps on either side of verification: KV compaction after acceptance, and one level
// of draft tree expansion before it.
//
// KV compaction ("Aurora" post, section 2, and TIDE overview: the target keeps the accepted continuation).
//   The root's K/V sit at cache position L (the first tree slot) and accepted node path[j] at L + path[j];
//   compaction moves path[j] to L + 1 + j so the committed tokens form a causal prefix of length
//   L + 1 + accept_len.  One CTA per (request, kv head); thread t owns one 16-byte column of the K or V
//   rows.  A path walks down the tree, so path[j] >= j + 1 and is increasing: the slot element j writes
//   (L + 1 + j) is never read by a later element, and the slot element j reads is never written by an
//   earlier one.  A thread therefore only has to read a batch of sources before writing that batch, and
//   the in-place copy needs no barrier and no staging buffer.
//
// Draft tree expansion (the draft proposes tokens that the target verifies in one pass: "Aurora" post,
//   section 2; TIDE overview).  Kernel 1: a thread-block cluster per frontier row, 128-bit loads, one pass
//   that keeps the running max / sum of exp (online softmax) and a per-thread sorted top-KT list;
//   warps, CTAs and the cluster merge their lists (distributed shared memory).  Kernel 2: one CTA per
//   request ranks the n_front * k candidates by path score and keeps the n_keep best in (slot, rank) order.
#include <cooperative_groups.h>

#include <atomic>

#include "sv_internal.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

// ------------------------------------------------------------------------------------ KV compaction
constexpr int kCompactBatch = 8;

__global__ void kv_compact_kernel(CompactArgs a, int chunks) {
    __shared__ int32_t s_par[SV_MAX_T];
    __shared__ int32_t s_path[SV_MAX_T];
    const int b = blockIdx.x / a.Hkv, hk = blockIdx.x % a.Hkv;
    const int T = a.T, tid = threadIdx.x;
    const int L = a.kv_len[b], n = a.accept_len[b];
    for (int i = tid; i < T; i += blockDim.x) {
        s_par[i] = a.parent[(size_t)b * T + i];
        s_path[i] = a.path[(size_t)b * T + i];
    }
    __syncthreads();
    int st = block_tree_check(s_par, T);
    if (st == SV_OK && (L < 0 || (long long)L + T > a.kv_cap || n < 0 || n > T - 1)) st = SV_ERR_INVALID_ARG;
    if (st == SV_OK) {
        int bad = 0;
        for (int j = tid; j < n; j += blockDim.x) {
            const int node = s_path[j], up = j == 0 ? 0 : s_path[j - 1];
            bad |= node < 1 || node >= T || s_par[node] != up;
        }
        if (__syncthreads_or(bad)) st = SV_ERR_INVALID_ARG;
    }
    if (hk == 0 && tid == 0) {
        a.new_kv_len[b] = st == SV_OK ? L + 1 + n : L;
        if (a.status) a.status[b] = st;
    }
    if (st != SV_OK || tid >= 2 * chunks) return;
    const int which = tid / chunks, c = tid % chunks;
    uint4* rows = (uint4*)(which ? a.v : a.k) + (((size_t)b * a.Hkv + hk) * a.kv_cap + L) * chunks + c;
    for (int j0 = 0; j0 < n; j0 += kCompactBatch) {
        uint4 buf[kCompactBatch];
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int j = j0 + u;
            if (j < n && s_path[j] != j + 1) buf[u] = rows[(size_t)s_path[j] * chunks];
        }
#pragma unroll
        for (int u = 0; u < kCompactBatch; ++u) {
            const int j = j0 + u;
            if (j < n && s_path[j] != j + 1) rows[(size_t)(j + 1) * chunks] = buf[u];
        }
    }
}

// ------------------------------------------------------------------------------------ tree expansion
constexpr int kExpThreads = 256;
constexpr int kExpMaxCluster = 8;
constexpr int kExpBatch = 4;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int LDT> struct Row;
template <> struct Row<SV_F32> {
    using T = float;
    static constexpr int kVec = 4;
    __device__ static void load_vec(const T* p, float* z) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        z[0] = v.x; z[1] = v.y; z[2] = v.z; z[3] = v.w;
    }
    __device__ static float load(const T* p) { return __ldg(p); }
};
template <> struct Row<SV_BF16> {
    using T = uint16_t;
    static constexpr int kVec = 8;
    __device__ static void load_vec(const T* p, float* z) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            z[2 * i] = __uint_as_float(w[i] << 16);
            z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static float load(const T* p) { return bf16_bits_to_float(__ldg(p)); }
};

// (value, index) order of the proposals: larger logit first, lower token id first on equal logits
__device__ __forceinline__ bool beats(float v, int i, float v2, int i2) { return v > v2 || (v == v2 && i < i2); }

// Sorted top-KT list of one thread.  Elements arrive in increasing index order, so an equal value never
// displaces an earlier one and the strict comparison keeps the lower index first.
template <int KT> struct TopK {
    float v[KT];
    int i[KT];
    __device__ void init() {
#pragma unroll
        for (int q = 0; q < KT; ++q) { v[q] = -INFINITY; i[q] = 0x7fffffff; }
    }
    __device__ __forceinline__ void push(float z, int k) {
        if (!(z > v[KT - 1])) return;
        v[KT - 1] = z;
        i[KT - 1] = k;
#pragma unroll
        for (int q = KT - 1; q > 0; --q) {
            if (v[q] > v[q - 1]) {
                const float tv = v[q]; v[q] = v[q - 1]; v[q - 1] = tv;
                const int ti = i[q]; i[q] = i[q - 1]; i[q - 1] = ti;
            }
        }
    }
    __device__ __forceinline__ void pop() {   // drop the head, shift the rest up
#pragma unroll
        for (int q = 0; q < KT - 1; ++q) { v[q] = v[q + 1]; i[q] = i[q + 1]; }
        v[KT - 1] = -INFINITY;
        i[KT - 1] = 0x7fffffff;
    }
};

// Merge the sorted lists held by the lanes of a warp into the warp's top KT (every lane gets the result
// in out_v / out_i).  Each round the best head wins and its lane pops.
template <int KT> __device__ void warp_merge(TopK<KT>& t, float* out_v, int* out_i) {
    const int lane = threadIdx.x & 31;
    for (int q = 0; q < KT; ++q) {
        float bv = t.v[0];
        int bi = t.i[0];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
            if (beats(v2, i2, bv, bi)) { bv = v2; bi = i2; }
        }
        out_v[q] = bv;
        out_i[q] = bi;
        if (t.i[0] == bi && t.v[0] == bv && bi != 0x7fffffff) t.pop();   // indices are unique: one owner
        (void)lane;
    }
}

template <int KT> struct ExpPart {
    float m;     // running max of the CTA's slice
    float s;     // sum of 2^((z - m) log2 e) over the slice
    int fin;     // slice finite
    float v[KT];
    int i[KT];
};

template <int LDT, int KT>
__global__ void __launch_bounds__(kExpThreads) expand_rows_kernel(ExpandArgs a, int CL, int chunk) {
    using RW = Row<LDT>;
    using LT = typename RW::T;
    constexpr int VEC = RW::kVec;
    constexpr int NW = kExpThreads / 32;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ ExpPart<KT> s_warp[NW];
    __shared__ ExpPart<KT> s_cta;

    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.x / CL;
    const int V = a.V, k = a.k;
    const LT* base = (const LT*)a.logits + (size_t)row * V;
    const int c0 = min(V, rank * chunk), c1 = min(V, c0 + chunk);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    TopK<KT> tk;
    tk.init();
    float m = -INFINITY, s = 0.f;
    int fin = 1;
    const bool vec_ok = (V % VEC) == 0;
    if (vec_ok) {
        // kExpBatch vectors a thread, all loads issued before any is used; elements still reach the top-k
        // lists in increasing index order
        constexpr int STRIDE = kExpThreads * VEC;
        for (int kb = c0 + tid * VEC; kb < c1; kb += kExpBatch * STRIDE) {
            float z[kExpBatch][VEC];
#pragma unroll
            for (int u = 0; u < kExpBatch; ++u)
                if (kb + u * STRIDE < c1) RW::load_vec(base + kb + u * STRIDE, z[u]);
#pragma unroll
            for (int u = 0; u < kExpBatch; ++u) {
                if (kb + u * STRIDE >= c1) break;
                float mx = m;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    fin &= fabsf(z[u][e]) <= 3.402823466e38f;
                    mx = fmaxf(mx, z[u][e]);
                }
                if (mx > m) {   // rescale the running sum to the new maximum
                    s *= ex2_approx((m - mx) * kLog2e);
                    m = mx;
                }
                const float ml = m * kLog2e;
#pragma unroll
                for (int e = 0; e < VEC; ++e) s += ex2_approx(__fmaf_rn(z[u][e], kLog2e, -ml));
#pragma unroll
                for (int e = 0; e < VEC; ++e) tk.push(z[u][e], kb + u * STRIDE + e);
            }
        }
    } else {
        for (int kk = c0 + tid; kk < c1; kk += kExpThreads) {
            const float z = RW::load(base + kk);
            fin &= fabsf(z) <= 3.402823466e38f;
            if (z > m) {
                s *= ex2_approx((m - z) * kLog2e);
                m = z;
            }
            s += ex2_approx(__fmaf_rn(z, kLog2e, -m * kLog2e));
            tk.push(z, kk);
        }
    }
    if (!fin) { m = 0.f; s = 0.f; }   // the request fails; keep the arithmetic finite
    // warp: (m, s) and the top-KT lists
    float wm = m;
#pragma unroll
    for (int o = 16; o; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    float ws = (m == -INFINITY) ? 0.f : s * ex2_approx((m - wm) * kLog2e);
#pragma unroll
    for (int o = 16; o; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    const int wfin = __all_sync(0xffffffffu, fin);
    float mv[KT];
    int mi[KT];
    warp_merge<KT>(tk, mv, mi);
    if (lane == 0) {
        s_warp[warp].m = wm;
        s_warp[warp].s = ws;
        s_warp[warp].fin = wfin;
#pragma unroll
        for (int q = 0; q < KT; ++q) { s_warp[warp].v[q] = mv[q]; s_warp[warp].i[q] = mi[q]; }
    }
    __syncthreads();
    // CTA: warp 0 merges the NW warp lists (lane w holds list w)
    if (warp == 0) {
        TopK<KT> t2;
        t2.init();
        float pm = -INFINITY, ps = 0.f;
        int pf = 1;
        if (lane < NW) {
#pragma unroll
            for (int q = 0; q < KT; ++q) { t2.v[q] = s_warp[lane].v[q]; t2.i[q] = s_warp[lane].i[q]; }
            pm = s_warp[lane].m;
            ps = s_warp[lane].s;
            pf = s_warp[lane].fin;
        }
        float cm = pm;
#pragma unroll
        for (int o = 16; o; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        float cs = (pm == -INFINITY) ? 0.f : ps * ex2_approx((pm - cm) * kLog2e);
#pragma unroll
        for (int o = 16; o; o >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, o);
        const int cf = __all_sync(0xffffffffu, pf);
        warp_merge<KT>(t2, mv, mi);
        if (lane == 0) {
            s_cta.m = cm;
            s_cta.s = cs;
            s_cta.fin = cf;
#pragma unroll
            for (int q = 0; q < KT; ++q) { s_cta.v[q] = mv[q]; s_cta.i[q] = mi[q]; }
        }
    }
    cluster.sync();
    // cluster: CTA 0's warp 0 merges the CL CTA lists through distributed shared memory
    if (rank == 0 && warp == 0) {
        TopK<KT> t3;
        t3.init();
        float pm = -INFINITY, ps = 0.f;
        int pf = 1;
        if (lane < CL) {
            const ExpPart<KT>* p = cluster.map_shared_rank(&s_cta, lane);
#pragma unroll
            for (int q = 0; q < KT; ++q) { t3.v[q] = p->v[q]; t3.i[q] = p->i[q]; }
            pm = p->m;
            ps = p->s;
            pf = p->fin;
        }
        float rm = pm;
#pragma unroll
        for (int o = 16; o; o >>= 1) rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, o));
        float rs = (pm == -INFINITY) ? 0.f : ps * ex2_approx((pm - rm) * kLog2e);
#pragma unroll
        for (int o = 16; o; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
        const int rf = __all_sync(0xffffffffu, pf);
        warp_merge<KT>(t3, mv, mi);
        const float lse = rm + logf(rs);
        if (lane < k) {
            // lists are at least k long and the row has at least k tokens, so every entry is real
            float outv = mv[0];
            int outi = mi[0];
#pragma unroll
            for (int q = 1; q < KT; ++q) if (q == lane) { outv = mv[q]; outi = mi[q]; }
            a.topk_token[(size_t)row * k + lane] = rf ? outi : -1;
            a.topk_logprob[(size_t)row * k + lane] = rf ? outv - lse : -INFINITY;
        }
    }
    cluster.sync();   // keep every CTA's shared memory alive until CTA 0 has read it
    pdl_launch_dependents();
}

constexpr int kSelThreads = 1024;

// One CTA per request: rank the candidates by (score desc, slot asc, rank asc) and keep the n_keep best,
// listed in (slot, rank) order.
__global__ void __launch_bounds__(kSelThreads) expand_select_kernel(ExpandArgs a) {
    __shared__ float s_score[kSelThreads];
    __shared__ int s_warp_cnt[kSelThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = a.k, NF = a.n_front, N = NF * k;
    pdl_wait_prior();
    const size_t r0 = (size_t)b * NF;
    int bad = 0;
    float sc = -INFINITY;
    if (tid < N) {
        const int slot = tid / k;
        const float fs = a.front_score[r0 + slot];
        const int tok = a.topk_token[(r0 + slot) * k + tid % k];
        bad = tok < 0 || !(fabsf(fs) <= 3.402823466e38f);
        sc = __fadd_rn(fs, a.topk_logprob[(r0 + slot) * k + tid % k]);
        s_score[tid] = sc;
    }
    const int fail = __syncthreads_or(bad);
    if (fail) {
        if (tid < N) {
            a.topk_token[r0 * k + tid] = -1;
            a.topk_logprob[r0 * k + tid] = -INFINITY;
        }
        for (int i = tid; i < a.n_keep; i += kSelThreads) {
            a.child_parent[(size_t)b * a.n_keep + i] = -1;
            a.child_token[(size_t)b * a.n_keep + i] = -1;
            a.child_score[(size_t)b * a.n_keep + i] = -INFINITY;
        }
        if (tid == 0 && a.status) a.status[b] = SV_ERR_NONFINITE;
        return;
    }
    int before = 0;   // candidates that beat this one
    if (tid < N) {
        for (int d = 0; d < N; ++d) {
            const float o = s_score[d];
            before += (o > sc) || (o == sc && d < tid);
        }
    }
    const bool kept = tid < N && before < a.n_keep;
    const unsigned bal = __ballot_sync(0xffffffffu, kept);
    if (lane == 0) s_warp_cnt[warp] = __popc(bal);
    __syncthreads();
    if (kept) {
        int pos = __popc(bal & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) pos += s_warp_cnt[w];
        const int slot = tid / k;
        a.child_parent[(size_t)b * a.n_keep + pos] = slot;
        a.child_token[(size_t)b * a.n_keep + pos] = a.topk_token[(r0 + slot) * k + tid % k];
        a.child_score[(size_t)b * a.n_keep + pos] = sc;
    }
    if (tid == 0 && a.status) a.status[b] = SV_OK;
}

// SM count of the current device (cached per device)
int expand_sm_count() {
    static std::atomic<int> cached[64] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && (n = cached[dev].load()) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    if (dev >= 0 && dev < 64) cached[dev].store(n);
    return n;
}

template <int LDT, int KT>
cudaError_t launch_expand_rows(const ExpandArgs& a, cudaStream_t s) {
    constexpr int VEC = Row<LDT>::kVec;
    const int rows = a.B * a.n_front;
    // a cluster of CTAs per row, at most about 8 CTAs per SM in all, each slice at least 4 vectors a thread
    int cap = (a.V + kExpThreads * VEC * 4 - 1) / (kExpThreads * VEC * 4);
    cap = cap < 1 ? 1 : (cap > kExpMaxCluster ? kExpMaxCluster : cap);
    int CL = 1;
    while (CL * 2 <= cap && (long long)rows * CL * 2 <= 8LL * expand_sm_count()) CL *= 2;
    int chunk = (a.V + CL - 1) / CL;
    chunk = (chunk + VEC - 1) / VEC * VEC;
    return launch_ex(expand_rows_kernel<LDT, KT>, dim3(rows * CL), dim3(kExpThreads), 0, s, CL, false, a, CL, chunk);
}

template <int LDT>
cudaError_t launch_expand_typed(const ExpandArgs& a, cudaStream_t s) {
    if (a.k <= 1) return launch_expand_rows<LDT, 1>(a, s);
    if (a.k <= 2) return launch_expand_rows<LDT, 2>(a, s);
    if (a.k <= 4) return launch_expand_rows<LDT, 4>(a, s);
    if (a.k <= 8) return launch_expand_rows<LDT, 8>(a, s);
    return launch_expand_rows<LDT, 16>(a, s);
}

}  // namespace

cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t s) {
    if (a.B == 0 || a.Hkv == 0) return cudaSuccess;
    const int esz = a.kv_dt == SV_F32 ? 4 : a.kv_dt == SV_BF16 ? 2 : 1;
    const int chunks = a.D * esz / 16;
    int threads = (2 * chunks + 31) / 32 * 32;
    if (threads < 64) threads = 64;
    kv_compact_kernel<<<a.B * a.Hkv, threads, 0, s>>>(a, chunks);
    return cudaGetLastError();
}

cudaError_t launch_tree_expand(const ExpandArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    cudaError_t e = a.logit_dt == SV_F32 ? launch_expand_typed<SV_F32>(a, s) : launch_expand_typed<SV_BF16>(a, s);
    if (e != cudaSuccess) return e;
    return launch_ex(expand_select_kernel, dim3(a.B), dim3(kSelThreads), 0, s, 1, true, a);
}

}  // namespace sv
