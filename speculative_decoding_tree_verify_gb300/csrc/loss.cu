// loss.cu -- acceptance + rejection loss of the draft over logged trees, with its bf16 gradient.
//
// "Aurora" post, section 2: the draft learns from accepted tokens by cross-entropy (imitation) and from
// rejected branches by a rejection loss.  Per non-root node j with parent p and token x:
//   accepted (x == label of p):  -log q_p(x)              rejected:  -log(1 - q_p(x)),  q_p(x) <= 1 - 1e-6
// loss = (sum of terms) / n_terms with n_terms = N * (T - 1).  With A accepted children, rejected children
// r (token x_r, c_r = q(x_r) / (1 - q(x_r)) = 1 / expm1(a_r), a_r = lse - z(x_r)) and C = sum_r c_r, the
// gradient of row p is  g_k = ( q_k (A - C) - A [k == label] + sum_r c_r [k == x_r] ) / n_terms.
//
// Kernel 1: one cluster of CL CTAs per row (each a contiguous vocabulary slice, 128-bit loads).  Rows
// without children only write a zero gradient (their logits are never read).  Pass 1 is an online
// max / sum-exp, combined across the cluster in distributed shared memory; pass 2 re-reads the CTA's own
// slice (L2-resident) and writes the gradient; the few indices that carry a delta term are then
// rewritten with their full value.  Kernel 2: a fixed-order reduction of the per-row sums.
#include <cooperative_groups.h>

#include "sv_internal.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxCluster = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

struct MS { float m, s; };   // running max (log2 units) and sum of 2^(u - m)

__device__ __forceinline__ MS ms_combine(MS a, MS b) {
    if (a.m == -INFINITY) return b;
    if (b.m == -INFINITY) return a;
    float m = fmaxf(a.m, b.m);
    return MS{m, a.s * exp2f(a.m - m) + b.s * exp2f(b.m - m)};
}

__device__ __forceinline__ float log1mexp_f(float a) {   // log(1 - e^-a), a > 0
    return a <= kLn2 ? logf(-expm1f(-a)) : log1pf(-expf(-a));
}

struct LossShared {
    int32_t par[SV_MAX_T];
    int32_t tok[SV_MAX_T];
    int32_t ch[SV_MAX_T];     // children of this row's node
    float cr[SV_MAX_T];       // c_r of each child (0 for accepted ones)
    MS warp_ms[kThreads / 32];
    MS cta_ms;                // read by the whole cluster
    int nch, st, label;
    float A, C, acc, rej;
};

__global__ void __launch_bounds__(kThreads) loss_rows_kernel(LossArgs a, int CL, int chunk, float inv_n) {
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ LossShared sh;
    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.x / CL;
    const int T = a.T, V = a.V;
    const int n = row / T, p = row - n * T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int i = tid; i < T; i += kThreads) {
        sh.par[i] = a.parent[(size_t)n * T + i];
        sh.tok[i] = a.tokens[(size_t)n * T + i];
    }
    __syncthreads();
    int st = block_tree_check(sh.par, T);
    int bad = 0;
    for (int c = 1 + tid; c < T && st == SV_OK; c += kThreads) {
        int lab = a.labels[(size_t)n * T + sh.par[c]];
        bad |= sh.tok[c] < 0 || sh.tok[c] >= V || lab < 0 || lab >= V;
    }
    if (__syncthreads_or(bad) && st == SV_OK) st = SV_ERR_INVALID_ARG;
    if (tid == 0) {
        int k = 0;
        if (st == SV_OK)
            for (int c = p + 1; c < T; ++c) if (sh.par[c] == p) sh.ch[k++] = c;
        sh.nch = k;
        sh.label = a.labels[(size_t)n * T + p];
        if (p == 0 && rank == 0 && a.status) a.status[n] = st;
    }
    __syncthreads();
    const int c0 = min(V, rank * chunk), c1 = min(V, c0 + chunk);
    uint16_t* grow = a.grad ? (uint16_t*)a.grad + (size_t)row * V : nullptr;
    const bool vec_ok = (V % 8) == 0;
    float* wsf = (float*)a.ws;

    if (sh.nch == 0) {   // leaf row or failed trace: zero gradient, no terms; logits are not read
        if (grow) {
            if (vec_ok) for (int k = c0 + tid * 8; k < c1; k += kThreads * 8) *reinterpret_cast<uint4*>(grow + k) = make_uint4(0, 0, 0, 0);
            else for (int k = c0 + tid; k < c1; k += kThreads) grow[k] = 0;
        }
        if (rank == 0 && tid == 0) {
            a.row_loss[row] = 0.f;
            wsf[row] = 0.f;
            wsf[(size_t)a.N * T + row] = 0.f;
        }
        return;
    }

    const uint16_t* z = (const uint16_t*)a.logits + (size_t)row * V;
    // pass 1: online max / sum of 2^(z*log2e - m)
    MS ms{-INFINITY, 0.f};
    auto visit = [&](float zz) {
        float u = zz * kLog2e;
        if (u > ms.m) { ms.s = ms.s * exp2f(ms.m - u) + 1.f; ms.m = u; }
        else ms.s += exp2f(u - ms.m);
    };
    if (vec_ok) {
        for (int k = c0 + tid * 8; k < c1; k += kThreads * 8) {
            uint4 v = __ldg(reinterpret_cast<const uint4*>(z + k));
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) { visit(__uint_as_float(w[i] << 16)); visit(__uint_as_float(w[i] & 0xffff0000u)); }
        }
    } else {
        for (int k = c0 + tid; k < c1; k += kThreads) visit(bf16_bits_to_float(z[k]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        MS other{__shfl_xor_sync(0xffffffffu, ms.m, o), __shfl_xor_sync(0xffffffffu, ms.s, o)};
        ms = ms_combine(ms, other);
    }
    if (lane == 0) sh.warp_ms[warp] = ms;
    __syncthreads();
    if (tid == 0) {
        MS t = sh.warp_ms[0];
        for (int w = 1; w < kThreads / 32; ++w) t = ms_combine(t, sh.warp_ms[w]);
        sh.cta_ms = t;
    }
    cluster.sync();
    MS tot = *cluster.map_shared_rank(&sh.cta_ms, 0);
    for (int q = 1; q < CL; ++q) tot = ms_combine(tot, *cluster.map_shared_rank(&sh.cta_ms, q));
    cluster.sync();
    const float lse2 = tot.m + log2f(tot.s);     // log2-sum-exp2 of z*log2e
    const float lse = lse2 * kLn2;

    // terms (every CTA of the cluster computes them; only rank 0 stores them)
    if (tid == 0) {
        float A = 0.f, C = 0.f, acc = 0.f, rej = 0.f;
        for (int i = 0; i < sh.nch; ++i) {
            int x = sh.tok[sh.ch[i]];
            float ax = lse - bf16_bits_to_float(z[x]);
            if (x == sh.label) {
                A += 1.f;
                acc += ax;
                sh.cr[i] = 0.f;
            } else {
                float aa = fmaxf(ax, 1e-6f);
                rej += -log1mexp_f(aa);
                float c = 1.f / expm1f(aa);
                sh.cr[i] = c;
                C += c;
            }
        }
        sh.A = A; sh.C = C; sh.acc = acc; sh.rej = rej;
        if (rank == 0) {
            a.row_loss[row] = acc + rej;
            wsf[row] = acc;
            wsf[(size_t)a.N * T + row] = rej;
        }
    }
    __syncthreads();
    if (!grow) return;

    // pass 2: dense part q_k (A - C) / n_terms
    const float coef = (sh.A - sh.C) * inv_n;
    auto gval = [&](float zz) { return exp2f(zz * kLog2e - lse2) * coef; };
    if (vec_ok) {
        for (int k = c0 + tid * 8; k < c1; k += kThreads * 8) {
            uint4 v = __ldg(reinterpret_cast<const uint4*>(z + k));
            uint32_t w[4] = {v.x, v.y, v.z, v.w}, o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t lo = float_to_bf16_bits(gval(__uint_as_float(w[i] << 16)));
                uint32_t hi = float_to_bf16_bits(gval(__uint_as_float(w[i] & 0xffff0000u)));
                o[i] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4*>(grow + k) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    } else {
        for (int k = c0 + tid; k < c1; k += kThreads) grow[k] = float_to_bf16_bits(gval(bf16_bits_to_float(z[k])));
    }
    __syncthreads();
    // delta terms: one thread per distinct child token that falls in this CTA's slice
    if (tid < sh.nch) {
        const int x = sh.tok[sh.ch[tid]];
        bool first = x >= c0 && x < c1;
        for (int i = 0; i < tid && first; ++i) first = sh.tok[sh.ch[i]] != x;
        if (first) {
            float extra = 0.f;
            for (int i = 0; i < sh.nch; ++i) if (sh.tok[sh.ch[i]] == x) extra += sh.cr[i];
            if (x == sh.label) extra -= sh.A;
            grow[x] = float_to_bf16_bits(gval(bf16_bits_to_float(z[x])) + extra * inv_n);
        }
    }
}

__global__ void __launch_bounds__(kThreads) loss_sums_kernel(LossArgs a) {
    pdl_wait_prior();
    __shared__ double s_acc[kThreads], s_rej[kThreads];
    const int rows = a.N * a.T;
    const float* wsf = (const float*)a.ws;
    double acc = 0.0, rej = 0.0;
    for (int r = threadIdx.x; r < rows; r += kThreads) {   // fixed assignment and order: deterministic
        acc += (double)wsf[r];
        rej += (double)wsf[(size_t)rows + r];
    }
    s_acc[threadIdx.x] = acc;
    s_rej[threadIdx.x] = rej;
    __syncthreads();
    for (int w = kThreads / 2; w; w >>= 1) {
        if ((int)threadIdx.x < w) {
            s_acc[threadIdx.x] += s_acc[threadIdx.x + w];
            s_rej[threadIdx.x] += s_rej[threadIdx.x + w];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.sums[0] = (float)s_acc[0];
        a.sums[1] = (float)s_rej[0];
        a.sums[2] = (float)((double)a.N * (double)(a.T - 1));
    }
}

}  // namespace

size_t loss_workspace_size(int N, int T, int V) {
    (void)V;
    return ((size_t)2 * N * T * sizeof(float) + 255) / 256 * 256;
}

cudaError_t launch_loss(const LossArgs& a, cudaStream_t s) {
    if (a.N > 0) {
        int CL = (a.V + kThreads * 8 * 4 - 1) / (kThreads * 8 * 4);
        CL = CL < 1 ? 1 : (CL > kMaxCluster ? kMaxCluster : CL);
        int chunk = (a.V + CL - 1) / CL;
        chunk = (chunk + 7) / 8 * 8;
        const double n_terms = (double)a.N * (double)(a.T - 1);
        const float inv_n = n_terms > 0 ? (float)(1.0 / n_terms) : 0.f;
        cudaError_t e = launch_ex(loss_rows_kernel, dim3(CL * a.N * a.T), dim3(kThreads), 0, s, CL, false, a, CL,
                                  chunk, inv_n);
        if (e != cudaSuccess) return e;
    }
    return launch_ex(loss_sums_kernel, dim3(1), dim3(kThreads), 0, s, 1, a.N > 0, a);
}

}  // namespace sv
