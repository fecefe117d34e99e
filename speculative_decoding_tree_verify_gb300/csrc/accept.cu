// accept.cu -- verification of draft trees against the target's per-node logits.
//
// The target checks every draft node in one pass ("Aurora" post, section 2; TIDE overview) and the
// acceptance length is the number of draft tokens accepted per verification step (TIDE evaluation).
//
// Kernel 1 (rows): one thread-block cluster of CL CTAs per logit row, each CTA one contiguous slice of
//   the vocabulary, 128-bit loads.  Greedy: (max, first index) -> argmax.  Stochastic (fp32 rows, or rows
//   whose length breaks 16-byte alignment): max of y = z*invT, then the fixed-point weight sum S of the
//   integer contract over a second, cache-served pass.  Partial results meet in distributed shared memory.
// Kernel 1b (staged rows, stochastic bf16): each CTA bulk-copies its slice into shared memory, so the row
//   is read from HBM once, and computes max / min and then the weights from there.
// Kernel 2 (walk): one cluster per request.  Greedy: a single thread follows the argmax matches.
//   Stochastic: every thread of the cluster runs the same walk on broadcast scalars; the residual sums and
//   the bonus draw are cluster-wide passes over the stopping row only.
//
// Integer contract (stated in include/sv.h, implemented here from that text):
//   y = fp32(z) * invT;  m = max y;  t = (y - m) * log2(e);  W = 0 if t < -24 else
//   floor(P(t - rint(t)) * 2^(24 + rint(t))), P(f) = sum_j fp32((ln 2)^j / j!) f^j (degree 7, Horner, fma);
//   accept child c (token x) iff U_c * Wq(x) * S'_p < 2^32 * W'_p(x) * S_q; on rejection
//   W'_p(k) <- floor(max(0, W'_p(k) * S_q - Wq(k) * S'_p) / S_q); bonus = smallest j with
//   prefix_sum(j) > floor(U_0 * R / 2^32).
#include <cooperative_groups.h>

#include <atomic>
#include <mutex>

#include "sv_internal.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

typedef unsigned long long u64;
typedef unsigned __int128 u128;

constexpr int kRowThreads = 256;
constexpr int kWalkThreads = 512;
constexpr int kLazySumsMinT = 16;   // nodes per request from which the walk computes the weight sums itself
constexpr int kSearchSteps = 8;     // warp steps of a bonus search above which the segment is split first
constexpr int kLazyLoads = 4;       // 16-byte loads in flight per lane in the walk's one-hot row-sum pass
constexpr int kMaxCluster = 8;

struct RowStat {
    float zmax;   // max of z
    int arg;      // first index of the max of z, -1 if the row holds a non-finite z
    float ymax;   // max of y = z * invT (stochastic)
    int fin;      // row usable: z finite (greedy) / y finite (stochastic)
    u64 S;        // sum of fixed-point weights (stochastic)
};

// ------------------------------------------------------------------------------------ the contract
__device__ __forceinline__ float fx_exp2_poly(float f) {
    float p = 0x1.ffcbfcp-17f;
    p = __fmaf_rn(p, f, 0x1.430912p-13f);
    p = __fmaf_rn(p, f, 0x1.5d87fep-10f);
    p = __fmaf_rn(p, f, 0x1.3b2ab6p-7f);
    p = __fmaf_rn(p, f, 0x1.c6b08ep-5f);
    p = __fmaf_rn(p, f, 0x1.ebfbe0p-3f);
    p = __fmaf_rn(p, f, 0x1.62e430p-1f);
    p = __fmaf_rn(p, f, 1.0f);
    return p;
}

// W = 0 if t < -24, else floor(P(t - rint t) * 2^(24 + rint t)), t = (y - m) * log2(e).  rint comes from
// the 1.5 * 2^23 rounding constant (round half to even, exact for |t| < 2^22), which also leaves n in the
// low bits of the sum, so only the final floor needs a conversion instruction.
__device__ __forceinline__ uint32_t fx_weight(float y, float m) {
    const float t = __fmul_rn(__fsub_rn(y, m), 0x1.715476p+0f);
    if (!(t >= -24.0f)) return 0u;
    const float r = __fadd_rn(t, 12582912.0f);                     // 1.5 * 2^23 + rint(t), exactly
    const int n = (int)__float_as_uint(r) - 0x4B400000;            // rint(t) in [-24, 0]
    const float f = __fsub_rn(t, __fsub_rn(r, 12582912.0f));
    const float scale = __uint_as_float((uint32_t)(127 + 24 + n) << 23);   // 2^(24+n), exact
    return __float2uint_rd(__fmul_rn(fx_exp2_poly(f), scale));
}

// ---- packed f32x2 helpers (each lane an IEEE fp32 operation rounded to nearest)
__device__ __forceinline__ u64 f2_pack(float lo, float hi) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(u64 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ u64 f2_fma(u64 a, u64 b, u64 c) {
    u64 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ u64 f2_splat(float x) { return f2_pack(x, x); }

// One rejection step of the residual, exactly in integers:
//   floor(max(0, w * d - wq * X) / d)  =  max(0, w - ceil(wq * X / d)),
// with X = a * d + b (b < d) and F = floor(2^64 * b / d) prepared once per rejection.  For wq < 2^32,
// q0 = floor(wq * F / 2^64) is floor(wq * b / d) or one less (wq * F / 2^64 is below wq * b / d by less
// than wq / 2^64 < 1), so r0 = wq * b - q0 * d lies in [0, 2d) and, for d <= 2^63, is exact in 64-bit
// wrapping arithmetic; r0 >= d decides the last unit and r0 mod d == 0 tells an exact quotient.
struct ResidStep {
    u64 a, b, F;
};

// floor(2^64 * b / d) for b < d < 2^63 (the quotient fits 64 bits), by one 128-bit integer division (once
// per rejection)
__device__ u64 frac64(u64 b, u64 d) {
    return (u64)(((u128)b << 64) / (u128)d);
}

__device__ __forceinline__ u64 resid_step(u64 w, u64 wq64, const ResidStep& k, u64 d) {
    const u64 wq = (uint32_t)wq64;   // a weight: at most 2^24.5
    const u64 q0 = __umul64hi(wq, k.F);
    const u64 r0 = wq * k.b - q0 * d;
    const bool ge = r0 >= d;
    const u64 rem = ge ? r0 - d : r0;
    const u64 c = wq * k.a + q0 + (ge ? 1u : 0u) + (rem != 0 ? 1u : 0u);
    return w > c ? w - c : 0u;
}

template <int LDT> struct Logit;
template <> struct Logit<SV_F32> {
    using T = float;
    using Raw = float4;   // one 16-byte vector as loaded
    static constexpr int kVec = 4;
    __device__ static Raw load_raw(const T* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
    __device__ static void unpack(const Raw& v, float* z) { z[0] = v.x; z[1] = v.y; z[2] = v.z; z[3] = v.w; }
    __device__ static void load_vec(const T* p, float* z) { unpack(load_raw(p), z); }
    __device__ static float load(const T* p) { return __ldg(p); }
};
template <> struct Logit<SV_BF16> {
    using T = uint16_t;
    using Raw = uint4;
    static constexpr int kVec = 8;
    __device__ static Raw load_raw(const T* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
    __device__ static void unpack(const Raw& v, float* z) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            z[2 * i] = __uint_as_float(w[i] << 16);
            z[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void load_vec(const T* p, float* z) { unpack(load_raw(p), z); }
    __device__ static float load(const T* p) { return bf16_bits_to_float(__ldg(p)); }
};

// ------------------------------------------------------------------------------------ kernel 1: rows
struct RowPart {
    float zmax;
    int zarg;
    float ymax;
    int fin;
    u64 S;
};

__device__ __forceinline__ void argmax_combine(float& v, int& i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

template <int LDT, bool STOCH>
__global__ void __launch_bounds__(kRowThreads) accept_rows_kernel(AcceptArgs a, int CL, int chunk, int rows_src, int lazy) {
    using LG = Logit<LDT>;
    using LT = typename LG::T;
    constexpr int VEC = LG::kVec;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ RowPart s_warp[kRowThreads / 32];
    __shared__ RowPart s_part;   // this CTA's partial, read by the whole cluster
    __shared__ float s_wymin[kRowThreads / 32], s_ymin;   // stochastic rows: min y per warp, per CTA

    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.x / CL;
    const bool is_draft = row >= rows_src;
    const int r = is_draft ? row - rows_src : row;
    const int V = a.V;
    const LT* base = (const LT*)(is_draft ? a.draft : a.target) + (size_t)r * V;
    const int c0 = min(V, rank * chunk), c1 = min(V, c0 + chunk);
    const float invT = a.invT;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // y = fp32(z) * invT with invT > 0 is non-decreasing in z, so max y = fp32(max z * invT) and every y is
    // finite iff every z is and the two extremes stay finite: no per-token multiply in this pass
    float zmax = -INFINITY, zmin = INFINITY, ymax = -INFINITY;
    int zarg = 0x7fffffff;
    int zfin = 1, yfin = 1;
    auto visit = [&](float z, int k) {
        zfin &= (fabsf(z) <= 3.402823466e38f) ? 1 : 0;
        if (z > zmax) { zmax = z; zarg = k; }
        if (STOCH) zmin = fminf(zmin, z);
    };
    const bool vec_ok = (V % VEC) == 0;   // every row 16-byte aligned (base checked on the host)
    if (vec_ok) {
#pragma unroll 4
        for (int k = c0 + tid * VEC; k < c1; k += kRowThreads * VEC) {
            float z[VEC];
            LG::load_vec(base + k, z);
#pragma unroll
            for (int e = 0; e < VEC; ++e) visit(z[e], k + e);
        }
    } else {
        for (int k = c0 + tid; k < c1; k += kRowThreads) visit(LG::load(base + k), k);
    }
    float ymin = INFINITY;
    if (STOCH) {
        ymax = __fmul_rn(zmax, invT);
        ymin = zmin == INFINITY ? INFINITY : __fmul_rn(zmin, invT);
        yfin = (zmax == -INFINITY || isfinite(ymax)) && (zmin == INFINITY || isfinite(ymin));
    }
    // block combine
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float v2 = __shfl_xor_sync(0xffffffffu, zmax, o);
        int i2 = __shfl_xor_sync(0xffffffffu, zarg, o);
        argmax_combine(zmax, zarg, v2, i2);
        ymax = fmaxf(ymax, __shfl_xor_sync(0xffffffffu, ymax, o));
    }
    if (STOCH) {
#pragma unroll
        for (int o = 16; o; o >>= 1) ymin = fminf(ymin, __shfl_xor_sync(0xffffffffu, ymin, o));
        if (lane == 0) s_wymin[warp] = ymin;
    }
    zfin = __all_sync(0xffffffffu, zfin);
    yfin = __all_sync(0xffffffffu, yfin);
    if (lane == 0) s_warp[warp] = RowPart{zmax, zarg, ymax, zfin & yfin, 0};
    __syncthreads();
    if (tid == 0) {
        RowPart p = s_warp[0];
        for (int w = 1; w < kRowThreads / 32; ++w) {
            argmax_combine(p.zmax, p.zarg, s_warp[w].zmax, s_warp[w].zarg);
            p.ymax = fmaxf(p.ymax, s_warp[w].ymax);
            p.fin &= s_warp[w].fin;
        }
        s_part = p;
        if (STOCH) {
            float m = s_wymin[0];
            for (int w = 1; w < kRowThreads / 32; ++w) m = fminf(m, s_wymin[w]);
            s_ymin = m;
        }
    }
    // z-finiteness of this CTA (for the argmax output)
    __shared__ int s_zfin;
    int zfin_blk = __syncthreads_and(zfin);
    if (tid == 0) s_zfin = zfin_blk;
    cluster.sync();
    // cluster combine: every CTA reads every partial, so all agree on the row maximum
    RowPart tot = *cluster.map_shared_rank(&s_part, 0);
    float tot_ymin = STOCH ? *cluster.map_shared_rank(&s_ymin, 0) : INFINITY;
    int zfin_all = *cluster.map_shared_rank(&s_zfin, 0);
    for (int q = 1; q < CL; ++q) {
        RowPart p = *cluster.map_shared_rank(&s_part, q);
        argmax_combine(tot.zmax, tot.zarg, p.zmax, p.zarg);
        tot.ymax = fmaxf(tot.ymax, p.ymax);
        tot.fin &= p.fin;
        if (STOCH) tot_ymin = fminf(tot_ymin, *cluster.map_shared_rank(&s_ymin, q));
        zfin_all &= *cluster.map_shared_rank(&s_zfin, q);
    }
    cluster.sync();   // partials consumed; s_part may be reused

    u64 S = 0;
    const bool sums = STOCH && !lazy;   // else the walk computes the sums of the rows it visits
    if (sums && tot.fin) {
        const float m = tot.ymax;
        if (vec_ok) {
#pragma unroll 2
            for (int k = c0 + tid * VEC; k < c1; k += kRowThreads * VEC) {
                float z[VEC];
                LG::load_vec(base + k, z);
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    uint32_t w0, w1;
                    w0 = fx_weight(__fmul_rn(z[e], invT), m);
                    w1 = fx_weight(__fmul_rn(z[e + 1], invT), m);
                    S += (u64)w0 + w1;
                }
            }
        } else {
            for (int k = c0 + tid; k < c1; k += kRowThreads) S += fx_weight(__fmul_rn(LG::load(base + k), invT), m);
        }
    }
    if (sums) {
        S = warp_sum_u64(S);
        __shared__ u64 s_ws[kRowThreads / 32];
        if (lane == 0) s_ws[warp] = S;
        __syncthreads();
        if (tid == 0) {
            u64 t = 0;
            for (int w = 0; w < kRowThreads / 32; ++w) t += s_ws[w];
            s_part.S = t;
        }
        cluster.sync();
        if (rank == 0 && tid == 0) {
            u64 t = 0;
            for (int q = 0; q < CL; ++q) t += cluster.map_shared_rank(&s_part, q)->S;
            tot.S = t;
        }
        cluster.sync();
    }
    if (rank == 0 && tid == 0) {
        RowStat st;
        st.zmax = tot.zmax;
        st.arg = zfin_all ? tot.zarg : -1;
        st.ymax = tot.ymax;
        // stochastic: 1 finite with every t = (y - max y) log2 e above -2^22 (the shift form of the weights
        // applies), 2 finite otherwise, 0 non-finite
        const bool fast = tot.fin && __fsub_rn(tot.ymax, tot_ymin) < 2097152.0f;
        st.fin = STOCH ? (tot.fin ? (fast ? 1 : 2) : 0) : zfin_all;
        st.S = sums ? tot.S : 0;
        ((RowStat*)a.ws)[row] = st;
        if (a.argmax && !is_draft) a.argmax[r] = st.arg;
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------------------------ kernel 1b: staged rows
// Stochastic rows of bf16 logits (rows 16-byte aligned): each CTA of the row's cluster copies its slice
// into shared memory with bulk copies (kStoPieces pieces, one mbarrier each), so the row is read from HBM
// once.  Pass 1 takes the max and min of z with packed bf16x2 instructions while the pieces arrive; the
// cluster agrees on m = fp32(max z * invT); pass 2 computes the fixed-point weights from shared memory.
//
// Pass 2 uses two exact identities of the contract's arithmetic:
//  * the Horner polynomial with every coefficient scaled by 2^24 returns exactly P(f) * 2^24 (scaling by a
//    power of two commutes with round-to-nearest in the normal range), and that value lies in
//    [2^23.5, 2^24.5), where every float is an integer;
//  * floor(x * 2^n) for n <= 0 and an integer x is x >> -n, and x >> s is 0 for s >= 25 > log2(x), so the
//    t < -24 case needs no test (t in [-24.5, -24) gives P < 1 at n = -24, also 0).
// The identities need |t| < 2^22 (rint by the 1.5 * 2^23 constant); rows whose range of y is wider take
// the scalar contract instead.
constexpr int kStoThreads = 256;
constexpr int kStoPieces = 4;
constexpr int kStoMaxSlice = 96 * 1024;   // bytes of shared memory for one CTA's slice

__device__ __forceinline__ uint32_t shr_clamped(uint32_t x, uint32_t s) {   // PTX clamps shifts above 32
    uint32_t r;
    asm("shr.b32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(s));
    return r;
}
__device__ __forceinline__ uint32_t f2u_floor(float x) {
    uint32_t r;
    asm("cvt.rmi.u32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// the contract's weights of two tokens with logits z0, z1 against the row maximum m of y = z * invT, for
// rows whose every t is above -2^22 (see above); bit for bit fx_weight's.  The rounding steps before the
// polynomial (y, y - m, t, rint t, f) are scalar round-to-nearest intrinsics, which the compiler never
// fuses: packed f32x2 multiplies whose product feeds a packed add (also when written as an fma with a unit
// multiplier) were measured to be fused into one rounding, which moves rint(t) at half-integers.  The
// polynomial is an explicit fma chain, evaluated on both tokens at once.  UNIT_T: invT == 1, so y = z.
template <bool UNIT_T>
__device__ __forceinline__ void fx_weight2_fast(float z0, float z1, float invT, float m, uint32_t& w0, uint32_t& w1) {
    const float y0 = UNIT_T ? z0 : __fmul_rn(z0, invT), y1 = UNIT_T ? z1 : __fmul_rn(z1, invT);
    const float t0 = __fmul_rn(__fsub_rn(y0, m), 0x1.715476p+0f);
    const float t1 = __fmul_rn(__fsub_rn(y1, m), 0x1.715476p+0f);
    const float r0 = __fadd_rn(t0, 12582912.0f), r1 = __fadd_rn(t1, 12582912.0f);
    const u64 f2 = f2_pack(__fsub_rn(t0, __fsub_rn(r0, 12582912.0f)), __fsub_rn(t1, __fsub_rn(r1, 12582912.0f)));
    u64 p = f2_splat(0x1.ffcbfcp-17f * 16777216.0f);
    p = f2_fma(p, f2, f2_splat(0x1.430912p-13f * 16777216.0f));
    p = f2_fma(p, f2, f2_splat(0x1.5d87fep-10f * 16777216.0f));
    p = f2_fma(p, f2, f2_splat(0x1.3b2ab6p-7f * 16777216.0f));
    p = f2_fma(p, f2, f2_splat(0x1.c6b08ep-5f * 16777216.0f));
    p = f2_fma(p, f2, f2_splat(0x1.ebfbe0p-3f * 16777216.0f));
    p = f2_fma(p, f2, f2_splat(0x1.62e430p-1f * 16777216.0f));
    p = f2_fma(p, f2, f2_splat(16777216.0f));
    float p0, p1;
    f2_unpack(p, p0, p1);
    w0 = shr_clamped(f2u_floor(p0), 0x4B400000u - __float_as_uint(r0));   // shift by -rint(t)
    w1 = shr_clamped(f2u_floor(p1), 0x4B400000u - __float_as_uint(r1));
}

// the sum of the weights of the two bf16 logits packed in `w` (fast-path rows)
template <bool UNIT_T>
__device__ __forceinline__ uint32_t fx_weight_pair_fast(uint32_t w, float invT, float m) {
    uint32_t w0, w1;
    fx_weight2_fast<UNIT_T>(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u), invT, m, w0, w1);
    return w0 + w1;
}

template <bool WANT_ARG>
__global__ void __launch_bounds__(kStoThreads) accept_rows_staged_kernel(AcceptArgs a, int CL, int chunk,
                                                                          int rows_src) {
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(128) unsigned char s_dyn[];
    __shared__ __align__(8) uint64_t s_bar[kStoPieces];
    __shared__ float s_red[2][kStoThreads / 32];
    __shared__ int s_redi[kStoThreads / 32];
    __shared__ u64 s_ws[kStoThreads / 32];
    __shared__ float s_zmax, s_zmin;
    __shared__ int s_arg;
    __shared__ u64 s_S;
    __shared__ int s_err;

    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.x / CL;
    const bool is_draft = row >= rows_src;
    const int r = is_draft ? row - rows_src : row;
    const int V = a.V;
    const uint16_t* base = (const uint16_t*)(is_draft ? a.draft : a.target) + (size_t)r * V;
    const int c0 = min(V, rank * chunk), c1 = min(V, c0 + chunk);
    const int nvec = (c1 - c0) / 8;                    // whole 16-byte vectors (V % 8 == 0)
    const int per = (nvec + kStoPieces - 1) / kStoPieces;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4* sv4 = reinterpret_cast<const uint4*>(s_dyn);

    if (tid == 0) {
        s_err = 0;
        s_S = 0;             // CTA 0's copies are the row's totals (every CTA adds after the first cluster barrier)
        s_arg = 0x7fffffff;
        for (int q = 0; q < kStoPieces; ++q) tc::mbar_init(&s_bar[q], 1);
        tc::mbar_fence_init();
        for (int q = 0; q < kStoPieces; ++q) {
            const int v0 = min(nvec, q * per), v1 = min(nvec, v0 + per);
            const uint32_t bytes = (uint32_t)(v1 - v0) * 16u;
            tc::mbar_arrive_expect_tx(&s_bar[q], bytes);
            if (bytes) tc::bulk_g2s(s_dyn + (size_t)v0 * 16, base + c0 + (size_t)v0 * 8, bytes, &s_bar[q]);
        }
    }
    __syncthreads();

    // pass 1: max and min of z (NaN propagates through max.NaN / min.NaN, infinities become the extremes)
    __nv_bfloat162 mx2 = __halves2bfloat162(__ushort_as_bfloat16(0xff80), __ushort_as_bfloat16(0xff80));   // -inf
    __nv_bfloat162 mn2 = __halves2bfloat162(__ushort_as_bfloat16(0x7f80), __ushort_as_bfloat16(0x7f80));   // +inf
    bool ok = true;
    for (int q = 0; q < kStoPieces; ++q) {
        ok = ok && tc::mbar_wait(&s_bar[q], 0, &s_err);
        if (!ok) break;
        const int v0 = min(nvec, q * per), v1 = min(nvec, v0 + per);
#pragma unroll 4
        for (int v = v0 + tid; v < v1; v += kStoThreads) {
            const uint4 x = sv4[v];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
                mx2 = __hmax2_nan(mx2, h);
                mn2 = __hmin2_nan(mn2, h);
            }
        }
    }
    float zmax = fmaxf(__low2float(mx2), __high2float(mx2));
    float zmin = fminf(__low2float(mn2), __high2float(mn2));
    if (isnan(__low2float(mx2)) || isnan(__high2float(mx2))) zmax = __int_as_float(0x7fc00000);
    // block and cluster: NaN-propagating max / min
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, zmax, o), n2 = __shfl_xor_sync(0xffffffffu, zmin, o);
        zmax = (isnan(zmax) || isnan(m2)) ? __int_as_float(0x7fc00000) : fmaxf(zmax, m2);
        zmin = fminf(zmin, n2);
    }
    if (lane == 0) { s_red[0][warp] = zmax; s_red[1][warp] = zmin; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kStoThreads / 32; ++w) {
            zmax = (isnan(zmax) || isnan(s_red[0][w])) ? __int_as_float(0x7fc00000) : fmaxf(zmax, s_red[0][w]);
            zmin = fminf(zmin, s_red[1][w]);
        }
        s_zmax = zmax;
        s_zmin = zmin;
    }
    cluster.sync();
    zmax = *cluster.map_shared_rank(&s_zmax, 0);
    zmin = *cluster.map_shared_rank(&s_zmin, 0);
    int err = *cluster.map_shared_rank(&s_err, 0);
    for (int q = 1; q < CL; ++q) {
        const float m2 = *cluster.map_shared_rank(&s_zmax, q);
        zmax = (isnan(zmax) || isnan(m2)) ? __int_as_float(0x7fc00000) : fmaxf(zmax, m2);
        zmin = fminf(zmin, *cluster.map_shared_rank(&s_zmin, q));
        err |= *cluster.map_shared_rank(&s_err, q);
    }
    // (no barrier here: s_zmax / s_zmin / s_err are not written again, and no CTA leaves before the cluster barrier
    // below, which every CTA reaches after these reads)

    // every z finite iff max and min are; every y finite iff the two extremes of y are (y monotone in z)
    const float invT = a.invT;
    const bool zfin = isfinite(zmax) && isfinite(zmin);
    const float m = __fmul_rn(zmax, invT);
    const float ymin = __fmul_rn(zmin, invT);
    const bool yfin = zfin && isfinite(m) && isfinite(ymin);
    u64 S = 0;
    int arg = 0x7fffffff;
    const bool fast_row = yfin && __fsub_rn(m, ymin) < 2097152.0f;    // every |t| < 1.45 * 2^21 < 2^22
    if (yfin && !err) {
        const bool fast = fast_row;
        const uint32_t zmax_bits = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(zmax));
        const uint32_t zmax2 = zmax_bits | (zmax_bits << 16);
        const bool unit_t = invT == 1.0f;
        if (fast) {
#pragma unroll 2
            for (int v = tid; v < nvec; v += kStoThreads) {
                const uint4 x = sv4[v];
                uint32_t acc;
                if (unit_t) {
                    acc = fx_weight_pair_fast<true>(x.x, invT, m) + fx_weight_pair_fast<true>(x.y, invT, m) +
                          fx_weight_pair_fast<true>(x.z, invT, m) + fx_weight_pair_fast<true>(x.w, invT, m);
                } else {
                    acc = fx_weight_pair_fast<false>(x.x, invT, m) + fx_weight_pair_fast<false>(x.y, invT, m) +
                          fx_weight_pair_fast<false>(x.z, invT, m) + fx_weight_pair_fast<false>(x.w, invT, m);
                }
                S += acc;
                if (WANT_ARG && arg == 0x7fffffff) {
                    const __nv_bfloat162 m2 = *reinterpret_cast<const __nv_bfloat162*>(&zmax2);
                    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                    uint32_t eq = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) eq |= __heq2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w[e]), m2);
                    if (eq) {
                        for (int e = 0; e < 8 && arg == 0x7fffffff; ++e)
                            if (__uint_as_float(e & 1 ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16)) == zmax)
                                arg = c0 + v * 8 + e;
                    }
                }
            }
        } else {
            for (int v = tid; v < nvec; v += kStoThreads) {
                const uint4 x = sv4[v];
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float z = __uint_as_float(e & 1 ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16));
                    S += fx_weight(__fmul_rn(z, invT), m);
                    if (WANT_ARG && z == zmax && arg == 0x7fffffff) arg = c0 + v * 8 + e;
                }
            }
        }
    } else if (WANT_ARG && zfin && !err) {
        // y overflowed but z is finite: the argmax is still defined
        for (int v = tid; v < nvec && arg == 0x7fffffff; v += kStoThreads) {
            const uint4 x = sv4[v];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            for (int e = 0; e < 8 && arg == 0x7fffffff; ++e)
                if (__uint_as_float(e & 1 ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16)) == zmax) arg = c0 + v * 8 + e;
        }
    }
    S = warp_sum_u64(S);
    if (WANT_ARG) {
#pragma unroll
        for (int o = 16; o; o >>= 1) arg = min(arg, __shfl_xor_sync(0xffffffffu, arg, o));
    }
    if (lane == 0) { s_ws[warp] = S; s_redi[warp] = arg; }
    __syncthreads();
    if (tid == 0) {
        // this CTA's sum and first argmax go into CTA 0's totals (atomics on distributed shared memory)
        u64 t = 0;
        int am = 0x7fffffff;
        for (int w = 0; w < kStoThreads / 32; ++w) { t += s_ws[w]; am = min(am, s_redi[w]); }
        atomicAdd(reinterpret_cast<unsigned long long*>(cluster.map_shared_rank(&s_S, 0)), (unsigned long long)t);
        if (WANT_ARG) atomicMin(cluster.map_shared_rank(&s_arg, 0), am);
    }
    cluster.sync();   // every CTA's share has reached CTA 0; nobody reads another CTA's shared memory after this
    if (rank == 0 && tid == 0) {
        const u64 t = s_S;
        const int am = s_arg;
        RowStat st;
        st.zmax = zmax;
        st.arg = (zfin && !err) ? am : -1;
        st.ymax = m;
        st.fin = err ? -1 : (yfin ? (fast_row ? 1 : 2) : 0);   // 1: finite with every t above -2^22
        st.S = (yfin && !err) ? t : 0;
        ((RowStat*)a.ws)[row] = st;
        if (a.argmax && !is_draft) a.argmax[r] = st.arg;
    }
    if (err && tid == 0) {
        // give the copies still in flight a bounded chance to land before the shared memory is released
        int e2 = 0;
        for (int q = 0; q < kStoPieces; ++q) tc::mbar_wait(&s_bar[q], 0, &e2);
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------------------------ kernel 2: walk
enum { MODE_GREEDY = 0, MODE_PROB = 1, MODE_ONEHOT = 2 };

struct WalkShared {
    int32_t par[SV_MAX_T];
    int32_t tok[SV_MAX_T];
    int32_t path[SV_MAX_T];
    int32_t arg[SV_MAX_T];    // greedy: each row's argmax, gathered once so the walk reads shared memory
    u64 hist[SV_MAX_T];       // PROB: residual sum before each rejection; ONEHOT: rejected tokens
    ResidStep rs[SV_MAX_T];   // PROB: the integer constants of each rejection step
    u64 red[kWalkThreads / 32];
    u64 cta_sum;              // this CTA's share of a cluster-wide sum (read remotely)
    u64 redq[kWalkThreads / 32];
    u64 sub[kWalkThreads / 32];   // bonus search: the sums of the selected warp segment's sub-segments
    float zc_p[SV_MAX_T], zc_q[SV_MAX_T];   // the current row's target (draft) logit at each child's token
    uint32_t uc[SV_MAX_T];                  // and each child's uniform
    u64 cta_sumq;             // the same for the draft row's weights
    int32_t found;            // sampled index found in this CTA (-1 if not)
    int st;
};

template <int LDT, int MODE, bool LAZY>
__global__ void __launch_bounds__(kWalkThreads, 2) accept_walk_kernel(AcceptArgs a, int CLW) {
    using LG = Logit<LDT>;
    using LT = typename LG::T;
    constexpr int VEC = LG::kVec;
    cg::cluster_group cluster = cg::this_cluster();
    __shared__ WalkShared sh;
    const bool vec_ok = (a.V % VEC) == 0;   // every logit row 16-byte aligned (base checked on the host)
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.x / CLW;
    const int T = a.T, V = a.V, B = a.B;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float invT = a.invT;

    for (int i = tid; i < T; i += kWalkThreads) {
        sh.par[i] = a.parent[(size_t)b * T + i];
        sh.tok[i] = a.tokens[(size_t)b * T + i];
    }
    pdl_wait_prior();   // row statistics of kernel 1 are visible from here on
    __syncthreads();
    const RowStat* stats = (const RowStat*)a.ws;
    int st = block_tree_check(sh.par, T);
    int bad = 0;
    for (int c = 1 + tid; c < T; c += kWalkThreads) bad |= (sh.tok[c] < 0 || sh.tok[c] >= V);
    if (__syncthreads_or(bad) && st == SV_OK) st = SV_ERR_INVALID_ARG;
    if (st == SV_OK) {
        int nf = 0, to = 0;
        for (int r = tid; r < T; r += kWalkThreads) {
            const RowStat rs = stats[(size_t)b * T + r];
            nf |= !rs.fin;
            to |= rs.fin < 0;
            if (MODE == MODE_GREEDY) sh.arg[r] = rs.arg;
            if (MODE == MODE_PROB) {
                const int fq = stats[(size_t)B * T + (size_t)b * T + r].fin;
                nf |= !fq;
                to |= fq < 0;
            }
        }
        if (__syncthreads_or(to)) st = SV_ERR_TIMEOUT;
        else if (__syncthreads_or(nf)) st = SV_ERR_NONFINITE;
    }
    if (st != SV_OK) {
        if (rank == 0) {
            for (int j = tid; j < T; j += kWalkThreads) {
                a.path[(size_t)b * T + j] = -1;
                a.out_tokens[(size_t)b * T + j] = -1;
            }
            if (tid == 0) {
                a.accept_len[b] = -1;
                a.bonus[b] = -1;
                if (a.status) a.status[b] = st;
            }
        }
        return;
    }

    int n = 0, cur = 0, bonus = -1;
    if (MODE == MODE_GREEDY) {
        // warp 0 walks: at each node the lanes test 32 later nodes at once (child of cur with the argmax token),
        // and the lowest hit is the first such child
        if (warp == 0) {
            for (;;) {
                const int am = sh.arg[cur];
                int next = -1;
                for (int c0 = cur + 1; c0 < T; c0 += 32) {
                    const int c = c0 + lane;
                    const unsigned hit = __ballot_sync(0xffffffffu, c < T && sh.par[c] == cur && sh.tok[c] == am);
                    if (hit) { next = c0 + __ffs(hit) - 1; break; }
                }
                if (next < 0) { bonus = am; break; }
                if (lane == 0) sh.path[n] = next;
                ++n;
                cur = next;
            }
            if (lane == 0) {
                sh.st = n;
                sh.found = bonus;
            }
        }
        __syncthreads();
        n = sh.st;
        bonus = sh.found;
    } else {
        // every thread of the cluster follows the same walk on identical scalars
        const LT* P = (const LT*)a.target;
        const LT* Q = (const LT*)a.draft;
        const uint32_t* U = a.uniforms + (size_t)b * T;
        for (;;) {
            const size_t prow = (size_t)b * T + cur;
            const RowStat sp = stats[prow];
            RowStat sq;
            u64 Sq = 1;
            if (MODE == MODE_PROB) {
                sq = stats[(size_t)B * T + prow];
                Sq = sq.S;
            }
            const LT* prow_p = P + prow * V;
            const LT* prow_q = (MODE == MODE_PROB) ? Q + prow * V : nullptr;
            int nrej = 0;
            u64 Sp = sp.S;   // the row's weight sum (computed below when the row kernel left it to the walk)
            // residual weight of token k (target logit zp, draft logit zq) after the rejections so far
            auto wres_z = [&](float zp, float zq, int k) -> u64 {
                u64 w = fx_weight(__fmul_rn(zp, invT), sp.ymax);
                if (MODE == MODE_ONEHOT) {
                    for (int i = 0; i < nrej; ++i) if ((int)sh.hist[i] == k) w = 0;
                } else if (MODE == MODE_PROB) {
                    if (nrej) {
                        const u64 wq = fx_weight(__fmul_rn(zq, invT), sq.ymax);
                        for (int i = 0; i < nrej; ++i) w = resid_step(w, wq, sh.rs[i], Sq);
                    }
                }
                return w;
            };
            auto wres = [&](int k) -> u64 {
                return wres_z(LG::load(prow_p + k), MODE == MODE_PROB ? LG::load(prow_q + k) : 0.f, k);
            };
            // the VEC residual weights of tokens k .. k+VEC-1 (16-byte loads; rows are 16-byte aligned)
            // rows marked by the row kernels as having every t above -2^22 take the shift form of the
            // weights (identical integers, fewer instructions)
            const bool fastp = sp.fin == 1;
            const bool fastq = MODE == MODE_PROB ? sq.fin == 1 : true;
            auto wres_vec = [&](int k, u64 (&w)[VEC]) {
                float zp[VEC], zq[VEC];
                LG::load_vec(prow_p + k, zp);
                if (MODE == MODE_PROB && nrej) LG::load_vec(prow_q + k, zq);
#pragma unroll
                for (int e = 0; e < VEC; e += 2) {
                    uint32_t p0, p1;
                    if (fastp) fx_weight2_fast<false>(zp[e], zp[e + 1], invT, sp.ymax, p0, p1);
                    else { p0 = fx_weight(__fmul_rn(zp[e], invT), sp.ymax); p1 = fx_weight(__fmul_rn(zp[e + 1], invT), sp.ymax); }
                    w[e] = p0;
                    w[e + 1] = p1;
                    if (MODE == MODE_ONEHOT) {
                        for (int i = 0; i < nrej; ++i) {
                            if ((int)sh.hist[i] == k + e) w[e] = 0;
                            if ((int)sh.hist[i] == k + e + 1) w[e + 1] = 0;
                        }
                    } else if (MODE == MODE_PROB && nrej) {
                        uint32_t q0, q1;
                        if (fastq) fx_weight2_fast<false>(zq[e], zq[e + 1], invT, sq.ymax, q0, q1);
                        else { q0 = fx_weight(__fmul_rn(zq[e], invT), sq.ymax); q1 = fx_weight(__fmul_rn(zq[e + 1], invT), sq.ymax); }
                        for (int i = 0; i < nrej; ++i) {
                            w[e] = resid_step(w[e], q0, sh.rs[i], Sq);
                            w[e + 1] = resid_step(w[e + 1], q1, sh.rs[i], Sq);
                        }
                    }
                }
            };
            // Cluster layout of the vocabulary: CTA `rank` owns [k0, k1), its warp w the contiguous segment
            // [s0, s1) (whole vectors when vectorised).  seg_sums() leaves each warp's residual mass in
            // sh.red[w] and the CTA's in sh.cta_sum; the bonus draw then searches CTA, warp and token in order.
            const int per = vec_ok ? ((V + CLW - 1) / CLW + VEC - 1) / VEC * VEC : (V + CLW - 1) / CLW;
            const int k0 = min(V, rank * per), k1 = min(V, k0 + per);
            const int nw = kWalkThreads / 32;
            const int seg = vec_ok ? ((k1 - k0 + nw - 1) / nw + VEC - 1) / VEC * VEC : (k1 - k0 + nw - 1) / nw;
            const int s0 = min(k1, k0 + warp * seg), s1 = min(k1, s0 + seg);
            auto seg_sums = [&]() {
                u64 ws = 0;
                if (vec_ok) {
                    for (int k = s0 + lane * VEC; k < s1; k += 32 * VEC) {
                        u64 w[VEC];
                        wres_vec(k, w);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) ws += w[e];
                    }
                } else {
                    for (int k = s0 + lane; k < s1; k += 32) ws += wres(k);
                }
                ws = warp_sum_u64(ws);
                if (lane == 0) sh.red[warp] = ws;
                __syncthreads();
                if (tid == 0) {
                    u64 t = 0;
                    for (int w = 0; w < nw; ++w) t += sh.red[w];
                    sh.cta_sum = t;
                }
            };
            // the weight sums of this row (and of the draft's row) over the cluster, when the row kernel left them to
            // the walk, in one pass over both rows: the plain sums of row p then stay in sh.red / sh.cta_sum for a
            // bonus draw from the row itself
            // the logits and uniforms the acceptance tests of cur's children read, loaded at once
            for (int c = cur + 1 + tid; c < T; c += kWalkThreads) {
                if (sh.par[c] == cur) {
                    const int x = sh.tok[c];
                    sh.zc_p[c] = LG::load(prow_p + x);
                    if (MODE == MODE_PROB) sh.zc_q[c] = LG::load(prow_q + x);
                    sh.uc[c] = U[c];
                }
            }
            if (!LAZY) __syncthreads();   // (the sum pass below synchronises the CTA otherwise)
            bool plain_valid = false;
            if (LAZY) {
                u64 ws = 0, wsq = 0;
                if (vec_ok && MODE == MODE_ONEHOT) {
                    // one row: each lane keeps kLazyLoads 16-byte loads in flight
                    for (int kb = s0 + lane * VEC; kb < s1; kb += kLazyLoads * 32 * VEC) {
                        typename LG::Raw r[kLazyLoads];
#pragma unroll
                        for (int j = 0; j < kLazyLoads; ++j)
                            if (kb + j * 32 * VEC < s1) r[j] = LG::load_raw(prow_p + kb + j * 32 * VEC);
#pragma unroll
                        for (int j = 0; j < kLazyLoads; ++j) {
                            if (kb + j * 32 * VEC < s1) {
                                float z[VEC];
                                LG::unpack(r[j], z);
#pragma unroll
                                for (int e = 0; e < VEC; e += 2) {
                                    uint32_t w0, w1;
                                    if (fastp) fx_weight2_fast<false>(z[e], z[e + 1], invT, sp.ymax, w0, w1);
                                    else { w0 = fx_weight(__fmul_rn(z[e], invT), sp.ymax); w1 = fx_weight(__fmul_rn(z[e + 1], invT), sp.ymax); }
                                    ws += (u64)w0 + w1;
                                }
                            }
                        }
                    }
                } else if (vec_ok) {
                    for (int k = s0 + lane * VEC; k < s1; k += 32 * VEC) {
                        float z[VEC], zq[VEC];
                        LG::load_vec(prow_p + k, z);
                        if (MODE == MODE_PROB) LG::load_vec(prow_q + k, zq);
#pragma unroll
                        for (int e = 0; e < VEC; e += 2) {
                            uint32_t w0, w1;
                            if (fastp) fx_weight2_fast<false>(z[e], z[e + 1], invT, sp.ymax, w0, w1);
                            else { w0 = fx_weight(__fmul_rn(z[e], invT), sp.ymax); w1 = fx_weight(__fmul_rn(z[e + 1], invT), sp.ymax); }
                            ws += (u64)w0 + w1;
                            if (MODE == MODE_PROB) {
                                if (fastq) fx_weight2_fast<false>(zq[e], zq[e + 1], invT, sq.ymax, w0, w1);
                                else { w0 = fx_weight(__fmul_rn(zq[e], invT), sq.ymax); w1 = fx_weight(__fmul_rn(zq[e + 1], invT), sq.ymax); }
                                wsq += (u64)w0 + w1;
                            }
                        }
                    }
                } else {
                    for (int k = s0 + lane; k < s1; k += 32) {
                        ws += fx_weight(__fmul_rn(LG::load(prow_p + k), invT), sp.ymax);
                        if (MODE == MODE_PROB) wsq += fx_weight(__fmul_rn(LG::load(prow_q + k), invT), sq.ymax);
                    }
                }
                ws = warp_sum_u64(ws);
                if (MODE == MODE_PROB) wsq = warp_sum_u64(wsq);
                if (lane == 0) {
                    sh.red[warp] = ws;
                    if (MODE == MODE_PROB) sh.redq[warp] = wsq;
                }
                __syncthreads();
                if (tid == 0) {
                    u64 t = 0, tq = 0;
                    for (int w = 0; w < nw; ++w) {
                        t += sh.red[w];
                        if (MODE == MODE_PROB) tq += sh.redq[w];
                    }
                    sh.cta_sum = t;
                    sh.cta_sumq = tq;
                }
                cluster.sync();
                Sp = 0;
                if (MODE == MODE_PROB) Sq = 0;
                for (int q = 0; q < CLW; ++q) {
                    Sp += *cluster.map_shared_rank(&sh.cta_sum, q);
                    if (MODE == MODE_PROB) Sq += *cluster.map_shared_rank(&sh.cta_sumq, q);
                }
                cluster.sync();
                plain_valid = true;
            }
            u64 Sres = Sp;
            bool sums_valid = false;   // sh.red / sh.cta_sum hold the current residual
            int next = -1, has_child = 0;
            for (int c = cur + 1; c < T; ++c) {
                if (sh.par[c] != cur) continue;
                has_child = 1;
                const int x = sh.tok[c];
                const u64 wpx = wres_z(sh.zc_p[c], MODE == MODE_PROB ? sh.zc_q[c] : 0.f, x);
                const u64 wqx = (MODE == MODE_PROB) ? fx_weight(__fmul_rn(sh.zc_q[c], invT), sq.ymax) : 1u;
                if ((u128)sh.uc[c] * wqx * Sres < (((u128)wpx * Sq) << 32)) { next = c; break; }
                if (MODE == MODE_ONEHOT) {
                    sh.hist[nrej] = (u64)x;   // identical value written by every thread
                    ++nrej;
                    Sres -= wpx;
                } else {
                    if (tid == 0) {
                        sh.hist[nrej] = Sres;
                        ResidStep k;
                        k.a = Sres / Sq;
                        k.b = Sres - k.a * Sq;
                        k.F = frac64(k.b, Sq);
                        sh.rs[nrej] = k;
                    }
                    __syncthreads();
                    ++nrej;
                    Sres = 0;  // recomputed below, in the layout the bonus draw searches
                    plain_valid = false;
                    seg_sums();
                    cluster.sync();
                    for (int q = 0; q < CLW; ++q) Sres += *cluster.map_shared_rank(&sh.cta_sum, q);
                    cluster.sync();
                    sums_valid = true;
                }
            }
            if (next >= 0) {
                if (tid == 0) sh.path[n] = next;
                ++n;
                cur = next;
                __syncthreads();
                continue;
            }
            // the walk stops at `cur`: draw the bonus token from the residual (or the row itself)
            const bool use_res = has_child && Sres != 0;
            const u64 R = use_res ? Sres : Sp;
            if (!use_res) nrej = 0;
            const u128 thr = ((u128)U[0] * R) >> 32;
            // the last residual pass (or the row's own sums) already left the sums the draw searches
            if (MODE == MODE_ONEHOT && use_res && plain_valid) {
                // one-hot residual = the row's weights with the rejected tokens set to 0: take each distinct
                // rejected token's weight off the sums of the warp segment and CTA that hold it
                if (tid == 0) {
                    for (int i = 0; i < nrej; ++i) {
                        const int x = (int)sh.hist[i];
                        bool dup = false;
                        for (int j = 0; j < i; ++j) dup |= (int)sh.hist[j] == x;
                        if (dup || x < k0 || x >= k1) continue;
                        const u64 wx = fx_weight(__fmul_rn(LG::load(prow_p + x), invT), sp.ymax);
                        sh.red[(x - k0) / seg] -= wx;
                        sh.cta_sum -= wx;
                    }
                }
            } else if (!(use_res && sums_valid) && !(!use_res && plain_valid)) {
                seg_sums();
            }
            if (tid == 0) sh.found = -1;
            cluster.sync();
            u64 before = 0;   // weight mass of the CTAs before this one
            for (int q = 0; q < rank; ++q) before += *cluster.map_shared_rank(&sh.cta_sum, q);
            if (thr >= before && thr < before + sh.cta_sum) {
                // this CTA holds the draw: find the warp, then the element
                u64 wb = before;
                int wsel = -1;
                for (int w = 0; w < nw; ++w) {
                    if (thr < wb + sh.red[w]) { wsel = w; break; }
                    wb += sh.red[w];
                }
                if (vec_ok && wsel >= 0) {
                    // A segment longer than kSearchSteps warp steps is split into nw sub-segments of whole
                    // vectors, whose sums every warp computes at once; the warp of the segment (or sub-segment)
                    // holding the draw then scans it, 32 * VEC tokens per step: each lane one vector, a warp scan
                    // of the lane totals
                    const int t0 = min(k1, k0 + wsel * seg), t1 = min(k1, t0 + seg);
                    int u0 = t0, u1 = t1, usel = wsel;
                    u64 ub = wb;
                    if (t1 - t0 > kSearchSteps * 32 * VEC) {
                        const int sub = ((t1 - t0 + nw - 1) / nw + VEC - 1) / VEC * VEC;
                        u0 = min(t1, t0 + warp * sub);
                        u1 = min(t1, u0 + sub);
                        u64 us = 0;
                        for (int k = u0 + lane * VEC; k < u1; k += 32 * VEC) {
                            u64 w[VEC];
                            wres_vec(k, w);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) us += w[e];
                        }
                        us = warp_sum_u64(us);
                        if (lane == 0) sh.sub[warp] = us;
                        __syncthreads();
                        usel = -1;
                        for (int w = 0; w < nw; ++w) {
                            if (thr < ub + sh.sub[w]) { usel = w; break; }
                            ub += sh.sub[w];
                        }
                    }
                    u64 run = ub;
                    for (int kb = u0; warp == usel && kb < u1; kb += 32 * VEC) {
                        const int k = kb + lane * VEC;
                        u64 w[VEC];
                        u64 tl = 0;
                        if (k < u1) {
                            wres_vec(k, w);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) tl += w[e];
                        }
                        u64 incl = tl;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const u64 v = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += v;
                        }
                        const unsigned hit = __ballot_sync(0xffffffffu, k < u1 && (u128)run + incl > thr);
                        if (hit) {
                            if (lane == __ffs(hit) - 1) {
                                u128 acc = (u128)run + (incl - tl);
                                int e = 0;
                                for (; e < VEC - 1; ++e) {
                                    acc += w[e];
                                    if (acc > thr) break;
                                }
                                sh.found = k + e;
                            }
                            break;
                        }
                        run += __shfl_sync(0xffffffffu, incl, 31);
                    }
                } else if (!vec_ok && warp == wsel) {
                    u64 run = wb;
                    for (int k = s0; k < s1; k += 32) {
                        u64 w = (k + lane < s1) ? wres(k + lane) : 0;
                        u64 incl = w;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            u64 v = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += v;
                        }
                        unsigned hit = __ballot_sync(0xffffffffu, (u128)run + incl > thr && k + lane < s1);
                        if (hit) {
                            if (lane == 0) sh.found = k + __ffs(hit) - 1;
                            break;
                        }
                        run += __shfl_sync(0xffffffffu, incl, 31);
                    }
                }
            }
            cluster.sync();
            int f = -1;
            for (int q = 0; q < CLW && f < 0; ++q) f = *cluster.map_shared_rank(&sh.found, q);
            cluster.sync();
            bonus = f < 0 ? V - 1 : f;
            break;
        }
        __syncthreads();
    }
    if (rank == 0) {
        for (int j = tid; j < T; j += kWalkThreads) {
            a.path[(size_t)b * T + j] = j < n ? sh.path[j] : -1;
            a.out_tokens[(size_t)b * T + j] = j < n ? sh.tok[sh.path[j]] : (j == n ? bonus : -1);
        }
        if (tid == 0) {
            a.accept_len[b] = n;
            a.bonus[b] = bonus;
            if (a.status) a.status[b] = SV_OK;
        }
    }
}

// SM count of the current device (cached per device)
int sm_count() {
    static std::atomic<int> cached[64] = {};
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64 && (n = cached[dev].load()) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    if (dev >= 0 && dev < 64) cached[dev].store(n);
    return n;
}

int pick_cluster(int V, int per_cta) {
    int c = (V + per_cta - 1) / per_cta;
    return c < 1 ? 1 : (c > kMaxCluster ? kMaxCluster : c);
}

template <int LDT>
cudaError_t launch_typed(const AcceptArgs& a, cudaStream_t s) {
    constexpr int VEC = Logit<LDT>::kVec;
    const bool stoch = a.temperature > 0.f;
    // Stochastic rows of a tree with many more nodes than a walk visits (T >= 16): the row kernel takes only
    // the max, min and first argmax of every row (every row must still be checked for non-finite logits), and
    // the walk computes the weight sums of the rows it visits.  Chains and small trees, whose walks visit most
    // rows, compute every row's sums in the row pass (measured on 32 chains of 6 nodes: 103 us with the sums in
    // the row pass against 110 us; on 8 trees of 60 nodes 89 against 76 us, on 128 trees of 64 nodes 1040
    // against 498 us).
    const int lazy = (stoch && a.T >= kLazySumsMinT) ? 1 : 0;
    const int mode = !stoch ? MODE_GREEDY : (a.draft ? MODE_PROB : MODE_ONEHOT);
    const int rows_src = a.B * a.T;
    const int rows = rows_src * (mode == MODE_PROB ? 2 : 1);
    // Stochastic rows with their sums: one CTA per row when there are many (no cluster synchronisation), else a
    // cluster splits each row.  Greedy rows and stochastic rows without sums: the largest power-of-two cluster
    // with at most about 9 CTAs per SM in all, which evens out the last wave (measured on 480 and 192 rows of
    // 128K-152K logits: 2 and 4).
    int CL;
    if (stoch && !lazy) {
        CL = rows >= 8 * sm_count() ? 1 : pick_cluster(a.V, kRowThreads * VEC * 4);
    } else {
        const int cap = pick_cluster(a.V, kRowThreads * VEC * 4);
        CL = 1;
        while (CL * 2 <= cap && (long long)rows * CL * 2 <= 9LL * sm_count()) CL *= 2;
    }
    int chunk = (a.V + CL - 1) / CL;
    chunk = (chunk + VEC - 1) / VEC * VEC;
    cudaError_t e;
    // Stochastic bf16 rows whose slices fit in shared memory: the staged kernel (one HBM read per row).
    // The cluster is the smallest power of two that keeps a slice within about 40 KB (several CTAs per SM).
    int CLs = 1;
    const long long row_bytes = (long long)a.V * 2;
    while (CLs < kMaxCluster && row_bytes > (long long)CLs * 40 * 1024) CLs *= 2;
    int chunk_s = ((a.V + CLs - 1) / CLs + 7) / 8 * 8;
    const bool staged = stoch && !lazy && LDT == SV_BF16 && a.V % 8 == 0 && (long long)chunk_s * 2 <= kStoMaxSlice;
    if (staged) {
        const size_t smem = (size_t)chunk_s * 2;
        // room for the slice, and the whole unified L1 as shared memory so several CTAs fit on an SM; function
        // attributes belong to a device, so they are set once per device (and kernel variant)
        static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
        std::atomic<uint64_t>& done = attr_set[a.argmax ? 1 : 0];
        if (!bit || !(done.load() & bit)) {
            const void* fn = a.argmax ? (const void*)accept_rows_staged_kernel<true> : (const void*)accept_rows_staged_kernel<false>;
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kStoMaxSlice);
            if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
            if (e != cudaSuccess) return e;
            done.fetch_or(bit);
        }
        if (a.argmax) e = launch_ex(accept_rows_staged_kernel<true>, dim3(CLs * rows), dim3(kStoThreads), smem, s, CLs, false, a, CLs, chunk_s, rows_src);
        else          e = launch_ex(accept_rows_staged_kernel<false>, dim3(CLs * rows), dim3(kStoThreads), smem, s, CLs, false, a, CLs, chunk_s, rows_src);
    } else if (stoch) e = launch_ex(accept_rows_kernel<LDT, true>, dim3(CL * rows), dim3(kRowThreads), 0, s, CL, false, a, CL, chunk, rows_src, lazy);
    else       e = launch_ex(accept_rows_kernel<LDT, false>, dim3(CL * rows), dim3(kRowThreads), 0, s, CL, false, a, CL, chunk, rows_src, 0);
    if (e != cudaSuccess) return e;
    // walk clusters: enough CTAs per request for the residual passes, but no more than the walk kernel keeps
    // resident at once over all requests (a second wave would repeat each request's serial chain of steps)
    int CLW = 1;
    if (mode != MODE_GREEDY) {
        const int cap = pick_cluster(a.V, kWalkThreads * 8);
        while (CLW * 2 <= cap && (long long)a.B * CLW * 2 <= 2LL * sm_count()) CLW *= 2;
    }
    const dim3 gw(a.B * CLW), bw(kWalkThreads);
    switch (mode) {
    case MODE_GREEDY: return launch_ex(accept_walk_kernel<LDT, MODE_GREEDY, false>, gw, bw, 0, s, 1, true, a, 1);
    case MODE_PROB:
        if (lazy) return launch_ex(accept_walk_kernel<LDT, MODE_PROB, true>, gw, bw, 0, s, CLW, true, a, CLW);
        return launch_ex(accept_walk_kernel<LDT, MODE_PROB, false>, gw, bw, 0, s, CLW, true, a, CLW);
    default:
        if (lazy) return launch_ex(accept_walk_kernel<LDT, MODE_ONEHOT, true>, gw, bw, 0, s, CLW, true, a, CLW);
        return launch_ex(accept_walk_kernel<LDT, MODE_ONEHOT, false>, gw, bw, 0, s, CLW, true, a, CLW);
    }
}

// Scratch of the allocation-free entry point: row statistics for up to kNoAllocMaxRows target rows (and as
// many draft rows), 3 MiB of device memory that every GPU loading the library keeps until exit.
constexpr int kNoAllocMaxRows = 65536;
static_assert(sizeof(RowStat) == 24, "RowStat layout");

}  // namespace

static __device__ __align__(256) unsigned char g_accept_scratch[2ull * kNoAllocMaxRows * sizeof(RowStat)];

int accept_noalloc_max_rows() { return kNoAllocMaxRows; }

// Device address of the scratch array on the current device, looked up once per device with that device
// current (host code only sees a host-side stand-in for the symbol).  nullptr if the lookup fails.
void* accept_noalloc_scratch() {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

size_t accept_workspace_size(int B, int T, int V) {
    (void)V;
    size_t rows = (size_t)2 * B * T;
    return (rows * sizeof(RowStat) + 255) / 256 * 256;
}

cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    return a.logit_dt == SV_F32 ? launch_typed<SV_F32>(a, s) : launch_typed<SV_BF16>(a, s);
}

}  // namespace sv
