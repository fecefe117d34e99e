// attn_bwd_tc.cu -- backward of the tree-masked GQA attention on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA): bf16 Q, K, V, O and dO, D = 128, fp32 gradients.
//
// The draft trains on every accepted and rejected branch of its trees in one batched forward and backward pass
// ("Aurora" post, section 2).  With P recomputed from the forward's log-sum-exp, p = exp(s - lse), and
// delta = <dO, O> per query row:
//     dP = dO V^T,  dS = P o (dP - delta),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
// each a dense product over the (query rows x allowed positions) of a (request, kv head), under the same mask
// as the forward: the prefix [0, L) and the ancestors of the row's node in the tree block.
//
// Kernel 1 (dQ): one CTA per (128-row tile of the T*G query rows, kv head, request).  Per 128-position K/V tile:
//   S = Q K^T and dP = dO V^T (A = Q or dO, B = K or V, all K-major in shared memory) into TMEM; four warps, one
//   thread per row, form dS in bf16 over the S columns; dQ += dS K (A = dS from TMEM, B = K as an MN-major
//   operand, the forward's P V pattern).  Those warps also write delta of their rows for kernel 2.
// Kernel 2 (dK, dV): one CTA per (128-position tile, kv head, request) below L + T.  Per 128-row tile of the
//   query rows: S^T = K Q^T and dP^T = V dO^T (A = K or V, B = Q or dO); one thread per position forms P^T and
//   dS^T in bf16 over those columns; dV += P^T dO and dK += dS^T Q (B = dO or Q as MN-major operands).
// Cache rows past the tree block may hold anything (NaN included): their scores are replaced by zero weights with
// selects, and kernel 1 zeroes those rows of its K tile before dS K reads them.  Every mbarrier wait is bounded;
// a time-out marks the request SV_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sv_internal.cuh"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTile = 128;                  // positions per K/V tile, rows per query tile
constexpr int kSlotBytes = kTile * kD * 2;  // 32 KB: one bf16 tile, two 64-column boxes
constexpr int kBoxBytes = kSlotBytes / 2;
constexpr int kThreads = 256;               // warp 0 TMA, warp 1 MMA, warps 4-7 one TMEM lane quadrant each
constexpr int kSmemBytes = 6 * kSlotBytes;
constexpr int kSmemAlloc = kSmemBytes + 1024;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdShared {
    uint64_t in_full;                  // kernel 1: Q and dO; kernel 2: K and V
    uint64_t full[2], empty[2];        // the streamed ring: kernel 1 K (+ V), kernel 2 Q (+ dO)
    uint64_t s_full, d_full, acc_full, drain;
    float lse2[2][kTile], delta[2][kTile];   // kernel 2: the current query tile's rows
    unsigned long long anc[SV_MAX_T];
    int32_t par[SV_MAX_T];
    uint32_t tmem;
    int err;
};

__device__ __forceinline__ uint64_t at(uint64_t base, uint32_t saddr) { return base | (uint64_t)((saddr & 0x3FFFFu) >> 4); }

// bf16 pair of two floats, the first in the low half
__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// the request's parent array into shared memory and its status (parents, kv_len); every thread
__device__ int request_check(const AttnBwdArgs& a, int b, BwdShared& sh) {
    const int T = a.T;
    for (int i = threadIdx.x; i < T; i += blockDim.x) sh.par[i] = __ldg(a.parent + (size_t)b * T + i);
    __syncthreads();
    int st = block_tree_check(sh.par, T);
    const int L = __ldg(a.kv_len + b);
    if (st == SV_OK && (L < 0 || L + T > a.kv_cap)) st = SV_ERR_INVALID_ARG;
    return st;
}

// ------------------------------------------------------------------------------------------------ kernel 1: dQ
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                      const __grid_constant__ AttnBwdArgs a, float scale, float sl2) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ BwdShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rt = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G;
    const int st = request_check(a, b, sh);
    const int L = __ldg(a.kv_len + b);
    if (st != SV_OK) {   // zero gradients of the rows (kernel 2 writes nothing for this request)
        for (int i = tid; i < kTile * kD; i += kThreads) {
            const int r = i / kD, qi = rt * kTile + r;
            if (qi >= TG) continue;
            const int node = qi / G, gh = qi - node * G;
            const size_t orow = ((size_t)b * T + node) * a.Hq + (size_t)hk * G + gh;
            a.dq[orow * kD + (i - r * kD)] = 0.f;
            if (i - r * kD == 0) a.delta[orow] = 0.f;
        }
        if (a.status && rt == 0 && hk == 0 && tid == 0) a.status[b] = st;
        return;
    }
    // the request's status: SV_OK now, SV_ERR_TIMEOUT later from any CTA of it whose bounded wait gave up
    if (a.status && rt == 0 && hk == 0 && tid == 0) a.status[b] = SV_OK;
    const int ntiles = (L + T + kTile - 1) / kTile;
    const uint32_t sQ = smem_u32(smem), sG = sQ + kSlotBytes, sK = sQ + 2 * kSlotBytes, sV = sQ + 4 * kSlotBytes;
    if (tid == 0) {
        mbar_init(&sh.in_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.d_full, 4);   // the four dS warps
        mbar_init(&sh.acc_full, 1);
        mbar_init(&sh.drain, 1);
        sh.err = 0;
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(&sh.tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem;
    volatile int* err = &sh.err;
    const uint32_t cS = 0, cP = 128, cQ = 256;   // TMEM columns: S (then dS), dP, dQ

    if (warp == 0) {
        if (lane == 0) {
            // Q and dO of the 128 rows (128/G nodes x G heads per box), then K and V tiles into a 2-slot ring
            const int y0 = b * T + rt * kTile / G;
            mbar_arrive_expect_tx(&sh.in_full, 4 * kBoxBytes);
            for (int h = 0; h < 2; ++h) {
                tma_load_3d(smem + h * kBoxBytes, &tmQ, 64 * h, hk * G, y0, &sh.in_full);
                tma_load_3d(smem + kSlotBytes + h * kBoxBytes, &tmG, 64 * h, hk * G, y0, &sh.in_full);
            }
            const int yk = (b * a.Hkv + hk) * a.kv_cap;
            int t = 0;
            for (; t < ntiles && !*err; ++t) {
                const int s = t & 1;
                if (!mbar_wait(&sh.empty[s], ((t >> 1) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(&sh.full[s], 2 * kSlotBytes);
                for (int h = 0; h < 2; ++h) {
                    tma_load_2d(smem + 2 * kSlotBytes + s * kSlotBytes + h * kBoxBytes, &tmK, 64 * h, yk + t * kTile, &sh.full[s]);
                    tma_load_2d(smem + 4 * kSlotBytes + s * kSlotBytes + h * kBoxBytes, &tmV, 64 * h, yk + t * kTile, &sh.full[s]);
                }
            }
            // the copies this thread issued have landed before the CTA can exit
            volatile int local = 0;
            mbar_wait(&sh.in_full, 0, &local);
            for (int m = t > 2 ? t - 2 : 0; m < t && !local; ++m) mbar_wait(&sh.full[m & 1], (m >> 1) & 1, &local);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, kTile, false, false);
            const uint32_t idQ = idesc_bf16_f32(128, kD, false, true);
            const uint64_t dKm = sdesc_sw128(0, 16, 1024);          // K-major (Q, dO, K, V as B of S and dP)
            const uint64_t dMN = sdesc_sw128(0, kBoxBytes, 1024);   // MN-major (K as B of dS K)
            bool ok = mbar_wait(&sh.in_full, 0, err);
            tc_fence_after();
            for (int t = 0; t < ntiles && ok; ++t) {
                const int s = t & 1;
                ok = mbar_wait(&sh.full[s], (t >> 1) & 1, err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kb = sK + s * kSlotBytes, vb = sV + s * kSlotBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_f16_ss(tmem + cS, at(dKm, sQ + off), at(dKm, kb + off), idS, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_f16_ss(tmem + cP, at(dKm, sG + off), at(dKm, vb + off), idS, kk > 0);
                }
                mma_commit(&sh.s_full);
                ok = mbar_wait(&sh.d_full, t & 1, err);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    mma_f16_ts(tmem + cQ, tmem + cS + kk * 8, at(dMN, kb + kk * 2048), idQ, (t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&sh.empty[s]);
            }
            mma_commit(&sh.acc_full);
            mma_commit(&sh.drain);
            volatile int local = 0;
            mbar_wait(&sh.drain, 0, &local);
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int quad = warp & 3, row = quad * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const int qi = rt * kTile + row;
        const bool valid = qi < TG;
        const int node = valid ? qi / G : 0, gh = qi - node * G;
        const size_t orow = ((size_t)b * T + node) * a.Hq + (size_t)hk * G + gh;
        uint64_t anc = 0;
        if (valid) {
            int x = node;
            for (int step = 0; step < T && x >= 0 && x < T; ++step) {
                anc |= 1ull << x;
                const int px = sh.par[x];
                if (px >= x) break;
                x = px;
            }
        }
        float lse2 = 0.f, delta = 0.f;
        if (valid) {
            lse2 = __ldg(a.lse + orow) * kLog2e;
            const uint4* go = (const uint4*)((const uint16_t*)a.dout + orow * kD);
            const uint4* o = (const uint4*)((const uint16_t*)a.out + orow * kD);
#pragma unroll 4
            for (int i = 0; i < kD / 8; ++i) {
                const uint4 x = __ldg(go + i), y = __ldg(o + i);
                const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    delta += __uint_as_float(xs[e] << 16) * __uint_as_float(ys[e] << 16) +
                             __uint_as_float(xs[e] & 0xffff0000u) * __uint_as_float(ys[e] & 0xffff0000u);
            }
            a.delta[orow] = delta;
        }
        bool dead = false;
        for (int t = 0; t < ntiles; ++t) {
            if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&sh.s_full, t & 1, err));
            tc_fence_after();
            const int tile0 = t * kTile;
#pragma unroll 1
            for (int c = 0; c < 4 && !dead; ++c) {
                uint32_t rs[32], rp[32];
                tmem_ld32(tmem + lane_addr + cS + 32 * c, rs);
                tmem_ld32(tmem + lane_addr + cP + 32 * c, rp);
                tmem_ld_wait();
                reg_fence(rs);
                reg_fence(rp);
                // allowed positions of the 32 columns: the prefix, or an ancestor of the row's node
                const int pos0 = tile0 + 32 * c, np = L - pos0, a0 = pos0 - L;
                const uint32_t pre = np >= 32 ? ~0u : np <= 0 ? 0u : (1u << np) - 1u;
                const uint32_t tree = a0 >= 64 ? 0u : a0 >= 0 ? (uint32_t)(anc >> a0) : a0 > -32 ? (uint32_t)(anc << -a0) : 0u;
                const uint32_t al = valid ? (pre | tree) : 0u;
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float ds[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int k = 2 * e + h;
                        const float p = ex2f(fmaf(__uint_as_float(rs[k]), sl2, -lse2));
                        const float v = p * (__uint_as_float(rp[k]) - delta);
                        ds[h] = ((al >> k) & 1u) ? v : 0.f;   // a select: junk (NaN) scores give exactly 0
                    }
                    pk[e] = bf16x2(ds[0], ds[1]);
                }
                tmem_st16(tmem + lane_addr + cS + 16 * c, pk);
            }
            // the last tile's cache rows past the tree block become zeros before dS K reads them
            const int r_lo = L + T - tile0;
            if (r_lo < kTile) {
                uint8_t* kt = smem + 2 * kSlotBytes + (t & 1) * kSlotBytes;
                for (int idx = tid - 128; idx < (kTile - r_lo) * 16; idx += 128) {
                    const int rr = r_lo + (idx >> 4), ch = idx & 15;
                    *(uint4*)(kt + (ch >> 3) * kBoxBytes + sw128_offset(rr, ch & 7)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.d_full);
        }
        if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&sh.acc_full, 0, err));
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_addr + cQ + 32 * c, r);
            tmem_ld_wait();
            reg_fence(r);
            if (valid) {
                float4* dst = (float4*)(a.dq + orow * kD + 32 * c);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(__uint_as_float(r[4 * e]) * scale, __uint_as_float(r[4 * e + 1]) * scale,
                                         __uint_as_float(r[4 * e + 2]) * scale, __uint_as_float(r[4 * e + 3]) * scale);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (sh.err && a.status && tid == 0) a.status[b] = SV_ERR_TIMEOUT;
}

// ------------------------------------------------------------------------------------------------ kernel 2: dK, dV
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                       const __grid_constant__ AttnBwdArgs a, float scale, float sl2, int log2g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ BwdShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G;
    const int st = request_check(a, b, sh);
    const int L = __ldg(a.kv_len + b);
    if (st != SV_OK || t * kTile >= L + T) return;   // kernel 1 reports the status; nothing past L + T is written
    const int nq = (TG + kTile - 1) / kTile;
    const uint32_t sK = smem_u32(smem), sV = sK + kSlotBytes, sQ = sK + 2 * kSlotBytes, sG = sK + 4 * kSlotBytes;
    if (tid == 0) {
        mbar_init(&sh.in_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.s_full, 1);
        mbar_init(&sh.d_full, 4);
        mbar_init(&sh.acc_full, 1);
        mbar_init(&sh.drain, 1);
        sh.err = 0;
        for (int i = 0; i < T; ++i) sh.anc[i] = (1ull << i) | (i ? sh.anc[sh.par[i]] : 0ull);
        mbar_fence_init();
    }
    if (warp == 1) tmem_alloc(&sh.tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem;
    volatile int* err = &sh.err;
    const uint32_t cS = 0, cP = 128, cV = 256, cK = 384;   // TMEM: S^T (then P^T), dP^T (then dS^T), dV, dK

    if (warp == 0) {
        if (lane == 0) {
            const int yk = (b * a.Hkv + hk) * a.kv_cap + t * kTile;
            mbar_arrive_expect_tx(&sh.in_full, 2 * kSlotBytes);
            for (int h = 0; h < 2; ++h) {
                tma_load_2d(smem + h * kBoxBytes, &tmK, 64 * h, yk, &sh.in_full);
                tma_load_2d(smem + kSlotBytes + h * kBoxBytes, &tmV, 64 * h, yk, &sh.in_full);
            }
            int r = 0;
            for (; r < nq && !*err; ++r) {
                const int s = r & 1;
                if (!mbar_wait(&sh.empty[s], ((r >> 1) & 1) ^ 1, err)) break;
                const int y0 = b * T + r * kTile / G;
                mbar_arrive_expect_tx(&sh.full[s], 4 * kBoxBytes);
                for (int h = 0; h < 2; ++h) {
                    tma_load_3d(smem + 2 * kSlotBytes + s * kSlotBytes + h * kBoxBytes, &tmQ, 64 * h, hk * G, y0, &sh.full[s]);
                    tma_load_3d(smem + 4 * kSlotBytes + s * kSlotBytes + h * kBoxBytes, &tmG, 64 * h, hk * G, y0, &sh.full[s]);
                }
            }
            volatile int local = 0;
            mbar_wait(&sh.in_full, 0, &local);
            for (int m = r > 2 ? r - 2 : 0; m < r && !local; ++m) mbar_wait(&sh.full[m & 1], (m >> 1) & 1, &local);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, kTile, false, false);
            const uint32_t idO = idesc_bf16_f32(128, kD, false, true);
            const uint64_t dKm = sdesc_sw128(0, 16, 1024);
            const uint64_t dMN = sdesc_sw128(0, kBoxBytes, 1024);
            bool ok = mbar_wait(&sh.in_full, 0, err);
            tc_fence_after();
            for (int r = 0; r < nq && ok; ++r) {
                const int s = r & 1;
                ok = mbar_wait(&sh.full[s], (r >> 1) & 1, err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qb = sQ + s * kSlotBytes, gb = sG + s * kSlotBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_f16_ss(tmem + cS, at(dKm, sK + off), at(dKm, qb + off), idS, kk > 0);
                }
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    mma_f16_ss(tmem + cP, at(dKm, sV + off), at(dKm, gb + off), idS, kk > 0);
                }
                mma_commit(&sh.s_full);
                ok = mbar_wait(&sh.d_full, r & 1, err);
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint32_t acc = (r > 0 || kk > 0) ? 1u : 0u;
                    mma_f16_ts(tmem + cV, tmem + cS + kk * 8, at(dMN, gb + kk * 2048), idO, acc);
                    mma_f16_ts(tmem + cK, tmem + cP + kk * 8, at(dMN, qb + kk * 2048), idO, acc);
                }
                mma_commit(&sh.empty[s]);
            }
            mma_commit(&sh.acc_full);
            mma_commit(&sh.drain);
            volatile int local = 0;
            mbar_wait(&sh.drain, 0, &local);
        }
        __syncwarp();
    } else if (warp >= 4) {
        const int quad = warp & 3, p = quad * 32 + lane;   // this thread's position in the tile (= TMEM lane)
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const int pos = t * kTile + p;
        const bool in_tree = pos >= L && pos < L + T, prefix = pos < L;
        const int slot_a = pos - L;   // the tree node whose K / V sit at pos (in_tree)
        const int st_id = tid - 128;  // 0 .. 127 among the four warps
        bool dead = false;
        for (int r = 0; r < nq; ++r) {
            // lse * log2 e and delta of the query tile's 128 rows (padding rows: no row)
            {
                const int qi = r * kTile + st_id;
                float l2 = INFINITY, dl = 0.f;
                if (qi < TG) {
                    const int node = qi >> log2g, gh = qi - (node << log2g);
                    const size_t orow = ((size_t)b * T + node) * a.Hq + (size_t)hk * G + gh;
                    l2 = __ldg(a.lse + orow) * kLog2e;
                    dl = a.delta[orow];
                }
                sh.lse2[r & 1][st_id] = l2;
                sh.delta[r & 1][st_id] = dl;
                asm volatile("bar.sync 1, 128;" ::: "memory");
            }
            if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&sh.s_full, r & 1, err));
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 4 && !dead; ++c) {
                uint32_t rs[32], rp[32];
                tmem_ld32(tmem + lane_addr + cS + 32 * c, rs);
                tmem_ld32(tmem + lane_addr + cP + 32 * c, rp);
                tmem_ld_wait();
                reg_fence(rs);
                reg_fence(rp);
                // rows 32c .. 32c+31 of the query tile that see this position
                uint32_t al = 0;
                const int qi0 = r * kTile + 32 * c;
#pragma unroll 4
                for (int j = 0; j < 32; ++j) {
                    const int qi = qi0 + j;
                    const bool ok = qi < TG && (prefix || (in_tree && ((sh.anc[qi >> log2g] >> slot_a) & 1ull)));
                    al |= ok ? (1u << j) : 0u;
                }
                uint32_t pkp[16], pkd[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 2 * e + h;
                        const float pr = ex2f(fmaf(__uint_as_float(rs[j]), sl2, -sh.lse2[r & 1][32 * c + j]));
                        const float ds = pr * (__uint_as_float(rp[j]) - sh.delta[r & 1][32 * c + j]);
                        const bool ok = (al >> j) & 1u;
                        pv[h] = ok ? pr : 0.f;
                        dv[h] = ok ? ds : 0.f;
                    }
                    pkp[e] = bf16x2(pv[0], pv[1]);
                    pkd[e] = bf16x2(dv[0], dv[1]);
                }
                tmem_st16(tmem + lane_addr + cS + 16 * c, pkp);
                tmem_st16(tmem + lane_addr + cP + 16 * c, pkd);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.d_full);
        }
        if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(&sh.acc_full, 0, err));
        tc_fence_after();
        const size_t kvrow = ((size_t)b * a.Hkv + hk) * (size_t)a.kv_cap + pos;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {   // dV (columns 256..383) then dK (384..511), 32 at a time
            uint32_t rr[32];
            tmem_ld32(tmem + lane_addr + cV + 32 * c, rr);
            tmem_ld_wait();
            reg_fence(rr);
            if (pos < L + T && !dead) {
                const float sc = c < 4 ? 1.f : scale;
                float4* dst = (float4*)((c < 4 ? a.dv : a.dk) + kvrow * kD + 32 * (c & 3));
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(__uint_as_float(rr[4 * e]) * sc, __uint_as_float(rr[4 * e + 1]) * sc,
                                         __uint_as_float(rr[4 * e + 2]) * sc, __uint_as_float(rr[4 * e + 3]) * sc);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (sh.err && a.status && tid == 0) a.status[b] = SV_ERR_TIMEOUT;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// a cache as [B * Hkv * kv_cap][128] bf16, 64-column x 128-row boxes, 128-byte swizzle
bool encode_cache(CUtensorMap* m, const void* base, long long rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)kTile};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q or dO as [B*T][Hq][128] bf16: a box of 64 d x G heads x 128/G nodes is one 64-column half of 128 query rows
bool encode_rows(CUtensorMap* m, const void* base, const AttnBwdArgs& a) {
    auto enc = encoder();
    const int G = a.Hq / a.Hkv;
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a.Hq * kD * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)(kTile / G)};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_bwd_tc_supported(const AttnBwdArgs& a) {
    const int G = a.Hkv > 0 ? a.Hq / a.Hkv : 0;
    const auto al16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
    return a.q_dt == SV_BF16 && a.kv_dt == SV_BF16 && a.D == kD && G >= 1 && G <= kTile && (G & (G - 1)) == 0 &&
           (long long)a.B * a.Hkv * a.kv_cap < (1LL << 31) - kTile && (long long)a.B * a.T < (1LL << 31) &&
           al16(a.q) && al16(a.k) && al16(a.v) && al16(a.out) && al16(a.dout) && al16(a.dq) && al16(a.dk) &&
           al16(a.dv) && encoder() != nullptr;
}

cudaError_t launch_attn_bwd_tc(const AttnBwdArgs& a, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tmK, tmV, tmQ, tmG;
    const long long rows = (long long)a.B * a.Hkv * a.kv_cap;
    if (!encode_cache(&tmK, a.k, rows) || !encode_cache(&tmV, a.v, rows) || !encode_rows(&tmQ, a.q, a) ||
        !encode_rows(&tmG, a.dout, a))
        return cudaErrorInvalidValue;
    const float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    const float sl2 = scale * kLog2e;
    const int G = a.Hq / a.Hkv;
    int log2g = 0;
    while ((1 << log2g) < G) ++log2g;
    const int nq = (a.T * G + kTile - 1) / kTile;
    attn_bwd_dq_tc_kernel<<<dim3(nq, a.Hkv, a.B), kThreads, kSmemAlloc, s>>>(tmK, tmV, tmQ, tmG, a, scale, sl2);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    attn_bwd_dkv_tc_kernel<<<dim3((a.kv_cap + kTile - 1) / kTile, a.Hkv, a.B), kThreads, kSmemAlloc, s>>>(
        tmK, tmV, tmQ, tmG, a, scale, sl2, log2g);
    return cudaGetLastError();
}

}  // namespace sv
