// attn_tc.cu -- tree-masked GQA attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Every draft-tree node attends to the request's KV prefix plus its own ancestors ("Aurora" post,
// section 2: a custom mask that follows the speculative tree's causal structure lets all branches of
// the tree be verified in one batched pass).  For one (request b, kv head hk) the T nodes x G query
// heads form T*G query rows that share every K/V tile, so the contraction is a real GEMM:
//   S = Q K^T  (M = 128 query rows, N = 64 kv positions, K = D = 128)   A, B from shared memory
//   O += P V   (M = 128 query rows, N = D = 128, K = 64 kv positions)    A = P from TMEM, B = V
// A "pair" is (request, kv head, group of <= 256 query rows); it owns ceil((L_b + T) / 64) KV tiles.
//
// Scheduling (balanced, stream-K style): the tiles of all pairs form one sequence and CTA c of the
// persistent grid takes the contiguous range [c * total / G, (c + 1) * total / G); every CTA derives its
// range from kv_len alone in a short prologue.  A pair that crosses a range boundary is processed in
// segments; each segment leaves a partial result (normalised O in bf16, running max m and sum l) and a
// second kernel, attn_merge_kernel, merges them, validates every request and writes the status array.
//
// Roles in one CTA of attn_tc_kernel (persistent, one per SM):
//   warp 0      TMA producer: K and V tiles (64 x 128 bf16, 128-byte swizzle) into a 10-slot ring.
//   warps 1, 2  one tcgen05.mma issuer per M tile (warp 1 also owns the 512 TMEM columns).
//   warps 4-7   softmax warpgroup for M tile 0, warps 8-11 for M tile 1: each thread owns one query row
//               (one TMEM lane); it reads its S row, applies the ancestor mask on the tree block only,
//               keeps a running max / sum (lazy rescale of O when the max grows by > 2^8), writes P
//               (bf16) back into the same TMEM columns, and finally normalises O and stores it.
// S/P is double-buffered in TMEM per M tile: S of tile n+1 is computed while the softmax works on tile
// n.  Every mbarrier wait is bounded; a time-out raises a flag that turns the statuses into
// SV_ERR_TIMEOUT, and the CTA winds down, waiting (bounded) for its own copies and MMAs before it frees
// TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sv_internal.cuh"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTileN = 64;                       // kv positions per tile
constexpr int kGroupRows = 256;                  // query rows per pair (two M = 128 tiles)
constexpr int kStages = 10;                      // ring slots (one K or one V tile each)
constexpr int kSlotBytes = kTileN * kD * 2;      // 16 KB
constexpr int kHalfBytes = kSlotBytes / 2;       // one 64-column box of a tile
constexpr int kThreads = 384;
constexpr int kMaxGrid = 160;                    // the workspace is sized for grids up to this size
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr int kMergeThreads = 256;              // 8 warps

constexpr int kSmemQ = 0;                        // [2 M tiles][2 halves][16 KB]
constexpr int kSmemRing = 65536;                 // [10][16 KB]
constexpr int kSmemBytes = kSmemRing + kStages * kSlotBytes;   // 229376
constexpr int kSmemAlloc = kSmemBytes + 1024;                  // + alignment slack

// TMEM columns (fp32, one lane per query row): S / P of M tile j, buffer b at 64*(2j+b) (P, bf16 pairs,
// overwrites the first 32 columns of its S); O of M tile j at 256 + 128*j.  512 columns in all.
__host__ __device__ constexpr uint32_t col_S(int j, uint32_t b) { return 64u * (2u * (uint32_t)j + b); }
__host__ __device__ constexpr uint32_t col_O(int j) { return 256u + 128u * (uint32_t)j; }

// Workspace: a 256-byte header (time-out flag); per CTA a record of the split pair it completes (if any);
// two partial-result slots per CTA.
// A slot holds O / l in bf16 [256 rows][128], then m (log2 units) [256] and l [256] in fp32.
struct SplitRec {
    int pair;            // -1: this CTA completes no split pair (or the request's tree is malformed)
    int b, hk, qg;       // request, kv head and query group of the pair
    int cf;              // first CTA holding a segment of the pair
    int cf_slot;         // that CTA's slot for the pair (2 cf, or 2 cf + 1 if it began in an earlier pair)
    int pad[2];
};
__host__ __device__ constexpr long long slot_bytes() { return (long long)kGroupRows * kD * 2 + kGroupRows * 8; }
__host__ __device__ constexpr long long rec_off() { return 256; }
__host__ __device__ inline long long slots_off(int B) {
    (void)B;
    return (rec_off() + kMaxGrid * (long long)sizeof(SplitRec) + 255) / 256 * 256;
}
__host__ __device__ inline long long workspace_bytes(int B) { return slots_off(B) + 2LL * kMaxGrid * slot_bytes(); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// tiles of one request: its prefix plus its tree block, in 64-position tiles (0 if kv_len is invalid)
__device__ __forceinline__ int tiles_of(const AttnArgs& a, int b) {
    const int L = __ldg(a.kv_len + b);
    return (L >= 0 && L + a.T <= a.kv_cap) ? (L + a.T + kTileN - 1) / kTileN : 0;
}

// CTA owning global tile t when `total` tiles are split into `grid` ranges [c*total/grid, (c+1)*total/grid)
__device__ __forceinline__ int owner_of(long long t, long long total, int grid) {
    return (int)(((t + 1) * grid - 1) / total);
}

// Exclusive block scan (block size a multiple of 32, <= 1024); returns the prefix of v and writes the
// block total to *tot.  All threads must call it.
__device__ long long block_scan(long long v, long long* s_warp, long long* tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const long long w = lane < nw ? s_warp[lane] : 0;
        long long wx = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, wx, o);
            if (lane >= o) wx += y;
        }
        if (lane < nw) s_warp[lane] = wx - w;
        if (lane == 31) s_warp[32] = wx;
    }
    __syncthreads();
    const long long r = s_warp[warp] + x - v;
    *tot = s_warp[32];
    __syncthreads();
    return r;
}

// ------------------------------------------------------------------------------------------------ plan
// Where a CTA's range starts: global tile range [lo, hi), the request b0 that holds lo and the number of
// tiles before b0.  Pairs of one request share its tile count, so prefix sums over requests suffice.
struct Plan {
    long long total, lo, hi, req_start0;
    int grid, b0;
};

__device__ void make_plan(const AttnArgs& a, int HQ, Plan* out, long long* s_warp) {
    long long sum = 0;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) sum += tiles_of(a, b);
    long long reqs;
    block_scan(sum, s_warp, &reqs);
    const long long total = reqs * HQ;
    const int grid = (long long)gridDim.x < total ? (int)gridDim.x : (int)total;
    const long long lo = grid > 0 ? (long long)blockIdx.x * total / grid : 0;
    const long long hi = grid > 0 ? (long long)(blockIdx.x + 1) * total / grid : 0;
    if (threadIdx.x == 0) {
        out->total = total;
        out->grid = grid;
        out->lo = lo;
        out->hi = hi;
        out->b0 = a.B;
        out->req_start0 = total;
    }
    __syncthreads();
    long long carry = 0;
    for (int base = 0; base < a.B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        const long long v = b < a.B ? (long long)tiles_of(a, b) * HQ : 0;
        long long chunk;
        const long long s0 = carry + block_scan(v, s_warp, &chunk);
        if (b < a.B && v > 0 && lo < hi && s0 <= lo && lo < s0 + v) {
            out->b0 = b;
            out->req_start0 = s0;
        }
        carry += chunk;
    }
    __syncthreads();
}

// The segments of one CTA's range, in order; every role walks the same sequence.
struct Seg {
    int pair, b, hk, qg, t0, t1;   // tiles [t0, t1) of the pair
    bool split;                    // the pair crosses a range boundary
    int slot;                      // partial-result slot (split segments only)
    long long s0, s1;              // global tiles of the whole pair
};

struct SegIter {
    long long lo, hi, t, req_start;
    int b, lp, tiles, HQ, QG, c;
    const AttnArgs* a;
    __device__ void init(const AttnArgs& args, const Plan& p, int hq, int qg) {
        a = &args;
        HQ = hq;
        QG = qg;
        c = blockIdx.x;
        lo = p.lo;
        hi = p.hi;
        t = lo;
        b = p.b0;
        req_start = p.req_start0;
        tiles = b < args.B ? tiles_of(args, b) : 0;
        lp = tiles > 0 ? (int)((lo - req_start) / tiles) : 0;
    }
    __device__ bool next(Seg& s) {
        while (t < hi && b < a->B) {
            if (lp >= HQ || tiles == 0) {   // next request
                req_start += (long long)HQ * tiles;
                ++b;
                lp = 0;
                tiles = b < a->B ? tiles_of(*a, b) : 0;
                continue;
            }
            const long long s0 = req_start + (long long)lp * tiles, s1 = s0 + tiles;
            const long long e = s1 < hi ? s1 : hi;
            s.pair = b * HQ + lp;
            s.b = b;
            s.hk = lp / QG;
            s.qg = lp - s.hk * QG;
            s.t0 = (int)(t - s0);
            s.t1 = (int)(e - s0);
            s.split = !(s0 >= lo && s1 <= hi);
            s.slot = (lo >= s0 && lo < s1) ? 2 * c : 2 * c + 1;
            s.s0 = s0;
            s.s1 = s1;
            t = e;
            ++lp;
            return true;
        }
        return false;
    }
};

// ------------------------------------------------------------------------------------------------ main kernel
struct MainShared {
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2][2], p_full[2][2], pv_done[2][2];   // [M tile][buffer]
    uint64_t q_full[2], o_full[2], drain[2];
    Plan plan;
    long long scan[33];
    int32_t par[2][SV_MAX_T];                              // parent array of the current request, per warpgroup
    uint32_t tmem;
    int err;
};

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs a,
               float scale_log2) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ MainShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sQ = smem_u32(smem + kSmemQ), sRing = smem_u32(smem + kSmemRing);
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G, QG = (TG + kGroupRows - 1) / kGroupRows, HQ = a.Hkv * QG;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 2);          // one release per MMA issuer
        }
        for (int j = 0; j < 2; ++j) {
            for (int bf = 0; bf < 2; ++bf) {
                mbar_init(&sh.s_full[j][bf], 1);
                mbar_init(&sh.p_full[j][bf], 4);
                mbar_init(&sh.pv_done[j][bf], 1);
            }
            mbar_init(&sh.q_full[j], 4);
            mbar_init(&sh.o_full[j], 1);
            mbar_init(&sh.drain[j], 1);
        }
        sh.err = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc(&sh.tmem, 512);
    make_plan(a, HQ, &sh.plan, sh.scan);      // ends with __syncthreads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem;
    const Plan plan = sh.plan;
    volatile int* err = &sh.err;
    const bool active = (int)blockIdx.x < plan.grid;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0 && active) {
            uint32_t use = 0;
            SegIter si;
            si.init(a, plan, HQ, QG);
            Seg sg;
            while (!*err && si.next(sg)) {
                const int row0 = (sg.b * a.Hkv + sg.hk) * a.kv_cap;
                for (int t = sg.t0; t < sg.t1 && !*err; ++t) {
                    for (int kv = 0; kv < 2; ++kv, ++use) {
                        const uint32_t slot = use % kStages, round = use / kStages;
                        if (!mbar_wait(&sh.empty[slot], (round & 1) ^ 1, err)) break;
                        mbar_arrive_expect_tx(&sh.full[slot], kSlotBytes);
                        uint8_t* dst = smem + kSmemRing + slot * kSlotBytes;
                        const void* tm = kv ? (const void*)&tmV : (const void*)&tmK;
                        tma_load_2d(dst, tm, 0, row0 + t * kTileN, &sh.full[slot]);
                        tma_load_2d(dst + kHalfBytes, tm, 64, row0 + t * kTileN, &sh.full[slot]);
                    }
                }
            }
            // wait (bounded) for every copy still in flight before the CTA may exit
            volatile int local = 0;
            const uint32_t first_u = use > (uint32_t)kStages ? use - kStages : 0;
            for (uint32_t u = first_u; u < use; ++u) mbar_wait(&sh.full[u % kStages], (u / kStages) & 1, &local);
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------------------------------------------------------- MMA issuers, one per M tile
        const int j = warp - 1;
        if (lane == 0 && active) {
            const uint32_t idS = idesc_bf16_f32(128, kTileN, false, false);
            const uint32_t idO = idesc_bf16_f32(128, kD, false, true);
            const uint64_t dK = sdesc_sw128(0, 16, 1024);          // K-major operands (Q, K)
            const uint64_t dV = sdesc_sw128(0, kHalfBytes, 1024);  // MN-major V
            auto at = [](uint64_t base, uint32_t saddr) { return base | (uint64_t)((saddr & 0x3FFFFu) >> 4); };
            const uint32_t qa = sQ + j * 32768;
            uint32_t use = 0, g = 0, nseg = 0;
            bool ok = true;
            SegIter si;
            si.init(a, plan, HQ, QG);
            Seg sg;
            while (ok && !*err && si.next(sg)) {
                const int MT = (min(kGroupRows, TG - sg.qg * kGroupRows) + 127) / 128;
                const int nt = sg.t1 - sg.t0;
                if (j >= MT) {   // this M tile is empty here: release the slots in order, issue nothing
                    for (int u = 0; u < 2 * nt && ok; ++u) {
                        const uint32_t uu = use + u;
                        ok = mbar_wait(&sh.full[uu % kStages], (uu / kStages) & 1, err);
                        if (ok) mbar_arrive(&sh.empty[uu % kStages]);
                    }
                    use += 2 * nt;
                    continue;
                }
                if (!mbar_wait(&sh.q_full[j], nseg & 1, err)) break;
                tc_fence_after();
                auto issue_S = [&](int i) -> bool {
                    const uint32_t gi = g + i, sb = gi & 1, k = gi >> 1, ku = use + 2 * i;
                    if (!mbar_wait(&sh.full[ku % kStages], (ku / kStages) & 1, err)) return false;
                    // this S/P buffer was last read (as P) by the PV two tiles ago
                    if (k >= 1 && !mbar_wait(&sh.pv_done[j][sb], (k - 1) & 1, err)) return false;
                    tc_fence_after();
                    const uint32_t kb = sRing + (ku % kStages) * kSlotBytes;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk)
                        mma_f16_ss(tmem + col_S(j, sb), at(dK, qa + (kk >> 2) * 16384 + (kk & 3) * 32),
                                   at(dK, kb + (kk >> 2) * kHalfBytes + (kk & 3) * 32), idS, kk > 0);
                    mma_commit(&sh.s_full[j][sb]);
                    mma_commit(&sh.empty[ku % kStages]);
                    return true;
                };
                auto issue_PV = [&](int i) -> bool {
                    const uint32_t gi = g + i, pb = gi & 1, k = gi >> 1, vu = use + 2 * i + 1;
                    if (!mbar_wait(&sh.full[vu % kStages], (vu / kStages) & 1, err)) return false;
                    if (!mbar_wait(&sh.p_full[j][pb], k & 1, err)) return false;
                    tc_fence_after();
                    const uint32_t vb = sRing + (vu % kStages) * kSlotBytes;
#pragma unroll
                    for (int kk = 0; kk < kTileN / 16; ++kk)
                        mma_f16_ts(tmem + col_O(j), tmem + col_S(j, pb) + kk * 8, at(dV, vb + kk * 2048), idO,
                                   (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&sh.pv_done[j][pb]);
                    mma_commit(&sh.empty[vu % kStages]);
                    return true;
                };
                // S of tile i is issued before PV of tile i-1, so the softmax always has the next S early
                ok = issue_S(0);
                for (int i = 1; i < nt && ok; ++i) ok = issue_S(i) && issue_PV(i - 1);
                ok = ok && issue_PV(nt - 1);
                if (!ok) break;
                mma_commit(&sh.o_full[j]);
                use += 2 * nt;
                g += nt;
                ++nseg;
            }
            // every MMA this thread issued has completed before TMEM is released
            mma_commit(&sh.drain[j]);
            volatile int local = 0;
            mbar_wait(&sh.drain[j], 0, &local);
        }
        __syncwarp();
    } else if (warp >= 4 && active) {
        // ---------------------------------------------------------------- softmax warpgroups
        const int j = (warp - 4) >> 2;           // M tile owned by this warpgroup
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;        // query row inside the M tile (= TMEM lane)
        const int grow = j * 128 + row;          // row inside the pair's query group
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        uint32_t g = 0, nseg = 0, use = 0;
        // A warp that hits a time-out stops waiting and touching TMEM but keeps walking the segments (and
        // the warpgroup barrier), so no thread of its warpgroup is left waiting on it.
        bool dead = false;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(bar, parity, err));
            return !dead;
        };
        auto wg_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(2 + j) : "memory"); };
        SegIter si;
        si.init(a, plan, HQ, QG);
        Seg sg;
        bool first_seg = true;
        while (si.next(sg)) {
            const int b = sg.b, hk = sg.hk;
            const int MT = (min(kGroupRows, TG - sg.qg * kGroupRows) + 127) / 128;
            const int nt = sg.t1 - sg.t0;
            const uint32_t use0 = use;
            use += 2u * nt;
            if (j >= MT) continue;
            const int L = __ldg(a.kv_len + b);
            const int qi = sg.qg * kGroupRows + grow;
            const bool valid_row = qi < TG;
            const int t_node = valid_row ? qi / G : 0, g_head = valid_row ? qi - (qi / G) * G : 0;
            const size_t out_row = ((size_t)b * T + t_node) * a.Hq + (size_t)hk * G + g_head;
            uint8_t* part = sg.split ? (uint8_t*)a.ws + slots_off(a.B) + (long long)sg.slot * slot_bytes() : nullptr;
            // ancestors of this row's node from the request's parent array (walk bounded by T, so a malformed
            // array cannot trap; such requests are zeroed and flagged by the merge kernel)
            wg_sync();
            if (row < T) sh.par[j][row] = __ldg(a.parent + (size_t)b * T + row);
            wg_sync();
            if (j == 0 && row == 0 && first_seg) {
                // the pair that began in an earlier CTA range and ends in this one is merged by attn_merge_kernel
                int bad = sh.par[0][0] != -1;
                for (int x = 1; x < T; ++x) bad |= sh.par[0][x] < 0 || sh.par[0][x] >= x;
                SplitRec r;
                r.pair = (sg.s0 < plan.lo && sg.s1 <= plan.hi && !bad) ? sg.pair : -1;
                r.b = b;
                r.hk = hk;
                r.qg = sg.qg;
                r.cf = owner_of(sg.s0, plan.total, plan.grid);
                r.cf_slot = ((long long)r.cf * plan.total / plan.grid == sg.s0) ? 2 * r.cf : 2 * r.cf + 1;
                r.pad[0] = r.pad[1] = 0;
                ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x] = r;
            }
            first_seg = false;
            uint64_t anc = 0;
            if (valid_row) {
                int x = t_node;
                for (int step = 0; step < T && x >= 0 && x < T; ++step) {
                    anc |= 1ull << x;
                    const int px = sh.par[j][x];
                    if (px >= x) break;
                    x = px;
                }
            }
            dead = __any_sync(0xffffffffu, dead || *err);
            // Q rows of this M tile -> shared memory (128-byte swizzle, two 64-column halves)
            if (!dead) {
                uint8_t* qdst = smem + kSmemQ + j * 32768;
                const uint4* src = (const uint4*)((const uint16_t*)a.q + out_row * kD);
                uint4 v[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) v[c] = valid_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < 16; ++c) *(uint4*)(qdst + (c >> 3) * 16384 + sw128_offset(row, c & 7)) = v[c];
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_full[j]);

            float m_run = -INFINITY, l_run = 0.f;    // running max (raw score units) and sum of 2^(...)
            for (int i = 0; i < nt; ++i) {
                const uint32_t gi = g + i, sb = gi & 1, k = gi >> 1;
                const int pos0 = (sg.t0 + i) * kTileN;
                if (!wait(&sh.s_full[j][sb], k & 1)) break;
                tc_fence_after();
                __syncwarp();
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_addr + col_S(j, sb), r0);
                tmem_ld32(tmem + lane_addr + col_S(j, sb) + 32, r1);
                tmem_ld_wait();
                float s[64];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    s[c] = __uint_as_float(r0[c]);
                    s[c + 32] = __uint_as_float(r1[c]);
                }
                if (!valid_row) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = -INFINITY;
                } else if (pos0 + kTileN > L) {   // tile reaches the tree block: ancestor mask
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int pos = pos0 + c;
                        const int a_idx = pos - L;
                        const bool allow = pos < L || (a_idx < T && ((anc >> (a_idx & 63)) & 1ull));
                        if (!allow) s[c] = -INFINITY;
                    }
                }
                float mx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    mx[c] = fmaxf(fmaxf(fmaxf(s[c], s[c + 8]), fmaxf(s[c + 16], s[c + 24])),
                                  fmaxf(fmaxf(s[c + 32], s[c + 40]), fmaxf(s[c + 48], s[c + 56])));
                const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const float m_new = fmaxf(m_run, tmax);
                const bool rescale = m_run != -INFINITY && (m_new - m_run) * scale_log2 > kRescaleThreshold;
                const float m_use = (m_run == -INFINITY || rescale) ? m_new : m_run;
                const float alpha = rescale ? ex2((m_run - m_use) * scale_log2) : 1.f;
                if (__any_sync(0xffffffffu, rescale)) {
                    // O holds PV of the previous tile: wait for it, then rescale this warp's rows
                    if (!wait(&sh.pv_done[j][(gi - 1) & 1], ((gi - 1) >> 1) & 1)) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        __syncwarp();
                        tmem_ld32(tmem + lane_addr + col_O(j) + c * 32, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tmem + lane_addr + col_O(j) + c * 32, o);
                    }
                    tmem_st_wait();
                }
                // P = 2^(s*scale - m) in bf16, packed in pairs (even k in the low half) into the S columns
                float ps[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
                {
                    const bool live = m_use != -INFINITY;
                    const float moff = live ? -m_use * scale_log2 : 0.f;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float p0 = live ? ex2(fmaf(s[2 * c], scale_log2, moff)) : 0.f;
                        const float p1 = live ? ex2(fmaf(s[2 * c + 1], scale_log2, moff)) : 0.f;
                        ps[c & 3] += p0 + p1;
                        const __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                        pk[c] = *reinterpret_cast<const uint32_t*>(&hb);
                    }
                }
                __syncwarp();
                tmem_st32(tmem + lane_addr + col_S(j, sb), pk);
                const float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
                l_run = (m_run == -INFINITY) ? psum : l_run * alpha + psum;
                m_run = m_use;
                // the last tile may hold cache rows past the tree block: zero those V rows (NaN-safe).
                // Both warpgroups write the same zeros; each fences its own writes before its PV.
                if (pos0 + kTileN > L + T) {
                    const uint32_t vu = use0 + 2u * i + 1u;
                    if (wait(&sh.full[vu % kStages], (vu / kStages) & 1)) {
                        const int r_lo = max(0, L + T - pos0);
                        uint8_t* vdst = smem + kSmemRing + (vu % kStages) * kSlotBytes;
                        for (int idx = row; idx < (kTileN - r_lo) * 16; idx += 128) {
                            const int r = r_lo + (idx >> 4), c = idx & 15;
                            *(uint4*)(vdst + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7)) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[j][sb]);
                if (dead) break;
            }
            // epilogue: all MMAs of the segment are complete
            if (wait(&sh.o_full[j], nseg & 1)) tc_fence_after();
            g += nt;
            ++nseg;
            if (dead) continue;
            const float m_log2 = m_run * scale_log2;
            // normalised O (bf16) either to the output row or to this segment's partial slot
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            uint16_t* dst_row = part ? (uint16_t*)part + (size_t)grow * kD : (uint16_t*)a.out + out_row * kD;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                __syncwarp();
                tmem_ld32(tmem + lane_addr + col_O(j) + c * 32, o);
                tmem_ld_wait();
                if (valid_row) {
                    uint4* dst = (uint4*)(dst_row + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t v[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const __nv_bfloat162 bb = __floats2bfloat162_rn(__uint_as_float(o[8 * e + 2 * h]) * inv_l,
                                                                            __uint_as_float(o[8 * e + 2 * h + 1]) * inv_l);
                            v[h] = *reinterpret_cast<const uint32_t*>(&bb);
                        }
                        dst[e] = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                }
            }
            if (valid_row) {
                if (part) {
                    float* ml = (float*)(part + (size_t)kGroupRows * kD * 2);
                    ml[grow] = m_log2;
                    ml[kGroupRows + grow] = l_run;
                } else if (a.lse) {
                    a.lse[out_row] = (m_log2 + __log2f(l_run)) * 0.69314718055994531f;
                }
            }
        }
    }
    if (!active && tid == 0) {   // CTAs beyond the used grid complete no split pair
        SplitRec r = {};
        r.pair = -1;
        ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x] = r;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && sh.err) *(volatile int*)a.ws = 1;   // a bounded wait gave up: statuses become TIMEOUT
}

// ------------------------------------------------------------------------------------------------ merge kernel
// Runs after attn_tc_kernel (programmatic dependent launch): validates every request (statuses, zero
// outputs for failed ones) and merges the segments of every pair that crossed a CTA range boundary.
// One merge unit = (record of CTA c, 16 rows): each warp merges two rows, lanes covering 4 of the 128 dims
// (coalesced 8-byte loads), with every load of a row issued before any of them is used.
constexpr int kMergeRows = 16;
constexpr int kMergeUnits = kGroupRows / kMergeRows;   // per record

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(AttnArgs a, int grid_main) {
    __shared__ int s_bad;
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait_prior();   // attention results are visible from here on
    const bool timeout = *(volatile const int*)a.ws != 0;

    // 1. statuses, and zero outputs of failed requests
    for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        if (tid == 0) s_bad = 0;
        __syncthreads();
        if (tid < T) {
            const int p = __ldg(a.parent + (size_t)b * T + tid);
            if (tid == 0 ? p != -1 : (p < 0 || p >= tid)) s_bad = 1;
        }
        __syncthreads();
        const int L = __ldg(a.kv_len + b);
        int st = s_bad ? SV_ERR_BAD_TREE : SV_OK;
        if (st == SV_OK && (L < 0 || L + T > a.kv_cap)) st = SV_ERR_INVALID_ARG;
        if (timeout) st = SV_ERR_TIMEOUT;
        if (tid == 0 && a.status) a.status[b] = st;
        if (st != SV_OK && st != SV_ERR_TIMEOUT) {
            const size_t n = (size_t)T * a.Hq;
            uint16_t* o = (uint16_t*)a.out + (size_t)b * n * kD;
            for (size_t i = tid; i < n * kD / 8; i += blockDim.x) ((uint4*)o)[i] = make_uint4(0, 0, 0, 0);
            if (a.lse) for (size_t i = tid; i < n; i += blockDim.x) a.lse[(size_t)b * n + i] = 0.f;
        }
        __syncthreads();
    }
    if (timeout) return;
    // 2. merges
    const SplitRec* recs = (const SplitRec*)((const uint8_t*)a.ws + rec_off());
    const uint8_t* slots = (const uint8_t*)a.ws + slots_off(a.B);
    for (int u = blockIdx.x; u < grid_main * kMergeUnits; u += gridDim.x) {
        const int cl = u / kMergeUnits, rb = u - cl * kMergeUnits;
        const SplitRec rec = recs[cl];
        if (rec.pair < 0) continue;
        const int rows = min(kGroupRows, TG - rec.qg * kGroupRows);
        float m[2][4], l[2][4];
        uint2 x[2][4];
        int rr[2];
        // contributors are CTAs cf..cl; CTA c > cf holds the pair in its first slot 2c
        for (int h = 0; h < 2; ++h) rr[h] = rb * kMergeRows + warp * 2 + h;
        float M[2] = {-INFINITY, -INFINITY}, Ls[2] = {0.f, 0.f}, acc[2][4] = {};
        for (int c0 = rec.cf; c0 <= cl; c0 += 4) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = min(c0 + i, cl);
                    const int sidx = c == rec.cf ? rec.cf_slot : 2 * c;
                    const uint8_t* base = slots + (long long)sidx * slot_bytes();
                    const int r = min(rr[h], rows - 1);
                    const float* ml = (const float*)(base + (size_t)kGroupRows * kD * 2);
                    m[h][i] = c0 + i <= cl ? __ldcg(ml + r) : -INFINITY;
                    l[h][i] = __ldcg(ml + kGroupRows + r);
                    x[h][i] = __ldcg((const uint2*)((const uint16_t*)base + (size_t)r * kD) + lane);
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float mn = M[h];
#pragma unroll
                for (int i = 0; i < 4; ++i) mn = fmaxf(mn, m[h][i]);
                const float sc = M[h] == -INFINITY ? 0.f : ex2(M[h] - mn);   // rescale the running sums
                Ls[h] *= sc;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[h][e] *= sc;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float w = m[h][i] == -INFINITY ? 0.f : l[h][i] * ex2(m[h][i] - mn);
                    Ls[h] += w;
                    acc[h][0] += __uint_as_float(x[h][i].x << 16) * w;
                    acc[h][1] += __uint_as_float(x[h][i].x & 0xffff0000u) * w;
                    acc[h][2] += __uint_as_float(x[h][i].y << 16) * w;
                    acc[h][3] += __uint_as_float(x[h][i].y & 0xffff0000u) * w;
                }
                M[h] = mn;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = rr[h];
            if (r >= rows) continue;
            const int qi = rec.qg * kGroupRows + r, t_node = qi / G, g_head = qi - t_node * G;
            const size_t out_row = ((size_t)rec.b * T + t_node) * a.Hq + (size_t)rec.hk * G + g_head;
            const float inv = Ls[h] > 0.f ? 1.f / Ls[h] : 0.f;
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[h][0] * inv, acc[h][1] * inv);
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[h][2] * inv, acc[h][3] * inv);
            ((uint2*)((uint16_t*)a.out + out_row * kD))[lane] =
                make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
            if (a.lse && lane == 0) a.lse[out_row] = (M[h] + __log2f(Ls[h])) * 0.69314718055994531f;
        }
    }
}

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            n = 1;
    }
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

bool encode_kv_map(CUtensorMap* m, const void* base, long long rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, kTileN};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t attn_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap) {
    (void)T; (void)kv_cap;
    if (D != kD || Hkv < 1 || Hq % Hkv) return 0;
    return (size_t)workspace_bytes(B);
}

bool attn_tc_supported(const AttnArgs& a) {
    return a.q_dt == SV_BF16 && a.kv_dt == SV_BF16 && a.D == kD && a.B >= 1 &&
           (long long)a.B * a.Hkv * a.kv_cap < (1LL << 31) - kTileN && (long long)a.T * (a.Hq / a.Hkv) < 65536 &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s) {
    const int grid = num_sms() < kMaxGrid ? num_sms() : kMaxGrid;
    CUtensorMap tmK, tmV;
    const long long rows = (long long)a.B * a.Hkv * a.kv_cap;
    if (!encode_kv_map(&tmK, a.k, rows) || !encode_kv_map(&tmV, a.v, rows)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    // the time-out flag starts clear; the attention kernel only ever sets it
    cudaError_t e = cudaMemsetAsync(a.ws, 0, 4, s);
    if (e != cudaSuccess) return e;
    const float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    e = launch_ex(attn_tc_kernel, dim3(grid), dim3(kThreads), (size_t)kSmemAlloc, s, 1, false, tmK, tmV, a,
                  scale * 1.4426950408889634f);
    if (e != cudaSuccess) return e;
    return launch_ex(attn_merge_kernel, dim3(grid * kMergeUnits), dim3(kMergeThreads), 0, s, 1, true, a, grid);
}

}  // namespace sv
