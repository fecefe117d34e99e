// attn_tc.cu -- tree-masked GQA attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Every draft-tree node attends to the request's KV prefix plus its own ancestors ("Aurora" post,
// section 2: a custom mask that follows the speculative tree's causal structure lets all branches of
// the tree be verified in one batched pass).  For one (request b, kv head hk) the T nodes x G query
// heads form T*G query rows that share every K/V tile, so the contraction is a real GEMM:
//   S = Q K^T  (M = 128 query rows, N = 64 kv positions, K = D = 128)      in TMEM
//   O += P V   (M = 128 query rows, N = D = 128, K = 64 kv positions)       in TMEM
// Work item = (request, kv head, group of <= 256 query rows, chunk of 64-position KV tiles).
//
// Roles in one CTA (persistent, one per SM):
//   warp 0      TMA producer: K and V tiles (64 x 128 bf16, 128-byte swizzle) into an 8-slot ring.
//   warp 1      TMEM owner (512 columns) and the single thread that issues tcgen05.mma.
//   warps 2-5   softmax warpgroup for M tile 0, warps 6-9 for M tile 1: each thread owns one query row
//               (one TMEM lane); it reads its S row, applies the ancestor mask on the tree block only,
//               keeps a running max / sum (log2 domain, lazy rescale of O when the max grows by > 2^8),
//               writes P (bf16) to shared memory, and finally normalises O and stores it.
// The S of tile n+1 is issued while the softmax still works on tile n.  Splits of one (request, head,
// group) write partial (O, m, l) to the workspace; the CTA that finishes the last chunk merges them.
// Every mbarrier wait is bounded; a time-out marks the requests SV_ERR_TIMEOUT and the CTA winds down,
// waiting (bounded) for its own copies and MMAs before it frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sv_internal.cuh"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTileN = 64;                       // kv positions per tile
constexpr int kGroupRows = 256;                  // query rows per work item (two M = 128 tiles)
constexpr int kStages = 8;                       // ring slots (one K or one V tile each)
constexpr int kSlotBytes = kTileN * kD * 2;      // 16 KB
constexpr int kHalfBytes = kSlotBytes / 2;       // one 64-column box of a tile
constexpr int kThreads = 320;
constexpr int kMinChunk = 4;                     // smallest split, in tiles
constexpr int kMaxSM = 160;                      // workspace is sized for up to this many SMs
constexpr float kRescaleThreshold = 8.0f;        // log2 units

constexpr int kSmemQ = 0;                        // [2 M tiles][2 halves][16 KB]
constexpr int kSmemP = 65536;                    // [2 M tiles][16 KB]
constexpr int kSmemRing = 98304;                 // [8][16 KB]
constexpr int kSmemBytes = kSmemRing + kStages * kSlotBytes;   // 229376
constexpr int kSmemAlloc = kSmemBytes + 1024;                  // + alignment slack

// TMEM columns: S of M tile j at 64*j, O of M tile j at 128 + 128*j (fp32, one lane per query row)
__host__ __device__ constexpr uint32_t col_S(int j) { return 64u * (uint32_t)j; }
__host__ __device__ constexpr uint32_t col_O(int j) { return 128u + 128u * (uint32_t)j; }

struct WorkItem {
    int b, hkqg, t0, t1, slot0, cn, pair, pad;   // hkqg = hk | qg << 16; cn = chunk | nchunks << 16
};

struct Header {
    int n_items;
    int total_tiles;
    int chunk;
    int pad[61];
};

struct Layout {
    long long items_off, done_off, valid_off, slots_off, total;
    int max_items, max_slots, pairs, qg;
};

__host__ __device__ inline long long align256(long long x) { return (x + 255) / 256 * 256; }
__host__ __device__ inline long long slot_bytes() { return (long long)kGroupRows * (kD + 2) * 4; }

__host__ __device__ inline Layout make_layout(int B, int T, int Hq, int Hkv, int kv_cap) {
    Layout l;
    const int G = Hq / Hkv;
    l.qg = (T * G + kGroupRows - 1) / kGroupRows;
    l.pairs = B * Hkv * l.qg;
    const int target = 2 * kMaxSM;
    const long long max_tiles = (long long)(kv_cap + kTileN - 1) / kTileN;
    long long ms = 2LL * target;
    if ((long long)l.pairs * max_tiles < ms) ms = (long long)l.pairs * max_tiles;
    l.max_slots = (int)ms;
    l.max_items = l.pairs + 2 * target;
    l.items_off = 256;
    l.done_off = align256(l.items_off + (long long)l.max_items * (long long)sizeof(WorkItem));
    l.valid_off = align256(l.done_off + (long long)l.pairs * 4);
    l.slots_off = align256(l.valid_off + (long long)B * 4);
    l.total = l.slots_off + (long long)l.max_slots * slot_bytes();
    return l;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// ------------------------------------------------------------------------------------------------ planner
// Block-wide exclusive scan over 1024 threads; returns the exclusive prefix, *total gets the sum.
__device__ int block_excl_scan(int v, int* s_warp, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
        int wx = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wx, o);
            if (lane >= o) wx += y;
        }
        s_warp[lane] = wx - w;          // exclusive warp offsets
        if (lane == 31) s_warp[32] = wx;
    }
    __syncthreads();
    int r = s_warp[warp] + x - v;
    *total = s_warp[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(1024) attn_plan_kernel(AttnArgs a, Layout lay, int target) {
    __shared__ int s_warp[33];
    __shared__ long long s_red[32];
    uint8_t* ws = (uint8_t*)a.ws;
    Header* hdr = (Header*)ws;
    WorkItem* items = (WorkItem*)(ws + lay.items_off);
    int* done = (int*)(ws + lay.done_off);
    int* valid = (int*)(ws + lay.valid_off);
    const int T = a.T, B = a.B, tid = threadIdx.x;
    const int G = a.Hq / a.Hkv;

    // 1. per-request validation
    for (int b = tid; b < B; b += blockDim.x) {
        const int32_t* par = a.parent + (size_t)b * T;
        int st = par[0] == -1 ? SV_OK : SV_ERR_BAD_TREE;
        for (int i = 1; i < T && st == SV_OK; ++i)
            if (par[i] < 0 || par[i] >= i) st = SV_ERR_BAD_TREE;
        const int L = a.kv_len[b];
        if (st == SV_OK && (L < 0 || L + T > a.kv_cap)) st = SV_ERR_INVALID_ARG;
        valid[b] = st == SV_OK;
        if (a.status) a.status[b] = st;
    }
    __syncthreads();
    // failed requests: zero outputs
    for (int b = 0; b < B; ++b) {
        if (valid[b]) continue;
        const size_t n = (size_t)T * a.Hq;
        uint16_t* o = (uint16_t*)a.out + (size_t)b * n * kD;
        for (size_t i = tid; i < n * kD; i += blockDim.x) o[i] = 0;
        if (a.lse) for (size_t i = tid; i < n; i += blockDim.x) a.lse[(size_t)b * n + i] = 0.f;
    }
    // 2. tiles per (request, head, group) and the chunk size
    auto tiles_of = [&](int p) -> int {
        const int b = p / (a.Hkv * lay.qg);
        return valid[b] ? (a.kv_len[b] + T + kTileN - 1) / kTileN : 0;
    };
    long long tot = 0;
    for (int p = tid; p < lay.pairs; p += blockDim.x) tot += tiles_of(p);
#pragma unroll
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if ((tid & 31) == 0) s_red[tid >> 5] = tot;
    __syncthreads();
    if (tid == 0) {
        long long t = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += s_red[w];
        s_red[0] = t;
    }
    __syncthreads();
    const long long total = s_red[0];
    long long chunk_ll = (total + target - 1) / target;
    const int chunk = (int)(chunk_ll < kMinChunk ? kMinChunk : chunk_ll);
    // 3. enumerate work items (exclusive scans over pairs, in rounds of blockDim)
    int carry_items = 0, carry_slots = 0;
    for (int base = 0; base < lay.pairs; base += blockDim.x) {
        const int p = base + tid;
        int nt = 0, nc = 0;
        if (p < lay.pairs) {
            nt = tiles_of(p);
            nc = (nt + chunk - 1) / chunk;
        }
        const int ns = nc > 1 ? nc : 0;
        int ti, ts;
        const int oi = block_excl_scan(nc, s_warp, &ti);
        const int os = block_excl_scan(ns, s_warp, &ts);
        if (p < lay.pairs) {
            done[p] = 0;
            const int b = p / (a.Hkv * lay.qg);
            const int rem = p - b * a.Hkv * lay.qg;
            const int hk = rem / lay.qg, qg = rem - hk * lay.qg;
            for (int c = 0; c < nc; ++c) {
                WorkItem w;
                w.b = b;
                w.hkqg = hk | (qg << 16);
                w.t0 = c * chunk;
                w.t1 = min(nt, (c + 1) * chunk);
                w.slot0 = nc > 1 ? carry_slots + os : -1;
                w.cn = c | (nc << 16);
                w.pair = p;
                w.pad = 0;
                items[carry_items + oi + c] = w;
            }
        }
        carry_items += ti;
        carry_slots += ts;
    }
    if (tid == 0) {
        hdr->n_items = carry_items;
        hdr->total_tiles = (int)total;
        hdr->chunk = chunk;
    }
    (void)G;
    __threadfence();
    pdl_launch_dependents();
}

// ------------------------------------------------------------------------------------------------ main kernel
struct MainShared {
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
    uint64_t q_full, o_full, drain;
    uint64_t anc[SV_MAX_T];
    uint32_t tmem;
    int err;
    int last;
};

__device__ __forceinline__ WorkItem load_item(const WorkItem* items, int i) { return items[i]; }

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs a,
               Layout lay, float scale_log2) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ MainShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sQ = smem_u32(smem + kSmemQ), sP = smem_u32(smem + kSmemP), sRing = smem_u32(smem + kSmemRing);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&sh.s_full[j], 1);
            mbar_init(&sh.s_free[j], 4);
            mbar_init(&sh.p_full[j], 4);
            mbar_init(&sh.pv_done[j], 1);
        }
        mbar_init(&sh.q_full, 8);
        mbar_init(&sh.o_full, 1);
        mbar_init(&sh.drain, 1);
        sh.err = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc(&sh.tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem;

    pdl_wait_prior();   // the work list written by the planner is visible from here on
    const uint8_t* ws = (const uint8_t*)a.ws;
    const int n_items = ((const volatile Header*)ws)->n_items;
    const WorkItem* items = (const WorkItem*)(ws + lay.items_off);
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G;
    volatile int* err = &sh.err;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t use = 0;
            for (int it = blockIdx.x; it < n_items && !*err; it += gridDim.x) {
                const WorkItem w = load_item(items, it);
                const int hk = w.hkqg & 0xffff;
                const int row0 = (w.b * a.Hkv + hk) * a.kv_cap;
                for (int t = w.t0; t < w.t1 && !*err; ++t) {
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
            const uint32_t first = use > (uint32_t)kStages ? use - kStages : 0;
            for (uint32_t u = first; u < use; ++u) mbar_wait(&sh.full[u % kStages], (u / kStages) & 1, &local);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idS = idesc_bf16_f32(128, kTileN, false, false);
            const uint32_t idO = idesc_bf16_f32(128, kD, false, true);
            uint32_t use = 0, gj[2] = {0, 0}, nit = 0;
            auto issue_S = [&](int j, uint32_t kslot) {
                const uint32_t qa = sQ + j * 32768, kb = sRing + kslot * kSlotBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t da = sdesc_sw128(qa + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = sdesc_sw128(kb + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
                    mma_f16_ss(tmem + col_S(j), da, db, idS, kk > 0);
                }
            };
            auto issue_PV = [&](int j, uint32_t vslot, bool acc) {
                const uint32_t pa = sP + j * 16384, vb = sRing + vslot * kSlotBytes;
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk) {
                    const uint64_t da = sdesc_sw128(pa + kk * 32, 16, 1024);
                    const uint64_t db = sdesc_sw128(vb + kk * 2048, kHalfBytes, 1024);
                    mma_f16_ss(tmem + col_O(j), da, db, idO, (acc || kk > 0) ? 1u : 0u);
                }
            };
            for (int it = blockIdx.x; it < n_items && !*err; it += gridDim.x, ++nit) {
                const WorkItem w = load_item(items, it);
                const int qg = w.hkqg >> 16;
                const int rows = min(kGroupRows, TG - qg * kGroupRows);
                const int MT = (rows + 127) / 128;
                const int nt = w.t1 - w.t0;
                if (!mbar_wait(&sh.q_full, nit & 1, err)) break;
                tc_fence_after();
                uint32_t kslot = use % kStages;
                if (!mbar_wait(&sh.full[kslot], (use / kStages) & 1, err)) break;
                ++use;
                tc_fence_after();
                for (int j = 0; j < MT; ++j) {
                    issue_S(j, kslot);
                    mma_commit(&sh.s_full[j]);
                }
                mma_commit(&sh.empty[kslot]);
                bool ok = true;
                for (int i = 0; i < nt && ok; ++i) {
                    const uint32_t vuse = use++;
                    const uint32_t vslot = vuse % kStages;
                    const bool has_next = i + 1 < nt;
                    uint32_t nslot = 0, nuse = 0;
                    if (has_next) {
                        nuse = use++;
                        nslot = nuse % kStages;
                    }
                    for (int j = 0; j < MT && ok; ++j) {
                        if (has_next) {
                            if (j == 0) ok = mbar_wait(&sh.full[nslot], (nuse / kStages) & 1, err);
                            ok = ok && mbar_wait(&sh.s_free[j], gj[j] & 1, err);
                            if (!ok) break;
                            tc_fence_after();
                            issue_S(j, nslot);
                            mma_commit(&sh.s_full[j]);
                        }
                        if (j == 0) ok = mbar_wait(&sh.full[vslot], (vuse / kStages) & 1, err);
                        ok = ok && mbar_wait(&sh.p_full[j], gj[j] & 1, err);
                        if (!ok) break;
                        tc_fence_after();
                        issue_PV(j, vslot, i > 0);
                        mma_commit(&sh.pv_done[j]);
                        ++gj[j];
                    }
                    if (!ok) break;
                    if (has_next) mma_commit(&sh.empty[nslot]);
                    mma_commit(&sh.empty[vslot]);
                }
                if (!ok) break;
                mma_commit(&sh.o_full);
            }
            // every MMA this thread issued has completed before TMEM is released
            mma_commit(&sh.drain);
            volatile int local = 0;
            mbar_wait(&sh.drain, 0, &local);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax warpgroups
        const int j = (warp - 2) >> 2;           // M tile owned by this warpgroup
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;        // query row inside the M tile (= TMEM lane)
        const int sm_tid = tid - 64;             // 0..255 over both warpgroups
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        uint32_t gj = 0, nit = 0, use = 0;
        // A warp that hits a time-out stops waiting and touching TMEM but still walks every named barrier,
        // so the other warpgroup can never be left waiting on it.
        bool dead = false;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(bar, parity, err));
            return !dead;
        };
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++nit) {
            const WorkItem w = load_item(items, it);
            const int b = w.b, hk = w.hkqg & 0xffff, qg = w.hkqg >> 16;
            const int rows = min(kGroupRows, TG - qg * kGroupRows);
            const int MT = (rows + 127) / 128;
            const int nt = w.t1 - w.t0;
            const int L = a.kv_len[b];
            const int qi = qg * kGroupRows + j * 128 + row;
            const bool valid_row = qi < TG;
            const int t_node = valid_row ? qi / G : 0, g_head = valid_row ? qi - (qi / G) * G : 0;
            // ancestor bitmasks of this request's nodes (the tree was validated by the planner)
            named_sync_softmax();
            if (sm_tid < T) {
                uint64_t m = 0;
                for (int x = sm_tid; x >= 0; x = a.parent[(size_t)b * T + x]) m |= 1ull << x;
                sh.anc[sm_tid] = m;
            }
            named_sync_softmax();
            dead = dead || *err;
            dead = __any_sync(0xffffffffu, dead);
            const uint64_t anc = valid_row ? sh.anc[t_node] : 0ull;
            // Q rows of this M tile -> shared memory (128-byte swizzle, two 64-column halves)
            if (!dead) {
                uint8_t* qdst = smem + kSmemQ + j * 32768;
                const uint4* src = (const uint4*)((const uint16_t*)a.q +
                                                  (((size_t)b * T + t_node) * a.Hq + (size_t)hk * G + g_head) * kD);
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 v = valid_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                    *(uint4*)(qdst + (c >> 3) * 16384 + sw128_offset(row, c & 7)) = v;
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_full);

            float m_run = -INFINITY, l_run = 0.f;
            const uint32_t use0 = use;
            use += 2u * nt;
            if (j < MT) {
                for (int i = 0; i < nt; ++i) {
                    const int pos0 = (w.t0 + i) * kTileN;
                    if (!wait(&sh.s_full[j], gj & 1)) break;
                    tc_fence_after();
                    __syncwarp();
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tmem + lane_addr + col_S(j), r0);
                    tmem_ld32(tmem + lane_addr + col_S(j) + 32, r1);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.s_free[j]);
                    float s[64];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        s[c] = __uint_as_float(r0[c]) * scale_log2;
                        s[c + 32] = __uint_as_float(r1[c]) * scale_log2;
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
                    float tmax = s[0];
#pragma unroll
                    for (int c = 1; c < 64; ++c) tmax = fmaxf(tmax, s[c]);
                    const float m_new = fmaxf(m_run, tmax);
                    const bool rescale = m_run != -INFINITY && m_new > m_run + kRescaleThreshold;
                    const float m_use = (m_run == -INFINITY || rescale) ? m_new : m_run;
                    // PV of the previous tile must be complete before P is overwritten / O rescaled
                    if (i > 0) {
                        if (!wait(&sh.pv_done[j], (gj - 1) & 1)) break;
                        tc_fence_after();
                    }
                    if (__any_sync(0xffffffffu, rescale)) {
                        const float alpha = rescale ? ex2(m_run - m_use) : 1.f;
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
                    float psum = 0.f;
                    {
                        uint8_t* pdst = smem + kSmemP + j * 16384;
                        const bool live = m_use != -INFINITY;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {   // 8 values -> one 16-byte chunk of the P row
                            uint32_t v[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float p0 = live ? ex2(s[8 * c + 2 * h] - m_use) : 0.f;
                                const float p1 = live ? ex2(s[8 * c + 2 * h + 1] - m_use) : 0.f;
                                psum += p0 + p1;
                                const __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                                v[h] = *reinterpret_cast<const uint32_t*>(&hb);
                            }
                            if (valid_row) *(uint4*)(pdst + sw128_offset(row, c)) = make_uint4(v[0], v[1], v[2], v[3]);
                        }
                    }
                    l_run = (m_run == -INFINITY) ? psum : l_run * (rescale ? ex2(m_run - m_use) : 1.f) + psum;
                    m_run = m_use;
                    // the last tile may hold cache rows past the tree block: zero those V rows (NaN-safe)
                    if (j == 0 && pos0 + kTileN > L + T) {
                        const uint32_t vuse = use0 + 2u * i + 1u;
                        if (!wait(&sh.full[vuse % kStages], (vuse / kStages) & 1)) break;
                        const int r_lo = max(0, L + T - pos0);
                        uint8_t* vdst = smem + kSmemRing + (vuse % kStages) * kSlotBytes;
                        for (int idx = row; idx < (kTileN - r_lo) * 16; idx += 128) {
                            const int r = r_lo + (idx >> 4), c = idx & 15;
                            *(uint4*)(vdst + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7)) = make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.p_full[j]);
                    ++gj;
                }
                // epilogue: all MMAs of the item are complete
                if (wait(&sh.o_full, nit & 1)) tc_fence_after();
            }
            const int chunk = w.cn & 0xffff, nchunks = w.cn >> 16;
            const size_t out_row = ((size_t)b * T + t_node) * a.Hq + (size_t)hk * G + g_head;
            const int grow = j * 128 + row;     // row inside the query group
            if (j < MT && !dead) {
                const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
                float* part = nullptr;
                if (w.slot0 >= 0)
                    part = (float*)((uint8_t*)a.ws + lay.slots_off + (long long)(w.slot0 + chunk) * slot_bytes());
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    __syncwarp();
                    tmem_ld32(tmem + lane_addr + col_O(j) + c * 32, o);
                    tmem_ld_wait();
                    if (valid_row) {
                        if (part) {
                            float4* dst = (float4*)(part + (size_t)grow * kD + c * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                                     __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
                        } else {
                            uint4* dst = (uint4*)((uint16_t*)a.out + out_row * kD + c * 32);
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
                }
                if (valid_row) {
                    if (part) {
                        part[(size_t)kGroupRows * kD + grow] = m_run;
                        part[(size_t)kGroupRows * kD + kGroupRows + grow] = l_run;
                    } else if (a.lse) {
                        a.lse[out_row] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
                    }
                }
            }
            if (w.slot0 >= 0) {
                // split: the CTA that completes the last chunk of this (request, head, group) merges
                __threadfence();
                named_sync_softmax();
                if (sm_tid == 0) {
                    const int prev = atomicAdd((int*)((uint8_t*)a.ws + lay.done_off) + w.pair, 1);
                    sh.last = prev == nchunks - 1;
                }
                named_sync_softmax();
                if (sh.last && j < MT && valid_row && !dead) {
                    __threadfence();
                    const uint8_t* base = (const uint8_t*)a.ws + lay.slots_off;
                    float M = -INFINITY;
                    for (int c = 0; c < nchunks; ++c) {
                        const float* pc = (const float*)(base + (long long)(w.slot0 + c) * slot_bytes());
                        M = fmaxf(M, __ldcg(pc + (size_t)kGroupRows * kD + grow));
                    }
                    float Lsum = 0.f;
                    for (int c = 0; c < nchunks; ++c) {
                        const float* pc = (const float*)(base + (long long)(w.slot0 + c) * slot_bytes());
                        const float mc = __ldcg(pc + (size_t)kGroupRows * kD + grow);
                        if (mc != -INFINITY) Lsum += __ldcg(pc + (size_t)kGroupRows * kD + kGroupRows + grow) * ex2(mc - M);
                    }
                    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
                    for (int d0 = 0; d0 < kD; d0 += 8) {
                        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        for (int c = 0; c < nchunks; ++c) {
                            const float* pc = (const float*)(base + (long long)(w.slot0 + c) * slot_bytes());
                            const float mc = __ldcg(pc + (size_t)kGroupRows * kD + grow);
                            if (mc == -INFINITY) continue;
                            const float wgt = ex2(mc - M);
                            const float4 x0 = __ldcg((const float4*)(pc + (size_t)grow * kD + d0));
                            const float4 x1 = __ldcg((const float4*)(pc + (size_t)grow * kD + d0 + 4));
                            acc[0] += x0.x * wgt; acc[1] += x0.y * wgt; acc[2] += x0.z * wgt; acc[3] += x0.w * wgt;
                            acc[4] += x1.x * wgt; acc[5] += x1.y * wgt; acc[6] += x1.z * wgt; acc[7] += x1.w * wgt;
                        }
                        uint32_t v[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const __nv_bfloat162 bb = __floats2bfloat162_rn(acc[2 * h] * inv, acc[2 * h + 1] * inv);
                            v[h] = *reinterpret_cast<const uint32_t*>(&bb);
                        }
                        *(uint4*)((uint16_t*)a.out + out_row * kD + d0) = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                    if (a.lse) a.lse[out_row] = (M + __log2f(Lsum)) * 0.69314718055994531f;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && sh.err) {   // a bounded wait gave up: mark every request this CTA touched
        for (int it = blockIdx.x; it < n_items; it += gridDim.x)
            if (a.status) a.status[items[it].b] = SV_ERR_TIMEOUT;
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
    if (D != kD || B < 1 || Hkv < 1 || Hq % Hkv) return 0;
    return (size_t)make_layout(B, T, Hq, Hkv, kv_cap).total;
}

bool attn_tc_supported(const AttnArgs& a) {
    return a.q_dt == SV_BF16 && a.kv_dt == SV_BF16 && a.D == kD && a.B >= 1 && a.B <= 4096 &&
           (long long)a.B * a.Hkv * a.kv_cap < (1LL << 31) - kTileN && (long long)a.T * (a.Hq / a.Hkv) < 65536 &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s) {
    const Layout lay = make_layout(a.B, a.T, a.Hq, a.Hkv, a.kv_cap);
    const int nsm = num_sms() < kMaxSM ? num_sms() : kMaxSM;
    CUtensorMap tmK, tmV;
    const long long rows = (long long)a.B * a.Hkv * a.kv_cap;
    if (!encode_kv_map(&tmK, a.k, rows) || !encode_kv_map(&tmV, a.v, rows)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    attn_plan_kernel<<<1, 1024, 0, s>>>(a, lay, 2 * nsm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    return launch_ex(attn_tc_kernel, dim3(nsm), dim3(kThreads), (size_t)kSmemAlloc, s, 1, true, tmK, tmV, a, lay,
                     scale * 1.4426950408889634f);
}

}  // namespace sv
