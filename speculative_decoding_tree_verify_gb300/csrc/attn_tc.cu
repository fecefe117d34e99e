// attn_tc.cu -- tree-masked GQA attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Every draft-tree node attends to the request's KV prefix plus its own ancestors ("Aurora" post,
// section 2: a custom mask that follows the speculative tree's causal structure lets all branches of
// the tree be verified in one batched pass).  For one (request b, kv head hk) the T nodes x G query
// heads form T*G query rows that share every K/V tile, so the contraction is a real GEMM.  Each CTA
// owns one M tile of 128 query rows:
//   S = Q K^T  (M = 128 query rows, N = 128 kv positions, K = D = 128)   A = Q, B = K, both in shared memory
//   O += P V   (M = 128 query rows, N = D = 128, K = 128 kv positions)   A = P from TMEM, B = V
// A "unit" is (request, kv head, group of query rows); it owns ceil((L_b + T) / 128) KV tiles.  When
// T*G > 128 a unit has 256 rows and is processed by a cluster of two CTAs (one M tile each) that receive
// every K/V tile together: CTA 0 loads the K tile and CTA 1 the V tile, each multicast to both, so
// L2 and HBM deliver each tile once.  Otherwise a unit is one M tile and one CTA.
//
// Scheduling (balanced, stream-K style): the tiles of all units form one sequence and cluster c of the
// persistent grid takes the contiguous range [c * total / G, (c + 1) * total / G); every CTA derives its
// range from kv_len alone in a short prologue.  A unit that crosses a range boundary is processed in
// segments; each segment leaves a partial result (normalised O in bf16, running max m and sum l) and a
// second kernel, attn_merge_kernel, merges them, validates every request and writes the status array.
//
// Roles in one CTA of attn_tc_kernel (persistent, 12 warps):
//   warps 0, 3   TMA producers (bf16 caches): warp 0 loads the K tiles into a 2-slot K ring, warp 3 the V
//                tiles into a 2-slot V ring (128 x 128 bf16 as two 64-column boxes, 128-byte swizzle), so
//                K tiles, released as soon as S is computed, run ahead of the V tiles held until the PV.
//                e4m3 caches: warp 0 loads both into a staging ring and warp 3 converts them to f16.
//   warp 1       S issuer (also owns the 512 TMEM columns); warp 2 PV issuer.
//   warps 4-11   softmax: two warps per TMEM lane quadrant, each owning 32 query rows x 64 of the 128
//                columns of every S tile.  A thread reads its part of an S row, applies the ancestor
//                mask on the tree block only, keeps a running max (shared with the other half of the
//                row once per tile) and a partial sum, rescales O lazily when the max grows by > 2^8,
//                writes P to TMEM, and finally normalises its half of the O row and stores it.
// Q sits in shared memory (the A operand of S = Q K^T); TMEM holds O, two S buffers and two P buffers, so
// S of tile n+1 is computed while the softmax works on tile n, and the PV of tile n may complete while the
// softmax writes P of tile n+1.  Every mbarrier wait is bounded;
// a time-out raises a flag that turns the statuses into SV_ERR_TIMEOUT, and the CTA winds down, waiting
// (bounded) for its own copies and MMAs before it frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "sv_internal.cuh"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTileN = 128;                      // kv positions per tile
constexpr int kRows = 128;                       // query rows per CTA (one M tile)
constexpr int kKSlots = 2, kVSlots = 2;          // bf16 KV: a K ring and a V ring (one 32 KB tile per slot)
constexpr int kRing16 = 3;                       // e4m3 KV: one ring of converted f16 K and V tiles, alternating
constexpr int kStage8 = 4;                       // e4m3 staging slots (FP8 KV only)
constexpr int kSlot8Bytes = kTileN * kD;         // 16 KB: one e4m3 K or V tile
constexpr int kSlotBytes = kTileN * kD * 2;      // 32 KB
constexpr int kBoxBytes = kSlotBytes / 2;        // one 64-column box: 128 rows x 128 bytes
constexpr int kSplit16 = 2;                      // bf16 caches: softmax warps per query row (4 measured slower)
constexpr int kThreads = 128 + 128 * kSplit16;   // 4 role warps + 4 * kSplit16 softmax warps (bf16 caches)
constexpr int kConv = 4;                         // e4m3 -> f16 converter warps (e4m3 caches): warps 3, 12, 13, 14
constexpr int kThreads8 = 480;                   // 15 warps (e4m3 caches)
template <bool KV8>
constexpr int threads_of() { return KV8 ? kThreads8 : kThreads; }
constexpr int kMaxGrid = 160;                    // the workspace is sized for grids up to this size
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr int kMergeThreads = 256;               // 8 warps

constexpr int kSmemQ = 0;                        // Q of the M tile: [buffer][2 halves][16 KB] (2 buffers for bf16)
// ring: bf16 KV: [2 K + 2 V][32 KB] after two Q buffers; FP8 KV: [3][32 KB] f16 slots after one Q buffer, then
template <bool KV8>
__host__ __device__ constexpr int ring_off() { return KV8 ? kSlotBytes : 2 * kSlotBytes; }
constexpr int kSmemStage = 4 * kSlotBytes;       //   the e4m3 staging slots [4][16 KB]
constexpr int kSmemBytes = 6 * kSlotBytes;       // 196608 either way
static_assert(kSmemStage + kStage8 * kSlot8Bytes == kSmemBytes, "FP8 smem layout");
constexpr int kSmemAlloc = kSmemBytes + 1024;                  // + alignment slack

// TMEM columns (32-bit, one lane per query row): O at 0 (128 columns), S buffer b at 128 + 128*b, P buffer
// b at 384 + 64*b (bf16 pairs).  S and P are double-buffered: S of tile n+1 is computed while the softmax
// works on tile n, and the PV of tile n may finish while the softmax writes P of tile n+1.
constexpr int kPBufs = 2;
__host__ __device__ constexpr uint32_t col_O() { return 0u; }
__host__ __device__ constexpr uint32_t col_S(uint32_t b) { return 128u + 128u * b; }
__host__ __device__ constexpr uint32_t col_P(uint32_t b) { return 384u + 64u * b; }

// Workspace: a 256-byte header (time-out flag); per CTA a record of the split unit it completes (if any);
// two partial-result slots per CTA.  A slot holds O / l in bf16 [128 rows][128], then m (log2 units)
// [128] and l [128] in fp32.
struct SplitRec {
    int unit;            // -1: this CTA completes no split unit (or the request's tree is malformed)
    int b, hk;           // request and kv head of the unit
    int row0;            // first query row (index into the T*G rows of the kv head) of this CTA's M tile
    int rows;            // valid rows of this CTA's M tile
    int cf;              // first CTA (same cluster rank) holding a segment of the unit
    int cf_slot;         // that CTA's slot for the unit (2 cf, or 2 cf + 1 if it began in an earlier unit)
    int err;             // 1: a bounded wait of this CTA gave up (written last, on every launch)
};
__host__ __device__ constexpr long long slot_bytes() { return (long long)kRows * kD * 2 + kRows * 8; }
__host__ __device__ constexpr long long rec_off() { return 256; }
__host__ __device__ constexpr long long slots_off() {
    return (rec_off() + kMaxGrid * (long long)sizeof(SplitRec) + 255) / 256 * 256;
}
__host__ __device__ constexpr long long workspace_bytes() { return slots_off() + 2LL * kMaxGrid * slot_bytes(); }

__device__ __forceinline__ float max3(float x, float y, float z) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
    return r;
}

// two e4m3 (low byte -> low half) to two f16, exactly
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// two floats to a bf16 or f16 pair (the first in the low half)
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (F16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// pairs of floats in one 64-bit register pair, and the packed two-lane f32 arithmetic of sm_100+ (each lane
// rounds exactly as the scalar instruction does)
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Slot (index into the ring's slots and full/empty barriers) and round of the n-th K (kv = 0) or V (kv = 1)
// tile a CTA consumes.  bf16 caches: separate K and V rings, so that K tiles, released as soon as S is
// computed, run ahead of the V tiles, which are held until the PV; e4m3 caches: one ring, K and V alternating.
template <bool KV8>
__device__ __forceinline__ void ring_pos(uint32_t n, int kv, uint32_t& slot, uint32_t& round) {
    if constexpr (KV8) {
        const uint32_t u = 2 * n + (uint32_t)kv;
        slot = u % kRing16;
        round = u / kRing16;
    } else if (kv == 0) {
        slot = n % kKSlots;
        round = n / kKSlots;
    } else {
        slot = kKSlots + n % kVSlots;
        round = n / kVSlots;
    }
}

// tiles of one request: its prefix plus its tree block, in 128-position tiles (0 if kv_len is invalid)
__device__ __forceinline__ int tiles_of(const AttnArgs& a, int b) {
    const int L = __ldg(a.kv_len + b);
    return (L >= 0 && L + a.T <= a.kv_cap) ? (L + a.T + kTileN - 1) / kTileN : 0;
}

// cluster owning global tile t when `total` tiles are split into `grid` ranges [c*total/grid, (c+1)*total/grid)
__device__ __forceinline__ int owner_of(int t, int total, int grid) {
    return (int)(((long long)(t + 1) * grid - 1) / total);
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
// Where a cluster's range starts: global tile range [lo, hi), the request b0 that holds lo and the number
// of tiles before b0.  Units of one request share its tile count, so prefix sums over requests suffice.
struct Plan {
    int total, lo, hi, req_start0;   // total < 2^24 (checked on the host)
    int grid, b0;                    // clusters in use; first request of the range
};

__device__ void make_plan(const AttnArgs& a, int UQ, int cid, int ncl, Plan* out, long long* s_warp) {
    long long sum = 0;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) sum += tiles_of(a, b);
    long long reqs;
    block_scan(sum, s_warp, &reqs);
    const int total = (int)(reqs * UQ);
    const int grid = ncl < total ? ncl : total;
    const int lo = cid < grid ? (int)((long long)cid * total / grid) : 0;
    const int hi = cid < grid ? (int)((long long)(cid + 1) * total / grid) : 0;
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
        const long long v = b < a.B ? (long long)tiles_of(a, b) * UQ : 0;
        long long chunk;
        const long long s0 = carry + block_scan(v, s_warp, &chunk);
        if (b < a.B && v > 0 && lo < hi && s0 <= lo && lo < s0 + v) {
            out->b0 = b;
            out->req_start0 = (int)s0;
        }
        carry += chunk;
    }
    __syncthreads();
}

// The segments of one cluster's range, in order; every role of both CTAs walks the same sequence.
struct Seg {
    int unit, b, hk, qg, t0, t1;   // tiles [t0, t1) of the unit
    bool split;                    // the unit crosses a range boundary
    int slot;                      // partial-result slot of this CTA (split segments only)
    int s0, s1;                    // global tiles of the whole unit
};

struct SegIter {
    int lo, hi, t, req_start;
    int b, lu, tiles, UQ, QG, cta;
    const AttnArgs* a;
    __device__ void init(const AttnArgs& args, const Plan& p, int uq, int qg) {
        a = &args;
        UQ = uq;
        QG = qg;
        cta = blockIdx.x;
        lo = p.lo;
        hi = p.hi;
        t = lo;
        b = p.b0;
        req_start = p.req_start0;
        tiles = b < args.B ? tiles_of(args, b) : 0;
        lu = tiles > 0 ? (lo - req_start) / tiles : 0;
    }
    __device__ bool next(Seg& s) {
        while (t < hi && b < a->B) {
            if (lu >= UQ || tiles == 0) {   // next request
                req_start += UQ * tiles;
                ++b;
                lu = 0;
                tiles = b < a->B ? tiles_of(*a, b) : 0;
                continue;
            }
            const int s0 = req_start + lu * tiles, s1 = s0 + tiles;
            const int e = s1 < hi ? s1 : hi;
            s.unit = b * UQ + lu;
            s.b = b;
            s.hk = lu / QG;
            s.qg = lu - s.hk * QG;
            s.t0 = t - s0;
            s.t1 = e - s0;
            s.split = !(s0 >= lo && s1 <= hi);
            s.slot = (lo >= s0 && lo < s1) ? 2 * cta : 2 * cta + 1;
            s.s0 = s0;
            s.s1 = s1;
            t = e;
            ++lu;
            return true;
        }
        return false;
    }
};

// ------------------------------------------------------------------------------------------------ main kernel
struct MainShared {
    uint64_t full[kKSlots + kVSlots], empty[kKSlots + kVSlots];
    uint64_t full8[kStage8], empty8[kStage8];              // e4m3 staging (FP8 KV only)
    uint64_t s_full[2], s_free[2], p_full[kPBufs], pv_done[kPBufs];   // per S / P buffer
    uint64_t q_full[2], o_full, drain[2];                  // per Q buffer
    uint64_t q_empty[2];                                   // per Q buffer: its segment's S MMAs are done
    uint64_t o_free;                                       // the segment's O has been read by the softmax
    float xch[2][4][kRows];                                // [tile parity][column part][row]: partial row max
    float lx[4][kRows];                                    // [column part][row]: partial row sum
    Plan plan;
    long long scan[33];
    int32_t par[SV_MAX_T];                                 // parent array of the current request
    uint32_t tmem;
    int err;
};

// KV8: the caches hold e4m3.  The producer then loads e4m3 tiles into a staging ring, warp 3 converts them
// exactly to f16 (every e4m3 value is an f16 value) into the MMA ring, and the MMAs run on f16 operands
// (Q and P rounded to f16); k_scale is folded into the softmax scale and v_scale into the epilogue.
template <int CL, bool KV8>
__global__ void __launch_bounds__(threads_of<KV8>(), 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, AttnArgs a, float scale_log2, int q_tma) {
    constexpr int kStages = KV8 ? kRing16 : kKSlots + kVSlots;
    constexpr int QB = KV8 ? 1 : 2;                  // Q buffers: segment s uses buffer s % QB
    constexpr int kSmemRing = ring_off<KV8>();
    constexpr int SPL = KV8 ? 2 : kSplit16;          // softmax warps per query row
    constexpr int COLS = kTileN / SPL;               // S columns (and O columns in the epilogue) per softmax warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ MainShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sQ = smem_u32(smem + kSmemQ), sRing = smem_u32(smem + kSmemRing);
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G;
    constexpr int kUnitRows = CL * kRows;
    const int QG = (TG + kUnitRows - 1) / kUnitRows, UQ = a.Hkv * QG;
    const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
    const int cid = blockIdx.x / CL, ncl = gridDim.x / CL;
    constexpr uint16_t kMask = (uint16_t)((1u << CL) - 1u);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], KV8 ? kConv : 1);   // the TMA transaction, or one arrival per converter
            mbar_init(&sh.empty[i], CL);             // one release per CTA of the cluster
        }
        for (int i = 0; i < kStage8; ++i) {
            mbar_init(&sh.full8[i], 1);
            mbar_init(&sh.empty8[i], kConv);
        }
        for (int bf = 0; bf < 2; ++bf) {
            mbar_init(&sh.s_full[bf], 1);
            mbar_init(&sh.s_free[bf], 4 * SPL);      // one arrival per softmax warp
            mbar_init(&sh.p_full[bf], 4 * SPL);
            mbar_init(&sh.pv_done[bf], 1);
        }
        mbar_init(&sh.drain[0], 1);
        mbar_init(&sh.drain[1], 1);
        // Q of a segment: loaded by TMA (q_tma: one expect_tx arrival) or written by the eight softmax warps
        for (int qb = 0; qb < 2; ++qb) {
            mbar_init(&sh.q_full[qb], q_tma ? 1 : 4 * SPL);
            mbar_init(&sh.q_empty[qb], 1);
        }
        mbar_init(&sh.o_free, 4 * SPL);
        mbar_init(&sh.o_full, 1);
        sh.err = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc(&sh.tmem, 512);
    make_plan(a, UQ, cid, ncl, &sh.plan, sh.scan);   // ends with __syncthreads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (CL > 1) cluster_sync_all();   // the peer's barriers are initialised before any multicast reaches them
    // the merge kernel may be scheduled now: its CTAs take SMs as CTAs of this grid leave them and wait there
    // (griddepcontrol.wait) until this whole grid has completed
    pdl_launch_dependents();
    const uint32_t tmem = sh.tmem;
    const Plan& plan = sh.plan;
    volatile int* err = &sh.err;
    const bool active = cid < plan.grid;

    if (warp == 0 || (!KV8 && warp == 3)) {
        // ---------------------------------------------------------------- TMA producers
        // bf16: warp 0 loads the K tiles, warp 3 the V tiles; e4m3: warp 0 loads both into the staging ring
        if (lane == 0 && active) {
            const int kv = warp == 0 ? 0 : 1;
            uint32_t n = 0, use = 0, nq = 0;
            SegIter si;
            si.init(a, plan, UQ, QG);
            Seg sg;
            while (!*err && si.next(sg)) {
                const int row0 = (sg.b * a.Hkv + sg.hk) * a.kv_cap;
                if (!KV8 && q_tma && kv == 0) {
                    // Q of the segment's M tile (128 query rows = 128/G nodes x G heads) once the previous
                    // segment's S MMAs no longer read the buffer
                    const uint32_t qb = nq % QB;
                    if (nq >= (uint32_t)QB && !mbar_wait(&sh.q_empty[qb], (nq / QB - 1) & 1, err)) break;
                    mbar_arrive_expect_tx(&sh.q_full[qb], 2 * kBoxBytes);
                    const int t0 = (sg.qg * kUnitRows + rank * kRows) / G;
                    uint8_t* qdst = smem + kSmemQ + qb * kSlotBytes;
                    tma_load_3d(qdst, &tmQ, 0, sg.hk * G, sg.b * T + t0, &sh.q_full[qb]);
                    tma_load_3d(qdst + kBoxBytes, &tmQ, 64, sg.hk * G, sg.b * T + t0, &sh.q_full[qb]);
                    ++nq;
                }
                for (int t = sg.t0; t < sg.t1 && !*err; ++t, ++n) {
                    if constexpr (KV8) {
                        // e4m3 K and V tiles into the staging ring (one 16 KB box each)
                        for (int x = 0; x < 2; ++x, ++use) {
                            const uint32_t slot = use % kStage8, round = use / kStage8;
                            if (!mbar_wait(&sh.empty8[slot], (round & 1) ^ 1, err)) break;
                            mbar_arrive_expect_tx(&sh.full8[slot], kSlot8Bytes);
                            tma_load_2d(smem + kSmemStage + slot * kSlot8Bytes, x ? (const void*)&tmV : (const void*)&tmK,
                                        0, row0 + t * kTileN, &sh.full8[slot]);
                        }
                    } else {
                        uint32_t slot, round;
                        ring_pos<KV8>(n, kv, slot, round);
                        // the slot is free in every CTA of the cluster
                        if (!mbar_wait(&sh.empty[slot], (round & 1) ^ 1, err)) break;
                        mbar_arrive_expect_tx(&sh.full[slot], kSlotBytes);
                        if (CL == 1 || kv == rank) {   // in a cluster CTA 0 loads K and CTA 1 loads V, for both
                            uint8_t* dst = smem + kSmemRing + slot * kSlotBytes;
                            const void* tm = kv ? (const void*)&tmV : (const void*)&tmK;
                            if (CL > 1) {
                                tma_load_2d_mc(dst, tm, 0, row0 + t * kTileN, &sh.full[slot], kMask);
                                tma_load_2d_mc(dst + kBoxBytes, tm, 64, row0 + t * kTileN, &sh.full[slot], kMask);
                            } else {
                                tma_load_2d(dst, tm, 0, row0 + t * kTileN, &sh.full[slot]);
                                tma_load_2d(dst + kBoxBytes, tm, 64, row0 + t * kTileN, &sh.full[slot]);
                            }
                        }
                    }
                }
            }
            // wait (bounded) until every CTA of the cluster has released the last slots, so no copy or
            // remote release is still in flight towards this CTA when it exits
            volatile int local = 0;
            if constexpr (KV8) {
                for (uint32_t u = use > kStage8 ? use - kStage8 : 0; u < use && !local; ++u)
                    mbar_wait(&sh.empty8[u % kStage8], (u / kStage8) & 1, &local);
            } else {
                const uint32_t nslots = kv ? kVSlots : kKSlots;
                for (uint32_t m = n > nslots ? n - nslots : 0; m < n && !local; ++m) {
                    uint32_t slot, round;
                    ring_pos<KV8>(m, kv, slot, round);
                    mbar_wait(&sh.empty[slot], round & 1, &local);
                }
                if (nq > 0 && !local)   // the last Q copy has landed
                    mbar_wait(&sh.q_full[(nq - 1) % QB], ((nq - 1) / QB) & 1, &local);
            }
        }
    } else if (KV8 && (warp == 3 || warp >= 12)) {
        // ---------------------------------------------------------------- e4m3 -> f16 converters (FP8 KV)
        // converter ci (warp 3, 12, 13, 14: one per SM sub-partition) converts rows 32 ci .. 32 ci + 31
        if (KV8 && active) {
            const int ci = warp == 3 ? 0 : warp - 11;
            uint32_t use = 0;
            SegIter si;
            si.init(a, plan, UQ, QG);
            Seg sg;
            bool ok = true;
            while (ok && !*err && si.next(sg)) {
                for (int t = sg.t0; t < sg.t1 && ok; ++t) {
                    for (int kv = 0; kv < 2 && ok; ++kv, ++use) {
                        const uint32_t s8 = use % kStage8, s16 = use % kStages;
                        ok = __all_sync(0xffffffffu, mbar_wait(&sh.full8[s8], (use / kStage8) & 1, err));
                        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sh.empty[s16], ((use / kStages) & 1) ^ 1, err));
                        if (!ok) break;
                        const uint8_t* src = smem + kSmemStage + s8 * kSlot8Bytes;
                        uint8_t* dst = smem + kSmemRing + s16 * kSlotBytes;
                        // chunk j: row j / 8, e4m3 bytes 16 (j % 8) .. +15 -> f16 d 16 (j % 8) .. +15, which is
                        // box (j % 8) / 4, 16-byte chunks 2 (j % 4) and 2 (j % 4) + 1 of that row
#pragma unroll 4
                        for (int j = ci * 256 + lane; j < (ci + 1) * 256; j += 32) {
                            const int r = j >> 3, c = j & 7;
                            const uint4 w = *(const uint4*)(src + r * 128 + c * 16);
                            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                            uint32_t hf[8];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                hf[2 * q] = e4m3x2_to_f16x2((uint16_t)(wv[q] & 0xffffu));
                                hf[2 * q + 1] = e4m3x2_to_f16x2((uint16_t)(wv[q] >> 16));
                            }
                            uint8_t* box = dst + (c >> 2) * kBoxBytes;
                            *(uint4*)(box + sw128_offset(r, 2 * (c & 3))) = make_uint4(hf[0], hf[1], hf[2], hf[3]);
                            *(uint4*)(box + sw128_offset(r, 2 * (c & 3) + 1)) = make_uint4(hf[4], hf[5], hf[6], hf[7]);
                        }
                        fence_proxy_async_smem();   // the MMAs (async proxy) read what this warp wrote
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&sh.full[s16]);
                            mbar_arrive(&sh.empty8[s8]);
                        }
                    }
                }
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------------------------------------------------------- MMA issuers: S (warp 1), PV (warp 2)
        const bool is_s = warp == 1;
        if (lane == 0 && active) {
            // S: Q and K from shared memory; PV: P from TMEM, V from shared memory; f16 operands for FP8 KV
            const uint32_t idS = KV8 ? idesc_f16_f32(128, kTileN, false, false) : idesc_bf16_f32(128, kTileN, false, false);
            const uint32_t idO = KV8 ? idesc_f16_f32(128, kD, false, true) : idesc_bf16_f32(128, kD, false, true);
            const uint64_t dK = sdesc_sw128(0, 16, 1024);          // K-major operands (Q, K)
            const uint64_t dV = sdesc_sw128(0, kBoxBytes, 1024);   // MN-major V: next 64 d one box further
            auto at = [](uint64_t base, uint32_t saddr) { return base | (uint64_t)((saddr & 0x3FFFFu) >> 4); };
            auto release = [&](uint32_t slot) {
                if (CL > 1) mma_commit_mc(&sh.empty[slot], kMask);
                else mma_commit(&sh.empty[slot]);
            };
            uint32_t gi = 0, nseg = 0;
            bool ok = true;
            SegIter si;
            si.init(a, plan, UQ, QG);
            Seg sg;
            while (ok && !*err && si.next(sg)) {
                const int nt = sg.t1 - sg.t0;
                // S: Q of this segment is in shared memory; PV: the previous segment's O has been read
                const uint32_t qb = nseg % QB;
                if (is_s ? !mbar_wait(&sh.q_full[qb], (nseg / QB) & 1, err)
                         : (nseg > 0 && !mbar_wait(&sh.o_free, (nseg - 1) & 1, err)))
                    break;
                tc_fence_after();
                for (int i = 0; i < nt && ok; ++i, ++gi) {
                    const uint32_t b = gi % kPBufs, k = gi / kPBufs;
                    if (is_s) {
                        uint32_t slot, round;
                        ring_pos<KV8>(gi, 0, slot, round);
                        ok = mbar_wait(&sh.full[slot], round & 1, err);
                        // S buffer b was last read by the softmax two tiles ago
                        if (ok && gi >= 2) ok = mbar_wait(&sh.s_free[b], (k - 1) & 1, err);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t kb = sRing + slot * kSlotBytes;
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk)
                            mma_f16_ss(tmem + col_S(b), at(dK, sQ + qb * kSlotBytes + (kk >> 2) * kBoxBytes + (kk & 3) * 32),
                                       at(dK, kb + (kk >> 2) * kBoxBytes + (kk & 3) * 32), idS, kk > 0);
                        mma_commit(&sh.s_full[b]);
                        release(slot);
                    } else {
                        uint32_t slot, round;
                        ring_pos<KV8>(gi, 1, slot, round);
                        ok = mbar_wait(&sh.full[slot], round & 1, err);
                        if (ok) ok = mbar_wait(&sh.p_full[b], k & 1, err);
                        if (!ok) break;
                        tc_fence_after();
                        const uint32_t vb = sRing + slot * kSlotBytes;
#pragma unroll
                        for (int kk = 0; kk < kTileN / 16; ++kk)
                            mma_f16_ts(tmem + col_O(), tmem + col_P(b) + kk * 8, at(dV, vb + kk * 2048), idO,
                                       (i > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&sh.pv_done[b]);
                        release(slot);
                    }
                }
                if (!ok) break;
                if (is_s) mma_commit(&sh.q_empty[qb]);   // after the segment's last S MMA
                else mma_commit(&sh.o_full);
                ++nseg;
            }
            // every MMA this thread issued has completed before TMEM is released
            mma_commit(&sh.drain[warp - 1]);
            volatile int local = 0;
            mbar_wait(&sh.drain[warp - 1], 0, &local);
        }
        __syncwarp();
    } else if (warp >= 4 && active) {
        // ---------------------------------------------------------------- softmax warps
        // Warp 4 + 4h + i owns TMEM lane quadrant q = warp % 4 (query rows 32q .. 32q+31) and columns
        // [64h, 64h + 64) of every S tile.  The two warps that share a quadrant (h = 0, 1) agree on the row
        // max through shared memory once per tile, and split the d columns of the epilogue.
        const int h = (warp - 4) >> 2;           // column part
        const int quad = warp & 3;               // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;        // query row inside the M tile (= TMEM lane)
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        uint32_t gi = 0, nseg = 0;
        // A warp that hits a time-out stops waiting and touching TMEM but keeps walking the segments, the
        // tiles and every barrier, so no partner is ever left waiting on it.
        bool dead = false;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(bar, parity, err));
            return !dead;
        };
        auto grp_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(128 * SPL) : "memory"); };
        auto pair_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(2 + quad), "n"(32 * SPL) : "memory"); };
        // Epilogue of a finished segment, run after the next segment's first tile (or after the last segment):
        // the softmax works on that tile while the segment's last PV completes.  O is normalised (bf16, this
        // warp's COLS d columns) into the output row or the partial slot, then released to the PV issuer.
        struct Pending {
            float m, l, sc, osc;
            size_t out_row;
            uint8_t* part;
            uint32_t nseg;
            bool valid, on;
        } pend;
        pend.on = false;
        auto epilogue = [&]() {
            if (wait(&sh.o_full, pend.nseg & 1)) tc_fence_after();
            sh.lx[h][row] = pend.l;                   // the row's sum is split between the row's warps
            pair_sync();
            float l_tot = 0.f;
#pragma unroll
            for (int j = 0; j < SPL; ++j) l_tot += sh.lx[j][row];
            if (!dead) {
                const float m_log2 = pend.m * pend.sc;
                const float inv_l = l_tot > 0.f ? pend.osc / l_tot : 0.f;
                uint16_t* dst_row = (pend.part ? (uint16_t*)pend.part + (size_t)row * kD : (uint16_t*)a.out + pend.out_row * kD) + COLS * h;
#pragma unroll
                for (int c = 0; c < COLS / 32; ++c) {
                    uint32_t o[32];
                    __syncwarp();
                    tmem_ld32(tmem + lane_addr + col_O() + COLS * h + 32 * c, o);
                    tmem_ld_wait();
                    if (pend.valid) {
                        uint4* dst = (uint4*)(dst_row + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            uint32_t v[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[8 * e + 2 * q]) * inv_l,
                                                                                __uint_as_float(o[8 * e + 2 * q + 1]) * inv_l);
                                v[q] = *reinterpret_cast<const uint32_t*>(&b2);
                            }
                            dst[e] = make_uint4(v[0], v[1], v[2], v[3]);
                        }
                    }
                }
                if (pend.valid && h == 0) {
                    if (pend.part) {
                        float* ml = (float*)(pend.part + (size_t)kRows * kD * 2);
                        ml[row] = m_log2;
                        ml[kRows + row] = l_tot;
                    } else if (a.lse) {
                        a.lse[pend.out_row] = (m_log2 + __log2f(l_tot)) * 0.69314718055994531f;
                    }
                }
                // O has been read: the PV issuer may start the next segment
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.o_free);
            pend.on = false;
        };

        SegIter si;
        si.init(a, plan, UQ, QG);
        Seg sg;
        bool first_seg = true;
        while (si.next(sg)) {
            const int b = sg.b, hk = sg.hk;
            const int nt = sg.t1 - sg.t0;
            const int L = __ldg(a.kv_len + b);
            // softmax scale in log2 units (times k_scale for e4m3 K); output scale (v_scale for e4m3 V)
            const float sc = KV8 ? scale_log2 * __ldg(a.k_scale + hk) : scale_log2;
            const float osc = KV8 ? __ldg(a.v_scale + hk) : 1.f;
            const int row0 = sg.qg * kUnitRows + rank * kRows;     // first query row of this M tile
            const int qi = row0 + row;
            const bool valid_row = qi < TG;
            const int t_node = valid_row ? qi / G : 0, g_head = valid_row ? qi - (qi / G) * G : 0;
            const size_t out_row = ((size_t)b * T + t_node) * a.Hq + (size_t)hk * G + g_head;
            uint8_t* part = sg.split ? (uint8_t*)a.ws + slots_off() + (long long)sg.slot * slot_bytes() : nullptr;
            dead = __any_sync(0xffffffffu, dead || *err);
            // Q by TMA (the producer), or else first, so that S of the segment's first tile is computed while the
            // ancestors are walked: this warp's half (64 of 128 d) of the Q row -> shared memory, box h of the
            // K-major 128-byte-swizzled A operand of the S MMA (bf16, or rounded to f16 when the caches are
            // e4m3), once the previous segment's S MMAs have completed (its epilogue comes later).
            const uint32_t qb = nseg % QB;
            if (!q_tma && nseg >= (uint32_t)QB) wait(&sh.q_empty[qb], (nseg / QB - 1) & 1);
            if (!dead && !q_tma) {
                const uint4* src = (const uint4*)((const uint16_t*)a.q + out_row * kD) + (COLS / 8) * h;
#pragma unroll
                for (int c = 0; c < COLS / 8; ++c) {
                    uint4 v = valid_row ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                    if constexpr (KV8) {
                        v.x = pack2<true>(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
                        v.y = pack2<true>(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
                        v.z = pack2<true>(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u));
                        v.w = pack2<true>(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
                    }
                    const int d8 = h * (COLS / 8) + c;   // 16-byte chunk of the row: box d8 / 8, chunk d8 % 8
                    *(uint4*)(smem + kSmemQ + qb * kSlotBytes + (d8 >> 3) * kBoxBytes + sw128_offset(row, d8 & 7)) = v;
                }
                fence_proxy_async_smem();   // the MMAs (async proxy) read what this thread wrote
            }
            __syncwarp();
            if (lane == 0 && !q_tma) mbar_arrive(&sh.q_full[qb]);

            // ancestors of this row's node from the request's parent array (walk bounded by T, so a malformed
            // array cannot trap; such requests are zeroed and flagged by the merge kernel)
            grp_sync();
            int bad = 0;   // this node's parent breaks the tree's topological order
            if (h == 0 && row < T) {
                const int px = __ldg(a.parent + (size_t)b * T + row);
                sh.par[row] = px;
                bad = row == 0 ? px != -1 : (px < 0 || px >= row);
            }
            // the barrier also ORs the flags: bad != 0 everywhere if any node's parent is out of order
            asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\t"
                         "selp.s32 %0, 1, 0, q;\n\t}"
                         : "=r"(bad) : "r"(bad), "n"(128 * SPL) : "memory");
            if (h == 0 && row == 0 && first_seg) {
                // the unit that began in an earlier cluster range and ends in this one is merged by
                // attn_merge_kernel
                SplitRec r;
                r.unit = (sg.s0 < plan.lo && sg.s1 <= plan.hi && !bad) ? sg.unit : -1;
                r.b = b;
                r.hk = hk;
                r.row0 = row0;
                r.rows = max(0, min(kRows, TG - row0));
                const int ccf = owner_of(sg.s0, plan.total, plan.grid);
                r.cf = ccf * CL + rank;
                r.cf_slot = ((int)((long long)ccf * plan.total / plan.grid) == sg.s0) ? 2 * r.cf : 2 * r.cf + 1;
                r.err = 0;
                ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x] = r;
            }
            first_seg = false;
            uint64_t anc = 0;
            if (valid_row) {
                int x = t_node;
                for (int step = 0; step < T && x >= 0 && x < T; ++step) {
                    anc |= 1ull << x;
                    const int px = sh.par[x];
                    if (px >= x) break;
                    x = px;
                }
            }

            float m_run = -INFINITY, l_run = 0.f;    // running max (raw score units); sum over this half
            for (int i = 0; i < nt; ++i, ++gi) {
                const uint32_t bb = gi % kPBufs, k = gi / kPBufs;
                const int tile0 = (sg.t0 + i) * kTileN;
                const int pos0 = tile0 + COLS * h;   // position of this warp's first column
                // this warp's 64 scores of the row, 32 at a time straight from TMEM into the registers the
                // arithmetic uses (a warp that has timed out still reads, harmlessly, and its results are discarded)
                const bool have = wait(&sh.s_full[bb], k & 1);
                // bit c of allow: column c of this warp's 64 is a prefix position or an ancestor of the row's node
                // (anc has no bit >= T); padding rows allow nothing
                uint64_t allow = ~0ull;
                if (!valid_row) {
                    allow = 0ull;
                } else if (pos0 + COLS > L) {   // columns reach the tree block: ancestor mask
                    const int np = L - pos0, a0 = pos0 - L;
                    const uint64_t pre = np >= 64 ? ~0ull : np <= 0 ? 0ull : (1ull << np) - 1ull;
                    const uint64_t tree = a0 >= 64 ? 0ull : a0 >= 0 ? (anc >> a0) : a0 > -64 ? (anc << -a0) : 0ull;
                    allow = pre | tree;
                }
                // P buffer bb was last read by the PV kPBufs tiles ago
                if (gi >= kPBufs) wait(&sh.pv_done[bb], (k - 1) & 1);
                tc_fence_after();
                __syncwarp();
                // P = 2^(s*scale - m) in bf16, packed in pairs (even position in the low half), into P buffer bb.
                // Fast path (every tile after a row's first): the exponentials use the running max m_run straight
                // away; only if some row's max grew by more than 2^8 do the two warps of the row take the slow path
                // and rewrite the tile's P against the new max, reading the scores again (S is freed only then).
                // (a row with no finite score has m = -inf and every s = -inf: moff = 0 gives p = 2^-inf = 0;
                // the arguments and the sums run two positions at a time, in packed f32x2 arithmetic)
                uint64_t ps2[4];
                float tmax_h = -INFINITY;
                auto chunk = [&](int ch, float m, bool do_exp) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_addr + col_S(bb) + COLS * h + 32 * ch, r);
                    tmem_ld_wait();
                    const uint32_t al = (uint32_t)(allow >> (32 * ch));
                    float s[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) s[c] = ((al >> c) & 1u) ? __uint_as_float(r[c]) : -INFINITY;
                    float mx[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        mx[c] = max3(max3(s[c], s[c + 4], s[c + 8]), max3(s[c + 12], s[c + 16], s[c + 20]),
                                     fmaxf(s[c + 24], s[c + 28]));
                    tmax_h = max3(tmax_h, max3(mx[0], mx[1], mx[2]), mx[3]);
                    if (!do_exp) return;
                    const float moff = m != -INFINITY ? -m * sc : 0.f;
                    const uint64_t sc2 = f2pack(sc, sc), mo2 = f2pack(moff, moff);
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        float x0, x1;
                        f2unpack(f2fma(f2pack(s[2 * c], s[2 * c + 1]), sc2, mo2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        ps2[c & 3] = f2add(ps2[c & 3], f2pack(p0, p1));
                        pk[c] = pack2<KV8>(p0, p1);
                    }
                    __syncwarp();
                    if (!dead) tmem_st16(tmem + lane_addr + col_P(bb) + (COLS / 2) * h + 16 * ch, pk);
                };
                float alpha = 1.f, m_use = m_run;
                bool slow = !__all_sync(0xffffffffu, m_run != -INFINITY || !valid_row);
                ps2[0] = ps2[1] = ps2[2] = ps2[3] = 0ull;
#pragma unroll 1
                for (int ch = 0; ch < COLS / 32; ++ch) chunk(ch, m_run, !slow);
                sh.xch[gi & 1][h][row] = tmax_h;   // double-buffered by tile parity: one barrier per tile
                pair_sync();
                float tmax = tmax_h;
#pragma unroll
                for (int j = 0; j < SPL; ++j) tmax = fmaxf(tmax, sh.xch[gi & 1][j][row]);
                if (!slow) slow = __any_sync(0xffffffffu, valid_row && (tmax - m_run) * sc > kRescaleThreshold);
                if (slow) {
                    const float m_new = fmaxf(m_run, tmax);
                    const bool rescale = m_run != -INFINITY && (m_new - m_run) * sc > kRescaleThreshold;
                    m_use = (m_run == -INFINITY || rescale) ? m_new : m_run;
                    alpha = rescale ? ex2((m_run - m_use) * sc) : 1.f;
                    // O holds PV of the previous tile: wait for it, then rescale this warp's half of O
                    if (__any_sync(0xffffffffu, rescale) && wait(&sh.pv_done[(gi - 1) % kPBufs], ((gi - 1) / kPBufs) & 1)) {
                        tc_fence_after();
                        for (int c = 0; c < COLS / 16; ++c) {   // 16 columns at a time
                            uint32_t o[16];
                            __syncwarp();
                            tmem_ld16(tmem + lane_addr + col_O() + COLS * h + 16 * c, o);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st16(tmem + lane_addr + col_O() + COLS * h + 16 * c, o);
                        }
                        tmem_st_wait();
                    }
                    tmem_st_wait();   // the fast path's P stores land before they are overwritten
                    ps2[0] = ps2[1] = ps2[2] = ps2[3] = 0ull;
#pragma unroll 1
                    for (int ch = 0; ch < COLS / 32; ++ch) chunk(ch, m_use, true);
                }
                if (have) {   // the scores have been read for the last time: S may take the tile after next
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.s_free[bb]);
                }
                float ps[4], ps2_hi[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) f2unpack(ps2[j], ps[j], ps2_hi[j]);
                const float psum = ((ps[0] + ps2_hi[0]) + (ps[1] + ps2_hi[1])) + ((ps[2] + ps2_hi[2]) + (ps[3] + ps2_hi[3]));
                l_run = (m_run == -INFINITY) ? psum : l_run * alpha + psum;
                m_run = m_use;
                // the last tile may hold cache rows past the tree block: zero those V rows in this CTA's copy
                // of the tile (NaN-safe), fenced before the PV by every writer
                if (!dead && tile0 + kTileN > L + T) {
                    uint32_t vslot, vround;
                    ring_pos<KV8>(gi, 1, vslot, vround);
                    if (wait(&sh.full[vslot], vround & 1)) {
                        const int r_lo = max(0, L + T - tile0);
                        uint8_t* vdst = smem + kSmemRing + vslot * kSlotBytes;
                        for (int idx = (warp - 4) * 32 + lane; idx < (kTileN - r_lo) * 16; idx += 128 * SPL) {
                            const int r = r_lo + (idx >> 4), c = idx & 15;
                            *(uint4*)(vdst + (c >> 3) * kBoxBytes + sw128_offset(r, c & 7)) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                }
                if (!dead) {
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.p_full[bb]);
                }
                if (pend.on) epilogue();   // the previous segment's
            }
            // the segment's epilogue waits until the next segment's first tile is done (or the last segment ends)
            pend.m = m_run;
            pend.l = l_run;
            pend.sc = sc;
            pend.osc = osc;
            pend.out_row = out_row;
            pend.part = part;
            pend.nseg = nseg++;
            pend.valid = valid_row;
            pend.on = true;
        }
        if (pend.on) epilogue();
    }
    if (!active && tid == 0) {   // CTAs beyond the used grid complete no split unit
        SplitRec r = {};
        r.unit = -1;
        ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x] = r;
    }
    tc_fence_before();
    __syncthreads();
    if (CL > 1) cluster_sync_all();   // no CTA leaves while its peer may still multicast to it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // this CTA's time-out flag (a bounded wait gave up: every status becomes TIMEOUT), written on every launch,
    // after the record itself
    if (tid == 0) ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x].err = sh.err;
}

// ------------------------------------------------------------------------------------------------ merge kernel
// Runs after attn_tc_kernel (programmatic dependent launch): validates every request (statuses, zero
// outputs for failed ones) and merges the segments of every unit that crossed a cluster range boundary.
// One merge unit = (record of CTA c, 16 rows): each warp merges two rows, lanes covering 4 of the 128 dims
// (coalesced 8-byte loads), with every load of a row issued before any of them is used.
constexpr int kMergeRows = 16;
constexpr int kMergeUnits = kRows / kMergeRows;   // per record

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(AttnArgs a, int grid_main, int CL) {
    __shared__ int s_bad;
    const int T = a.T, G = a.Hq / a.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait_prior();   // attention results are visible from here on
    const SplitRec* recs = (const SplitRec*)((const uint8_t*)a.ws + rec_off());
    // the time-out flags matter only to the CTAs that write statuses: after a time-out every status says so
    // and the merged outputs (garbage then) are never read
    bool timeout = false;
    if (blockIdx.x < a.B) {
        if (tid == 0) s_bad = 0;
        __syncthreads();
        for (int c = tid; c < grid_main; c += blockDim.x)
            if (__ldcg(&recs[c].err)) s_bad = 1;
        __syncthreads();
        timeout = s_bad != 0;
        __syncthreads();
    }

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
    // 2. merges
    const uint8_t* slots = (const uint8_t*)a.ws + slots_off();
    for (int u = blockIdx.x; u < grid_main * kMergeUnits; u += gridDim.x) {
        const int cl = u / kMergeUnits, rb = u - cl * kMergeUnits;
        const SplitRec rec = recs[cl];
        if (rec.unit < 0 || rec.rows <= 0) continue;
        float m[2][4], l[2][4];
        uint2 x[2][4];
        int rr[2];
        // contributors are CTAs cf, cf + CL, ..., cl; CTA c > cf holds the unit in its first slot 2c
        for (int h = 0; h < 2; ++h) rr[h] = rb * kMergeRows + warp * 2 + h;
        float M[2] = {-INFINITY, -INFINITY}, Ls[2] = {0.f, 0.f}, acc[2][4] = {};
        for (int c0 = rec.cf; c0 <= cl; c0 += 4 * CL) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = min(c0 + i * CL, cl);
                    const int sidx = c == rec.cf ? rec.cf_slot : 2 * c;
                    const uint8_t* base = slots + (long long)sidx * slot_bytes();
                    const int r = min(rr[h], rec.rows - 1);
                    const float* ml = (const float*)(base + (size_t)kRows * kD * 2);
                    m[h][i] = c0 + i * CL <= cl ? __ldcg(ml + r) : -INFINITY;
                    l[h][i] = __ldcg(ml + kRows + r);
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
            if (r >= rec.rows) continue;
            const int qi = rec.row0 + r, t_node = qi / G, g_head = qi - t_node * G;
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

// bf16 caches: boxes of 64 columns x 128 rows, 128-byte swizzle (the MMA layout).  e4m3 caches: whole
// 128-byte rows x 128 rows, unswizzled (the converter's input).
bool encode_kv_map(CUtensorMap* m, const void* base, long long rows, bool e4m3) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)kD * (e4m3 ? 1 : 2)};
    cuuint32_t box[2] = {e4m3 ? (cuuint32_t)kD : 64u, kTileN};
    cuuint32_t es[2] = {1, 1};
    return enc(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               e4m3 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q as a 3D tensor [B*T][Hq][D] (bf16): a box of 64 d x G heads x 128/G nodes is one 64-column half of an
// M tile's 128 query rows, landing in shared memory in the row order of the tile (node-major, then head).
bool encode_q_map(CUtensorMap* m, const AttnArgs& a) {
    auto enc = tensor_map_encoder();
    const int G = a.Hq / a.Hkv;
    if (!enc || G < 1 || kRows % G != 0 || ((uintptr_t)a.q & 15) != 0) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.Hq, (cuuint64_t)a.B * a.T};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)a.Hq * kD * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)(kRows / G)};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of CL CTAs that fit on the device at once with this kernel's resources (cached per CL); the
// persistent grid never exceeds it, so every cluster of the grid is resident from the start.
template <int CL, bool KV8>
int resident_clusters() {
    static int n = 0;
    if (!n) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL * 64);
        cfg.blockDim = dim3(threads_of<KV8>());
        cfg.dynamicSmemBytes = kSmemAlloc;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = CL;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, attn_tc_kernel<CL, KV8>, &cfg) != cudaSuccess || c < 1) c = num_sms() / CL;
        n = c;
    }
    return n;
}

template <int CL, bool KV8>
cudaError_t launch_main(const AttnArgs& a, cudaStream_t s, float scale_log2, int* grid_out) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<CL, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tmK, tmV, tmQ;
    const long long rows = (long long)a.B * a.Hkv * a.kv_cap;
    if (!encode_kv_map(&tmK, a.k, rows, KV8) || !encode_kv_map(&tmV, a.v, rows, KV8)) return cudaErrorInvalidValue;
    // bf16 caches: Q by TMA when the heads of a kv group tile the 128-row M tile; else the softmax writes it
    const int q_tma = (!KV8 && encode_q_map(&tmQ, a)) ? 1 : 0;
    if (!q_tma) tmQ = tmK;
    int ncl = resident_clusters<CL, KV8>();
    if (ncl * CL > kMaxGrid) ncl = kMaxGrid / CL;
    *grid_out = ncl * CL;
    return launch_ex(attn_tc_kernel<CL, KV8>, dim3(ncl * CL), dim3(threads_of<KV8>()), (size_t)kSmemAlloc, s, CL, false, tmK,
                     tmV, tmQ, a, scale_log2, q_tma);
}

}  // namespace

size_t attn_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap) {
    (void)B; (void)T; (void)kv_cap;
    if (D != kD || Hkv < 1 || Hq % Hkv) return 0;
    return (size_t)workspace_bytes();
}

// Units of two M tiles (2-CTA clusters sharing multicast tiles) for bf16 caches with more than 128 query
// rows per kv head; units of one M tile otherwise (e4m3 caches: every CTA converts its own tiles).
int cluster_size(const AttnArgs& a) {
    return (a.kv_dt == SV_BF16 && (long long)a.T * (a.Hq / a.Hkv) > kRows) ? 2 : 1;
}

bool attn_tc_supported(const AttnArgs& a) {
    const long long TG = (long long)a.T * (a.Hq / a.Hkv);
    const long long unit_rows = (long long)cluster_size(a) * kRows;
    return a.q_dt == SV_BF16 && (a.kv_dt == SV_BF16 || a.kv_dt == SV_E4M3) && a.D == kD && a.B >= 1 &&
           (long long)a.B * a.Hkv * a.kv_cap < (1LL << 31) - kTileN && TG < 65536 &&
           // tile indices of the whole call fit the kernel's 32-bit bookkeeping
           (long long)a.B * a.Hkv * ((TG + unit_rows - 1) / unit_rows) * ((a.kv_cap + kTileN - 1) / kTileN) < (1LL << 24) &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    const int CL = cluster_size(a);
    const float sl2 = scale * 1.4426950408889634f;
    int grid = 0;
    if (a.kv_dt == SV_E4M3) e = launch_main<1, true>(a, s, sl2, &grid);
    else e = CL == 2 ? launch_main<2, false>(a, s, sl2, &grid) : launch_main<1, false>(a, s, sl2, &grid);
    if (e != cudaSuccess) return e;
    return launch_ex(attn_merge_kernel, dim3(grid * kMergeUnits), dim3(kMergeThreads), 0, s, 1, true, a, grid, CL);
}

}  // namespace sv
