// attn_tc.cu -- tree-masked GQA attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Every draft-tree node attends to the request's KV prefix plus its own ancestors ("Aurora" post,
// section 2: a custom mask that follows the speculative tree's causal structure lets all branches of
// the tree be verified in one batched pass).  For one (request b, kv head hk) the T nodes x G query
// heads form T*G query rows that share every K/V tile, so the contraction is a real GEMM:
//   S = Q K^T  (M = 128 query rows, N = 128 kv positions, K = D = 128)   A = Q, B = K, both in shared memory
//   O += P V   (M = 128 query rows, N = D = 128, K = 128 kv positions)   A = P from TMEM, B = V
//
// A CTA works on two 128-row M tiles at once, "side A" and "side B", so that the tensor core runs the MMAs
// of one side while the softmax warps of the other side work:
//   * pair mode (a unit of 129..256 query rows): A holds rows 0..127 and B rows 128..255 of the unit; both
//     sides see every K/V tile, which is loaded (and, for 8-bit and 4-bit caches, converted) once for both;
//   * split mode (a unit of at most 128 query rows): A and B hold the same rows; A takes the even tiles and
//     B the odd tiles of the unit's KV range, and the two partial results are merged in the epilogue.
// A "unit" is (request, kv head, group of 256 query rows); it owns ceil((L_b + T) / 128) KV tiles.
//
// Scheduling (balanced, stream-K style): the tiles of all units form one sequence and CTA c of the
// persistent grid takes the contiguous range [c * total / G, (c + 1) * total / G); every CTA derives its range
// from kv_len alone in a short prologue.  A unit that crosses a range boundary is processed in segments; each
// segment leaves a partial result (normalised O in bf16, max m and sum l per row) and a second kernel,
// attn_merge_kernel, merges them, validates every request and writes the status array.
//
// Roles (bf16 caches: 12 warps; e4m3 / e2m1 caches: 16 warps):
//   warp 0       K producer: the segment's Q (TMA 3D boxes) and the K tiles into a 2-slot K ring
//   warp 1       MMA issuer (also owns the 512 TMEM columns): S_A, S_B, O_A += P_A V, O_B += P_B V in the
//                order that lets one side's MMAs overlap the other side's softmax
//   warp 2       (bf16 caches) V cleaner: passes every V tile to the MMAs, zeroing the cache rows past the tree
//                block in a unit's last tile
//   warp 3       V producer: the V tiles into a 2-slot V ring
//   warps 4-7    softmax of side A, warps 8-11 softmax of side B: one thread per query row (TMEM lane), all
//                128 scores of the row in registers; the row max needs no exchange between threads
//   warps 12-15  (8-bit / 4-bit caches) converters: the raw tile lands in the upper part of its ring slot and
//                is rewritten in place as f16 (every e4m3 value, and every e2m1 value times its e4m3 block
//                scale, is exactly an f16 value); Q is rounded to f16 in place the same way
// TMEM: O_A (columns 0..127), O_B (128..255), S_A (256..383), S_B (384..511); P of a side (bf16 or f16 pairs,
// 64 columns) is written over the side's S columns once they have been read.  The MMAs of one thread execute
// in issue order, so S_X of the next tile (issued after the PV that reads P_X) never overwrites P_X early.
// Every mbarrier wait is bounded; a time-out raises a flag that turns the statuses into SV_ERR_TIMEOUT, and
// the CTA winds down, waiting (bounded) for its own copies and MMAs before it frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "sv_internal.cuh"
#include "tc_ptx.cuh"

namespace sv {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kTileN = 128;                      // kv positions per tile
constexpr int kRows = 128;                       // query rows per M tile
constexpr int kUnitRows = 2 * kRows;             // query rows per unit (two M tiles)
constexpr int kSlotBytes = kTileN * kD * 2;      // 32 KB: one f16/bf16 K or V tile
constexpr int kBoxBytes = kSlotBytes / 2;        // one 64-column box: 128 rows x 128 bytes
enum { KV_BF16 = 0, KV_E4M3 = 1, KV_E2M1 = 2 };
template <int KVK>
constexpr int threads_of() { return KVK == KV_BF16 ? 384 : 512; }
constexpr int kMaxGrid = 160;                    // the workspace is sized for grids up to this size
constexpr float kRescaleThreshold = 8.0f;        // log2 units
constexpr int kMergeThreads = 256;               // 8 warps

// Dynamic shared memory (1024-byte aligned): Q [side][2 boxes][16 KB], the K ring [2][32 KB], the V ring [2][32 KB].
// Raw 8-bit tiles land in box 1 of their slot (bytes 16 KB..32 KB), raw 4-bit codes at 24 KB..32 KB with their
// block scales at 23 KB..24 KB; the converters rewrite the slot as two f16 boxes.
constexpr int kSmemQ = 0;
constexpr int kSmemV = 4 * kSlotBytes;
// KS K slots: 2 (Q holds two M tiles), or 3 when every unit of the launch is in split mode (one M tile of Q, and
// the second tile's 32 KB holds a third K slot, so K is prefetched two tiles ahead)
template <int KS>
__host__ __device__ constexpr int smem_k() { return KS == 3 ? kSlotBytes : 2 * kSlotBytes; }
// ring positions: the n-th K tile in slot n % KS (barrier index = slot), the n-th V tile in slot n % 2 (barrier
// index 3 + slot)
constexpr int kVBar = 3;
constexpr int kSmemBytes = 6 * kSlotBytes;       // 196608
constexpr int kSmemAlloc = kSmemBytes + 1024;    // + alignment slack
constexpr int kRaw8Off = kBoxBytes;              // e4m3 tile: [128 rows][128 B], 128-byte swizzle
constexpr int kRaw4Off = 24576;                  // e2m1 codes: [128 rows][64 B], 64-byte swizzle
constexpr int kRaw4ScaleOff = 23552;             // e4m3 block scales: [128 rows][8 B]
constexpr int kRaw4Bytes = 8192 + 1024;

__host__ __device__ constexpr uint32_t col_O(int side) { return 128u * (uint32_t)side; }
__host__ __device__ constexpr uint32_t col_S(int side) { return 256u + 128u * (uint32_t)side; }

// Workspace: a 256-byte header; per CTA a record of the split unit it completes (if any); two partial-result
// slots per CTA.  A slot holds O / l in bf16 [256 rows][128], then m (log2 units) [256] and l [256] in fp32.
struct SplitRec {
    int unit;            // -1: this CTA completes no split unit (or the request's tree is malformed)
    int b, hk;           // request and kv head of the unit
    int row0;            // first query row (index into the T*G rows of the kv head) of the unit
    int rows;            // valid rows of the unit
    int cf;              // first CTA holding a segment of the unit
    int cf_slot;         // that CTA's slot for the unit (2 cf, or 2 cf + 1 if it began in an earlier unit)
    int err;             // 1: a bounded wait of this CTA gave up (written last, on every launch)
};
__host__ __device__ constexpr long long slot_bytes() { return (long long)kUnitRows * kD * 2 + kUnitRows * 8; }
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
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)v16));
    return r;
}

// the four bytes of w, each two e2m1 codes (low nibble -> low half), to four f16 pairs, exactly
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
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

// a bf16 pair to an f16 pair (round to nearest)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack2<true>(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
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

// tiles of one request: its prefix plus its tree block, in 128-position tiles (0 if kv_len is invalid)
__device__ __forceinline__ int tiles_of(const AttnArgs& a, int b) {
    const int L = __ldg(a.kv_len + b);
    return (L >= 0 && L + a.T <= a.kv_cap) ? (L + a.T + kTileN - 1) / kTileN : 0;
}

// CTA owning global tile t when `total` tiles are split into `grid` ranges [c*total/grid, (c+1)*total/grid)
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
// Where a CTA's range starts: global tile range [lo, hi), the request b0 that holds lo and the number of tiles
// before b0.  Units of one request share its tile count, so prefix sums over requests suffice.
struct Plan {
    int total, lo, hi, req_start0;   // total < 2^24 (checked on the host)
    int grid, b0;                    // CTAs in use; first request of the range
};

__device__ void make_plan(const AttnArgs& a, int UQ, int cid, int ncta, Plan* out, long long* s_warp) {
    long long sum = 0;
    for (int b = threadIdx.x; b < a.B; b += blockDim.x) sum += tiles_of(a, b);
    long long reqs;
    block_scan(sum, s_warp, &reqs);
    const int total = (int)(reqs * UQ);
    const int grid = ncta < total ? ncta : total;
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

// The segments of one CTA's range, in order; every role walks the same sequence.
struct Seg {
    int unit, b, hk, qg, t0, t1;   // tiles [t0, t1) of the unit
    bool split;                    // the unit crosses a range boundary
    bool pair;                     // the unit has more than 128 query rows (two M tiles)
    int slot;                      // partial-result slot of this CTA (split segments only)
    int s0, s1;                    // global tiles of the whole unit
    int rows;                      // valid query rows of the unit
};

struct SegIter {
    int lo, hi, t, req_start;
    int b, lu, tiles, UQ, QG, TG, cta;
    const AttnArgs* a;
    __device__ void init(const AttnArgs& args, const Plan& p, int uq, int qg, int tg) {
        a = &args;
        UQ = uq;
        QG = qg;
        TG = tg;
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
            s.rows = min(kUnitRows, TG - s.qg * kUnitRows);
            s.pair = s.rows > kRows;
            t = e;
            ++lu;
            return true;
        }
        return false;
    }
};

// tiles of side `side` in a segment of nt tiles, and the segment-relative index of its i-th tile
__device__ __forceinline__ int side_tiles(bool pair, int nt, int side) { return pair ? nt : (nt + 1 - side) / 2; }
__device__ __forceinline__ int side_tile(bool pair, int i, int side) { return pair ? i : 2 * i + side; }

// ------------------------------------------------------------------------------------------------ producers
// TMA row coordinates of the box(es) of one K or V tile: contiguous caches one box of 128 rows; paged caches
// 128 / box_rows boxes, each a run of box_rows rows of one page, found through the page table (pages past the
// request's last used position, or page ids outside the pool, read as an out-of-range box: fill values).
struct TileRows {
    const AttnArgs* a;
    int box_rows, oob;
    __device__ int y(int b, int hk, int L, int t, int box) const {
        const int pos = t * kTileN + box * box_rows;
        if (!a->page_table) return (b * a->Hkv + hk) * a->kv_cap + pos;
        if (pos >= L + a->T) return oob;
        const int page = __ldg(a->page_table + (size_t)b * a->max_pages + (pos >> a->page_shift));
        if (page < 0 || page >= a->num_pages) return oob;
        return (page * a->Hkv + hk) * (1 << a->page_shift) + (pos & ((1 << a->page_shift) - 1));
    }
};

// ------------------------------------------------------------------------------------------------ main kernel
// A softmax warp's segment walk and the segment whose epilogue is pending (written by lane 0, read by all lanes).
struct SoftmaxState {
    SegIter it;
    Seg seg, pend;
    uint32_t pend_nseg;
    int pend_on, has;
};

struct MainShared {
    uint64_t full[5], raw[5], empty[5];                    // K slots 0 .. KS-1 and V slots 3, 4
    uint64_t s_full[2], p_full[2], o_full[2];              // per side
    uint64_t o_free[2][2];                                 // [O_A / O_B][dims 0..63 / 64..127] read by the epilogue
    uint64_t q_full, q_ready, q_empty, drain[2];
    uint64_t conv_bar;                                     // e2m1 caches: the converters have read the raw tile
    float ml[2][2][kRows];                                 // split-mode epilogue: [side][m][row]
    float pm[2][kRows], pl[2][kRows];                      // pending epilogue: the row's max and sum, per side
    SoftmaxState sm[8];                                    // per softmax warp: segment walk and pending epilogue
    Plan plan;
    long long scan[33];
    int32_t par[SV_MAX_T];                                 // parent array of the current request
    uint32_t tmem;
    int err;
};

// KVK: bf16, e4m3 or e2m1 caches.  8-bit and 4-bit caches are converted exactly to f16 and the MMAs run on f16
// operands (Q rounded to f16); the per-kv-head scale of K is folded into the softmax scale and that of V into
// the epilogue.
template <int KVK, int KS>
__global__ void __launch_bounds__(threads_of<KVK>(), 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKs,
               const __grid_constant__ CUtensorMap tmVs, const __grid_constant__ AttnArgs a, float scale_log2, int q_tma,
               int box_rows) {
    constexpr bool CONV = KVK != KV_BF16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ MainShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kSmemK = smem_k<KS>();
    const uint32_t sQ = smem_u32(smem + kSmemQ), sK = smem_u32(smem + kSmemK), sV = smem_u32(smem + kSmemV);
    const int T = a.T, G = a.Hq / a.Hkv, TG = T * G;
    const int QG = (TG + kUnitRows - 1) / kUnitRows, UQ = a.Hkv * QG;
    const int nbox = kTileN / box_rows;

    if (tid == 0) {
        for (int i = 0; i < 5; ++i) {
            // K (bf16): the TMA transaction; V (bf16): the V cleaner; 8-bit / 4-bit: one arrival per converter warp
            mbar_init(&sh.full[i], CONV ? 4 : 1);
            mbar_init(&sh.raw[i], 1);                // the raw tile's TMA transaction
            mbar_init(&sh.empty[i], 1);              // the MMA warp's commit after the tile's last reader
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.s_full[s], 1);
            mbar_init(&sh.p_full[s], 4);             // the side's four softmax warps
            mbar_init(&sh.o_full[s], 1);
            mbar_init(&sh.drain[s], 1);
        }
        for (int x = 0; x < 4; ++x) mbar_init(&sh.o_free[x >> 1][x & 1], 4);   // the four warps that read it
        mbar_init(&sh.q_full, q_tma ? 1 : 8);        // the TMA transaction, or the eight softmax warps
        mbar_init(&sh.q_ready, 4);                   // the converters rounded Q to f16 (8-bit / 4-bit caches)
        mbar_init(&sh.q_empty, 1);
        mbar_init(&sh.conv_bar, 4);
        sh.err = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmQ);
    }
    if (warp == 1) tmem_alloc(&sh.tmem, 512);
    make_plan(a, UQ, blockIdx.x, gridDim.x, &sh.plan, sh.scan);   // ends with __syncthreads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the merge kernel may be scheduled now: its CTAs take SMs as CTAs of this grid leave them and wait there
    // (griddepcontrol.wait) until this whole grid has completed
    pdl_launch_dependents();
    const uint32_t tmem = sh.tmem;
    const Plan& plan = sh.plan;
    volatile int* err = &sh.err;
    const bool active = (int)blockIdx.x < plan.grid;
    const uint32_t qbar_ready = CONV && q_tma;       // the MMAs wait for the converters' Q, else for Q itself

    if (warp == 0 || warp == 3) {
        // ---------------------------------------------------------------- TMA producers (K + Q: warp 0, V: warp 3)
        if (lane == 0 && active) {
            const int kv = warp == 0 ? 0 : 1;
            const CUtensorMap* tm = kv ? &tmV : &tmK;
            const CUtensorMap* tms = kv ? &tmVs : &tmKs;
            TileRows tr{&a, box_rows, a.page_table ? a.num_pages * a.Hkv * (1 << a.page_shift) : 0};
            uint32_t n = 0, nseg = 0;
            SegIter si;
            si.init(a, plan, UQ, QG, TG);
            Seg sg;
            while (!*err && si.next(sg)) {
                const int L = __ldg(a.kv_len + sg.b);
                if (kv == 0 && q_tma) {
                    // Q of the segment's M tile(s) (128 query rows = 128/G nodes x G heads each) once the previous
                    // segment's S MMAs no longer read it
                    if (nseg > 0 && !mbar_wait(&sh.q_empty, (nseg - 1) & 1, err, a.wait_cycles)) break;
                    const int mt = sg.pair ? 2 : 1;
                    mbar_arrive_expect_tx(&sh.q_full, mt * 2 * kBoxBytes);
                    for (int m = 0; m < mt; ++m) {
                        const int t0 = (sg.qg * kUnitRows + m * kRows) / G;
                        uint8_t* qdst = smem + kSmemQ + m * kSlotBytes;
                        tma_load_3d(qdst, &tmQ, 0, sg.hk * G, sg.b * T + t0, &sh.q_full);
                        tma_load_3d(qdst + kBoxBytes, &tmQ, 64, sg.hk * G, sg.b * T + t0, &sh.q_full);
                    }
                }
                ++nseg;
                for (int t = sg.t0; t < sg.t1 && !*err; ++t, ++n) {
                    const uint32_t slot = kv ? n & 1 : n % KS, round = kv ? n >> 1 : n / KS;
                    const uint32_t gslot = kv ? kVBar + slot : slot;
                    if (!mbar_wait(&sh.empty[gslot], (round & 1) ^ 1, err, a.wait_cycles)) break;
                    uint8_t* dst = smem + (kv ? kSmemV : kSmemK) + slot * kSlotBytes;
                    if constexpr (KVK == KV_BF16) {
                        // K tiles go straight to the MMAs; V tiles pass the V cleaner first
                        uint64_t* bar = kv ? &sh.raw[gslot] : &sh.full[gslot];
                        mbar_arrive_expect_tx(bar, kSlotBytes);
                        for (int bx = 0; bx < nbox; ++bx) {
                            const int y = tr.y(sg.b, sg.hk, L, t, bx);
                            tma_load_2d(dst + bx * box_rows * 128, tm, 0, y, bar);
                            tma_load_2d(dst + kBoxBytes + bx * box_rows * 128, tm, 64, y, bar);
                        }
                    } else if constexpr (KVK == KV_E4M3) {
                        mbar_arrive_expect_tx(&sh.raw[gslot], kBoxBytes);
                        for (int bx = 0; bx < nbox; ++bx)
                            tma_load_2d(dst + kRaw8Off + bx * box_rows * 128, tm, 0, tr.y(sg.b, sg.hk, L, t, bx),
                                        &sh.raw[gslot]);
                    } else {
                        // e2m1 codes (64-byte rows) and their block scales (two cache rows per 16-byte TMA row)
                        const int y = tr.y(sg.b, sg.hk, L, t, 0);
                        mbar_arrive_expect_tx(&sh.raw[gslot], kRaw4Bytes);
                        tma_load_2d(dst + kRaw4Off, tm, 0, y, &sh.raw[gslot]);
                        tma_load_2d(dst + kRaw4ScaleOff, tms, 0, y >> 1, &sh.raw[gslot]);
                    }
                }
            }
            // wait until the copies this thread issued have landed (their transaction barriers complete whatever the
            // consumers do), so no copy is still in flight towards this CTA when it exits; these waits keep the full
            // limit even when the work waits were given a short one
            volatile int local = 0;
            const uint32_t ns = kv ? 2u : (uint32_t)KS;
            for (uint32_t m = n > ns ? n - ns : 0; m < n && !local; ++m) {
                const uint32_t sl = kv ? m & 1 : m % KS, rd = kv ? m >> 1 : m / KS;
                const bool tx_on_raw = CONV || kv;   // 8-bit / 4-bit tiles and bf16 V tiles land on raw, bf16 K on full
                mbar_wait(tx_on_raw ? &sh.raw[kv ? kVBar + sl : sl] : &sh.full[sl], rd & 1, &local);
            }
            if (kv == 0 && q_tma && nseg > 0 && !local) mbar_wait(&sh.q_full, (nseg - 1) & 1, &local);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && active) {
            const uint32_t idS = CONV ? idesc_f16_f32(128, kTileN, false, false) : idesc_bf16_f32(128, kTileN, false, false);
            const uint32_t idO = CONV ? idesc_f16_f32(128, kD, false, true) : idesc_bf16_f32(128, kD, false, true);
            const uint64_t dK = sdesc_sw128(0, 16, 1024);          // K-major operands (Q, K)
            const uint64_t dV = sdesc_sw128(0, kBoxBytes, 1024);   // MN-major V: next 64 d one box further
            auto at = [](uint64_t base, uint32_t saddr) { return base | (uint64_t)((saddr & 0x3FFFFu) >> 4); };
            uint32_t g[2] = {0, 0};      // tiles each side has processed (s_full / p_full phases)
            uint32_t base = 0, nseg = 0;  // ring index of the segment's first tile; segments so far
            bool ok = true;
            SegIter si;
            si.init(a, plan, UQ, QG, TG);
            Seg sg;
            // S MMAs of the segment still to issue.  When every unit is in split mode (the 3-slot K ring), a segment
            // releases its Q tile after the last of them; otherwise Q is released with the segment's O (the next Q
            // then loads in the switch's bubble, not under the last tile's MMAs, which measured faster).
            int s_left = 0;
            // S_X = Q_X K(tile)^T; commit to s_full_X (and release the K slot when `release`)
            // (split mode: both sides multiply Q tile A)
            auto issue_s = [&](int side, uint32_t ridx, bool release, bool pair) -> bool {
                const uint32_t slot = ridx % KS;
                if (!mbar_wait(&sh.full[slot], (ridx / KS) & 1, err, a.wait_cycles)) return false;
                tc_fence_after();
                const uint32_t kb = sK + slot * kSlotBytes, qb = sQ + (pair ? (uint32_t)side : 0u) * kSlotBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk)
                    mma_f16_ss(tmem + col_S(side), at(dK, qb + (kk >> 2) * kBoxBytes + (kk & 3) * 32),
                               at(dK, kb + (kk >> 2) * kBoxBytes + (kk & 3) * 32), idS, kk > 0);
                mma_commit(&sh.s_full[side]);
                if (release) mma_commit(&sh.empty[slot]);
                if constexpr (KS == 3)
                    if (--s_left == 0) mma_commit(&sh.q_empty);   // Q may be overwritten once these complete
                return true;
            };
            // O_X += P_X V(tile) (P in the side's S columns); release the V slot when `release`.  The first PV of a
            // segment after the first (`o_wait`) overwrites O_X once the previous segment's epilogue has read both
            // halves of it.
            auto issue_pv = [&](int side, uint32_t ridx, bool first, bool release, bool o_wait) -> bool {
                const uint32_t slot = ridx & 1;
                if (!mbar_wait(&sh.full[kVBar + slot], (ridx >> 1) & 1, err, a.wait_cycles)) return false;
                if (!mbar_wait(&sh.p_full[side], g[side] & 1, err, a.wait_cycles)) return false;
                tc_fence_after();
                const uint32_t vb = sV + slot * kSlotBytes;
                if (!o_wait) {
#pragma unroll
                    for (int kk = 0; kk < kTileN / 16; ++kk)
                        mma_f16_ts(tmem + col_O(side), tmem + col_S(side) + kk * 8, at(dV, vb + kk * 2048), idO,
                                   (!first || kk > 0) ? 1u : 0u);
                } else {
                    for (int h = 0; h < 2; ++h)
                        if (!mbar_wait(&sh.o_free[side][h], (nseg - 1) & 1, err, a.wait_cycles)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kTileN / 16; ++kk)
                        mma_f16_ts(tmem + col_O(side), tmem + col_S(side) + kk * 8, at(dV, vb + kk * 2048), idO,
                                   (!first || kk > 0) ? 1u : 0u);
                }
                if (release) mma_commit(&sh.empty[kVBar + slot]);
                ++g[side];
                return true;
            };
            while (ok && !*err && si.next(sg)) {
                const int nt = sg.t1 - sg.t0;
                const int n0 = side_tiles(sg.pair, nt, 0), n1 = side_tiles(sg.pair, nt, 1);
                s_left = n0 + n1;
                ok = mbar_wait(qbar_ready ? &sh.q_ready : &sh.q_full, nseg & 1, err, a.wait_cycles);
                if (!ok) break;
                tc_fence_after();
                const bool rel0 = !sg.pair;                // pair mode: side B is a tile's last reader
                if (n0 > 0) ok = issue_s(0, base + side_tile(sg.pair, 0, 0), rel0, sg.pair);
                if (ok && n1 > 0) ok = issue_s(1, base + side_tile(sg.pair, 0, 1), true, sg.pair);
                const int nmax = n0 > n1 ? n0 : n1;
                for (int i = 0; i < nmax && ok; ++i) {
                    for (int side = 0; side < 2 && ok; ++side) {
                        const int ns = side ? n1 : n0;
                        if (i >= ns) continue;
                        const bool rel = side == 1 || !sg.pair;
                        ok = issue_pv(side, base + side_tile(sg.pair, i, side), i == 0, rel, i == 0 && nseg > 0);
                        if (ok && i + 1 < ns) ok = issue_s(side, base + side_tile(sg.pair, i + 1, side), rel, sg.pair);
                    }
                }
                if (!ok) break;
                mma_commit(&sh.o_full[0]);
                mma_commit(&sh.o_full[1]);
                if constexpr (KS != 3) mma_commit(&sh.q_empty);
                base += (uint32_t)nt;
                ++nseg;
            }
            // every MMA this thread issued has completed before TMEM is released
            mma_commit(&sh.drain[0]);
            volatile int local = 0;
            mbar_wait(&sh.drain[0], 0, &local);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------------------------------------------------------- V cleaner (bf16 caches)
        // every V tile passes here in ring order (so this warp never runs a barrier phase ahead of the ring): a
        // unit's last tile may hold cache rows past the tree block (junk, NaN possibly), which become zeros before
        // any PV reads the tile, so that P = 0 there contributes exactly nothing (the 8-bit and 4-bit converters
        // write those rows as zeros themselves)
        if (!CONV && active) {
            uint32_t n = 0;
            bool ok = true;
            SegIter si;
            si.init(a, plan, UQ, QG, TG);
            Seg sg;
            while (ok && !*err && si.next(sg)) {
                const int L = __ldg(a.kv_len + sg.b);
                for (int t = sg.t0; t < sg.t1 && ok; ++t, ++n) {
                    const uint32_t slot = n & 1;
                    ok = __all_sync(0xffffffffu, mbar_wait(&sh.raw[kVBar + slot], (n >> 1) & 1, err, a.wait_cycles));
                    if (!ok) break;
                    const int r_lo = L + T - t * kTileN;
                    if (r_lo < kTileN) {
                        uint8_t* vdst = smem + kSmemV + slot * kSlotBytes;
                        for (int idx = lane; idx < (kTileN - r_lo) * 16; idx += 32) {
                            const int rr = r_lo + (idx >> 4), c = idx & 15;
                            *(uint4*)(vdst + (c >> 3) * kBoxBytes + sw128_offset(rr, c & 7)) = make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.full[kVBar + slot]);
                }
            }
        }
    } else if (warp >= 12) {
        // ---------------------------------------------------------------- converters (8-bit / 4-bit caches)
        // converter ci (one per SM sub-partition) rewrites rows 32 ci .. 32 ci + 31 of every K and V tile, and a
        // quarter of Q, in place as f16
        if (CONV && active) {
            const int ci = warp - 12, r = 32 * ci + lane;
            uint32_t n = 0, nseg = 0, nconv = 0;
            SegIter si;
            si.init(a, plan, UQ, QG, TG);
            Seg sg;
            bool ok = true;
            while (ok && !*err && si.next(sg)) {
                const int L = __ldg(a.kv_len + sg.b);
                if (q_tma) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&sh.q_full, nseg & 1, err, a.wait_cycles));
                    if (!ok) break;
                    const int nq = (sg.pair ? 2 : 1) * kSlotBytes / 16;   // 16-byte chunks of Q
                    for (int c = ci * 32 + lane; c < nq; c += 128) {
                        uint4 v = *(const uint4*)(smem + kSmemQ + c * 16);
                        v.x = bf16x2_to_f16x2(v.x);
                        v.y = bf16x2_to_f16x2(v.y);
                        v.z = bf16x2_to_f16x2(v.z);
                        v.w = bf16x2_to_f16x2(v.w);
                        *(uint4*)(smem + kSmemQ + c * 16) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.q_ready);
                }
                ++nseg;
                for (int t = sg.t0; t < sg.t1 && ok; ++t, ++n) {
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        const uint32_t sl = kv ? n & 1 : n % KS, round = kv ? n >> 1 : n / KS;
                        const uint32_t gslot = kv ? kVBar + sl : sl;
                        ok = __all_sync(0xffffffffu, mbar_wait(&sh.raw[gslot], round & 1, err, a.wait_cycles));
                        if (!ok) break;
                        uint8_t* slot = smem + (kv ? kSmemV : kSmemK) + sl * kSlotBytes;
                        // V rows past the tree block hold junk (NaN possibly): they become zeros, so that P = 0 there
                        // contributes exactly nothing
                        const bool zero = kv == 1 && t * kTileN + r >= L + T;
                        if constexpr (KVK == KV_E4M3) {
                            // the raw row r (128 bytes, 128-byte swizzle) is read whole before the f16 row is written:
                            // box 1 of the f16 row occupies the raw row's bytes
                            uint4 w[8];
#pragma unroll
                            for (int c = 0; c < 8; ++c) w[c] = *(const uint4*)(slot + kRaw8Off + sw128_offset(r, c));
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const uint32_t wv[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
                                uint32_t hf[8];
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    hf[2 * q] = zero ? 0u : e4m3x2_to_f16x2(wv[q] & 0xffffu);
                                    hf[2 * q + 1] = zero ? 0u : e4m3x2_to_f16x2(wv[q] >> 16);
                                }
                                // e4m3 bytes 16c..16c+15 = d 16c..16c+15 -> box c/4, f16 chunks 2(c%4), 2(c%4)+1
                                uint8_t* box = slot + (c >> 2) * kBoxBytes;
                                *(uint4*)(box + sw128_offset(r, 2 * (c & 3))) = make_uint4(hf[0], hf[1], hf[2], hf[3]);
                                *(uint4*)(box + sw128_offset(r, 2 * (c & 3) + 1)) = make_uint4(hf[4], hf[5], hf[6], hf[7]);
                            }
                        } else {
                            // 64 code bytes (64-byte swizzle) and 8 block-scale bytes of row r, read by every converter
                            // before any f16 row is written (the f16 rows overwrite other rows' codes)
                            uint4 w[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                w[c] = *(const uint4*)(slot + kRaw4Off + r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
                            const uint2 sc = *(const uint2*)(slot + kRaw4ScaleOff + r * 8);
                            // rendezvous of the four converters (a bounded wait on an mbarrier, not a named barrier,
                            // so a converter that gave up cannot leave the others waiting forever)
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&sh.conv_bar);
                            ok = __all_sync(0xffffffffu, mbar_wait(&sh.conv_bar, nconv & 1, err, a.wait_cycles));
                            ++nconv;
                            if (!ok) break;
                            uint32_t s16[8];   // block scales as f16, each broadcast to a pair
                            {
                                const uint32_t p01 = e4m3x2_to_f16x2(sc.x & 0xffffu), p23 = e4m3x2_to_f16x2(sc.x >> 16);
                                const uint32_t p45 = e4m3x2_to_f16x2(sc.y & 0xffffu), p67 = e4m3x2_to_f16x2(sc.y >> 16);
                                const uint32_t pp[4] = {p01, p23, p45, p67};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    s16[2 * j] = (pp[j] & 0xffffu) * 0x10001u;
                                    s16[2 * j + 1] = (pp[j] >> 16) * 0x10001u;
                                }
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j) {   // f16 chunk j: d 8j..8j+7 = code bytes 4j..4j+3, block j/2
                                const uint4& wc = w[j >> 2];
                                const uint32_t word = (j & 3) == 0 ? wc.x : (j & 3) == 1 ? wc.y : (j & 3) == 2 ? wc.z : wc.w;
                                uint32_t h[4];
                                e2m1x8_to_f16x8(word, h);
#pragma unroll
                                for (int q = 0; q < 4; ++q) h[q] = zero ? 0u : hmul2_bits(h[q], s16[j >> 1]);
                                *(uint4*)(slot + (j >> 3) * kBoxBytes + sw128_offset(r, j & 7)) = make_uint4(h[0], h[1], h[2], h[3]);
                            }
                        }
                        fence_proxy_async_smem();   // the MMAs (async proxy) read what this warp wrote
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sh.full[gslot]);
                    }
                }
            }
        }
    } else if (warp >= 4 && active) {
        // ---------------------------------------------------------------- softmax warps
        // Warp 4 + 4 side + q owns TMEM lane quadrant q (query rows 32q .. 32q+31 of the side's M tile).  The
        // segment walk and the pending epilogue live in shared memory (sh.sm[warp - 4]), so the tile loop keeps
        // its registers for the scores.
        const int side = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;        // query row inside the M tile (= TMEM lane)
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const uint32_t tS = tmem + lane_addr + col_S(side), tO = tmem + lane_addr + col_O(side);
        SoftmaxState& ss = sh.sm[warp - 4];
        if (lane == 0) {
            ss.it.init(a, plan, UQ, QG, TG);
            ss.pend_on = 0;
        }
        __syncwarp();
        uint32_t g = 0, nseg = 0, base = 0;
        // A warp that hits a time-out stops waiting and touching TMEM but keeps walking the segments, the
        // tiles and every barrier, so no partner is ever left waiting on it.
        bool dead = false;
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (!dead) dead = __any_sync(0xffffffffu, !mbar_wait(bar, parity, err, a.wait_cycles));
            return !dead;
        };
        auto all_sync = [&]() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
        // Epilogue of a finished segment, run after the side's first tile of the next segment (or at once when the
        // side has no tile there): the softmax works on that tile while the segment's last PV completes.  O is
        // normalised (bf16) into the output rows or the partial slot, then released.
        auto epilogue = [&]() {
            const Seg& pg = ss.pend;
            const bool pr = pg.pair;
            const int urow = pr ? side * kRows + row : row;      // row inside the unit
            const int qi = pg.qg * kUnitRows + urow;
            const bool valid = urow < pg.rows;
            const int t_node = valid ? qi / G : 0, g_head = valid ? qi - t_node * G : 0;
            const size_t out_row = ((size_t)pg.b * T + t_node) * a.Hq + (size_t)pg.hk * G + g_head;
            const float sc = CONV ? scale_log2 * __ldg(a.k_scale + pg.hk) : scale_log2;
            const float osc = CONV ? __ldg(a.v_scale + pg.hk) : 1.f;
            const float pm = sh.pm[side][row], pl = sh.pl[side][row];
            const float m_log2 = pm == -INFINITY ? -INFINITY : pm * sc;
            float M = m_log2, Lsum = pl, wa = 1.f, wb = 0.f;
            if (!pr) {
                // split mode: both sides hold the same rows (A the even tiles, B the odd ones)
                sh.ml[side][0][row] = m_log2;
                all_sync();
                const float m0 = sh.ml[0][0][row], l0 = sh.pl[0][row], m1 = sh.ml[1][0][row], l1 = sh.pl[1][row];
                M = fmaxf(m0, m1);
                wa = (M == -INFINITY || l0 == 0.f) ? 0.f : ex2(m0 - M);
                wb = (M == -INFINITY || l1 == 0.f) ? 0.f : ex2(m1 - M);
                Lsum = l0 * wa + l1 * wb;
                all_sync();   // sh.ml / sh.pl may be rewritten only after both sides read them
            }
            if (wait(&sh.o_full[0], ss.pend_nseg & 1) && wait(&sh.o_full[1], ss.pend_nseg & 1)) tc_fence_after();
            // O is read 16 columns at a time, normalised to bf16 pairs and stored; each 64-column half is released
            // (o_free) as soon as it has been read.
            // Pair mode: this side reads its own O, both halves; split mode: side A reads dims 0..63 of O_A and O_B,
            // side B dims 64..127.
            const float inv = Lsum > 0.f ? osc / Lsum : 0.f;
            uint8_t* part = pg.split ? (uint8_t*)a.ws + slots_off() + (long long)pg.slot * slot_bytes() : nullptr;
            uint16_t* dst_row = part ? (uint16_t*)part + (size_t)urow * kD : (uint16_t*)a.out + out_row * kD;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if (!pr && h != side) continue;
                if (!dead) {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {   // 16 columns at a time
                        uint32_t oa[16], ob[16];
                        __syncwarp();
                        tmem_ld16(tmem + lane_addr + col_O(pr ? side : 0) + 64 * h + 16 * c, oa);
                        if (!pr) tmem_ld16(tmem + lane_addr + col_O(1) + 64 * h + 16 * c, ob);
                        tmem_ld_wait();
                        reg_fence(oa);
                        if (!pr) reg_fence(ob);
                        uint32_t pk[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            // a side that saw no finite score (weight 0) contributes exactly nothing
                            float x0 = wa > 0.f ? __uint_as_float(oa[2 * q]) * wa : 0.f;
                            float x1 = wa > 0.f ? __uint_as_float(oa[2 * q + 1]) * wa : 0.f;
                            if (!pr && wb > 0.f) {
                                x0 += __uint_as_float(ob[2 * q]) * wb;
                                x1 += __uint_as_float(ob[2 * q + 1]) * wb;
                            }
                            pk[q] = pack2<false>(x0 * inv, x1 * inv);
                        }
                        if (valid) {
                            uint4* dst = (uint4*)(dst_row + 64 * h + 16 * c);
                            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh.o_free[pr ? side : 0][h]);
                        if (!pr) mbar_arrive(&sh.o_free[1][h]);
                    }
                } else {
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&sh.o_free[pr ? side : 0][h]);
                        if (!pr) mbar_arrive(&sh.o_free[1][h]);
                    }
                }
            }
            if (!dead && valid && (pr || side == 0)) {
                if (part) {
                    float* ml = (float*)(part + (size_t)kUnitRows * kD * 2);
                    ml[urow] = M;
                    ml[kUnitRows + urow] = Lsum;
                } else if (a.lse) {
                    a.lse[out_row] = (M + __log2f(Lsum)) * 0.69314718055994531f;
                }
            }
            __syncwarp();
            if (lane == 0) ss.pend_on = 0;
            __syncwarp();
        };

        bool first_seg = true;
        int par_b = -1;   // the request whose parent array sh.par holds
        for (;;) {
            if (lane == 0) ss.has = ss.it.next(ss.seg) ? 1 : 0;
            __syncwarp();
            if (!ss.has) break;
            const int b = ss.seg.b, hk = ss.seg.hk;
            const int nt = ss.seg.t1 - ss.seg.t0, t0 = ss.seg.t0;
            const bool pair = ss.seg.pair;
            const int L = __ldg(a.kv_len + b);
            // softmax scale in log2 units (times k_scale for 8-bit / 4-bit K)
            const float sc = CONV ? scale_log2 * __ldg(a.k_scale + hk) : scale_log2;
            const int urow = pair ? side * kRows + row : row;
            const int qi = ss.seg.qg * kUnitRows + urow;
            const bool valid_row = urow < ss.seg.rows;
            const int t_node = valid_row ? qi / G : 0;
            dead = __any_sync(0xffffffffu, dead || *err);
            // Q written by the softmax warps when it is not loaded by TMA (G does not divide 128): this thread's row
            // (f16 for 8-bit / 4-bit caches), into the side's Q tile (pair mode) or tile A (split mode, side A)
            if (!q_tma) {
                if (nseg > 0) wait(&sh.q_empty, (nseg - 1) & 1);
                if (!dead && (pair || side == 0)) {
                    const int gh = valid_row ? qi - t_node * G : 0;
                    const size_t qrow = ((size_t)b * T + t_node) * a.Hq + (size_t)hk * G + gh;
                    const uint4* src = (const uint4*)((const uint16_t*)a.q + qrow * kD);
#pragma unroll 4
                    for (int d8 = 0; d8 < 16; ++d8) {
                        uint4 v = valid_row ? __ldg(src + d8) : make_uint4(0, 0, 0, 0);
                        if constexpr (CONV) {
                            v.x = bf16x2_to_f16x2(v.x);
                            v.y = bf16x2_to_f16x2(v.y);
                            v.z = bf16x2_to_f16x2(v.z);
                            v.w = bf16x2_to_f16x2(v.w);
                        }
                        *(uint4*)(smem + kSmemQ + (pair ? side : 0) * kSlotBytes + (d8 >> 3) * kBoxBytes +
                                  sw128_offset(row, d8 & 7)) = v;
                    }
                    fence_proxy_async_smem();   // the MMAs (async proxy) read what this thread wrote
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.q_full);
            }

            // ancestors of this row's node from the request's parent array (walk bounded by T, so a malformed
            // array cannot trap; such requests are zeroed and flagged by the merge kernel); the array is loaded
            // when the segment's request differs from the previous segment's
            int bad = 0;   // this node's parent breaks the tree's topological order
            if (b != par_b) {
                all_sync();   // every warp has walked the previous request's array
                if (side == 0 && row < T) {
                    const int px = __ldg(a.parent + (size_t)b * T + row);
                    sh.par[row] = px;
                    bad = row == 0 ? px != -1 : (px < 0 || px >= row);
                }
                // the barrier also ORs the flags: bad != 0 everywhere if any node's parent is out of order
                asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\t"
                             "selp.s32 %0, 1, 0, q;\n\t}"
                             : "=r"(bad) : "r"(bad) : "memory");
                par_b = b;
            }
            if (side == 0 && row == 0 && first_seg) {
                // the unit that began in an earlier CTA's range and ends in this one is merged by attn_merge_kernel
                const Seg& sg = ss.seg;
                SplitRec rc;
                rc.unit = (sg.s0 < plan.lo && sg.s1 <= plan.hi && !bad) ? sg.unit : -1;
                rc.b = b;
                rc.hk = hk;
                rc.row0 = sg.qg * kUnitRows;
                rc.rows = sg.rows;
                const int ccf = owner_of(sg.s0, plan.total, plan.grid);
                rc.cf = ccf;
                rc.cf_slot = ((int)((long long)ccf * plan.total / plan.grid) == sg.s0) ? 2 * ccf : 2 * ccf + 1;
                rc.err = 0;
                ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x] = rc;
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

            const int my_tiles = side_tiles(pair, nt, side);
            float m_run = -INFINITY, l_run = 0.f;    // running max (raw score units) and sum of the row
            // the previous segment's epilogue runs after this segment's first tile (outside the tile loop)
            int i = 0;
            for (;;) {
            while (i < my_tiles) {
                const int tile0 = (t0 + side_tile(pair, i, side)) * kTileN;
                // the side's S tile is complete (and every earlier MMA of this CTA with it)
                wait(&sh.s_full[side], g & 1);
                tc_fence_after();
                __syncwarp();
                // bit e of the mask word of the 32 columns 32c..32c+31: a prefix position or an ancestor of the row's
                // node (anc has no bit >= T); padding rows allow nothing; only tiles that reach the tree block are masked
                const bool masked = tile0 + kTileN > L;
                auto allow_word = [&](int c) -> uint32_t {
                    const int pos0 = tile0 + 32 * c;
                    const int np = L - pos0, a0 = pos0 - L;
                    const uint32_t pre = np >= 32 ? ~0u : np <= 0 ? 0u : (1u << np) - 1u;
                    const uint32_t tree = a0 >= 64 ? 0u : a0 >= 0 ? (uint32_t)(anc >> a0) : a0 > -32 ? (uint32_t)(anc << -a0) : 0u;
                    return valid_row ? (pre | tree) : 0u;
                };
                // pass 1: the row's max over the tile, two 32-column TMEM loads in flight at a time (tiles inside the
                // prefix take the variant without the mask)
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                auto pass1 = [&](auto mask_tag) {
                    constexpr bool MASK = decltype(mask_tag)::value;
                    auto fold = [&](const uint32_t (&r)[32], int c) {
                        const uint32_t al = MASK ? allow_word(c) : ~0u;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int k = q + 4 * e;
                                v[e] = (!MASK || ((al >> k) & 1u)) ? __uint_as_float(r[k]) : -INFINITY;
                            }
                            mx[q] = max3(mx[q], max3(v[0], v[1], v[2]), max3(max3(v[3], v[4], v[5]), v[6], v[7]));
                        }
                    };
#pragma unroll 1
                    for (int c = 0; c < 4; c += 2) {
                        uint32_t r0[32], r1[32];
                        tmem_ld32(tS + 32 * c, r0);
                        tmem_ld32(tS + 32 * c + 32, r1);
                        tmem_ld_wait();
                        reg_fence(r0);
                        reg_fence(r1);
                        fold(r0, c);
                        fold(r1, c + 1);
                    }
                };
                if (masked) pass1(std::true_type{});
                else pass1(std::false_type{});
                const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                // lazy rescaling: the row keeps its running max unless the tile's max exceeds it by more than 2^8
                const float m_new = fmaxf(m_run, tmax);
                const bool grow = m_run != -INFINITY && (m_new - m_run) * sc > kRescaleThreshold;
                const float m_use = (m_run == -INFINITY || grow) ? m_new : m_run;
                const float alpha = grow ? ex2((m_run - m_use) * sc) : 1.f;
                if (__any_sync(0xffffffffu, grow) && !dead) {
                    // O holds the PVs of earlier tiles, all complete (they were issued before this tile's S)
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * c, o);
                        tmem_ld_wait();
                        reg_fence(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tO + 32 * c, o);
                    }
                    tmem_st_wait();
                }
                // pass 2: P = 2^(s*scale - m) in bf16 (f16 for 8-bit / 4-bit caches), packed in pairs (even position in
                // the low half); the P of columns 32c..32c+31 goes to columns 16c..16c+15 of the side's S, which have
                // been read by then (a row with no finite score has m = -inf and every s = -inf: moff = 0 gives
                // p = 2^-inf = 0); the arguments and the sums run two positions at a time, in packed f32x2 arithmetic
                const float moff = m_use != -INFINITY ? -m_use * sc : 0.f;
                const uint64_t sc2 = f2pack(sc, sc), mo2 = f2pack(moff, moff);
                uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};
                auto pass2 = [&](auto mask_tag) {
                    constexpr bool MASK = decltype(mask_tag)::value;
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t r[32];
                        tmem_ld32(tS + 32 * c, r);
                        tmem_ld_wait();
                        reg_fence(r);
                        const uint32_t al = MASK ? allow_word(c) : ~0u;
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float s0 = (!MASK || ((al >> (2 * e)) & 1u)) ? __uint_as_float(r[2 * e]) : -INFINITY;
                            const float s1 = (!MASK || ((al >> (2 * e + 1)) & 1u)) ? __uint_as_float(r[2 * e + 1]) : -INFINITY;
                            float x0, x1;
                            f2unpack(f2fma(f2pack(s0, s1), sc2, mo2), x0, x1);
                            const float p0 = ex2(x0), p1 = ex2(x1);
                            ps2[e & 3] = f2add(ps2[e & 3], f2pack(p0, p1));
                            pk[e] = pack2<CONV>(p0, p1);
                        }
                        if (!dead) tmem_st16(tS + 16 * c, pk);
                    }
                };
                if (masked) pass2(std::true_type{});
                else pass2(std::false_type{});
                float ps[4], ps_hi[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) f2unpack(ps2[q], ps[q], ps_hi[q]);
                const float psum = ((ps[0] + ps_hi[0]) + (ps[1] + ps_hi[1])) + ((ps[2] + ps_hi[2]) + (ps[3] + ps_hi[3]));
                l_run = (m_run == -INFINITY) ? psum : l_run * alpha + psum;
                m_run = m_use;
                if (!dead) {
                    tmem_st_wait();
                    tc_fence_before();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[side]);
                ++i;
                ++g;
                if (ss.pend_on) break;
            }
            if (!ss.pend_on) break;
            epilogue();                    // the previous segment's (at once if the side has no tile here)
            }
            // this segment's epilogue waits until the side's first tile of the next segment is done
            sh.pm[side][row] = m_run;
            sh.pl[side][row] = l_run;
            __syncwarp();
            if (lane == 0) {
                ss.pend = ss.seg;
                ss.pend_nseg = nseg;
                ss.pend_on = 1;
            }
            __syncwarp();
            ++nseg;
            base += (uint32_t)nt;
        }
        if (ss.pend_on) epilogue();
    }
    if (!active && tid == 0) {   // CTAs beyond the used grid complete no split unit
        SplitRec r = {};
        r.unit = -1;
        ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x] = r;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    // this CTA's time-out flag (a bounded wait gave up: every status becomes TIMEOUT), written on every launch,
    // after the record itself
    if (tid == 0) ((SplitRec*)((uint8_t*)a.ws + rec_off()))[blockIdx.x].err = sh.err;
}

// ------------------------------------------------------------------------------------------------ merge kernel
// Runs after attn_tc_kernel (programmatic dependent launch), on a grid that is resident at once.  Before the
// attention grid has completed, CTA x checks requests x, x + grid, ... (parent array, kv_len, page table: inputs
// only).  Afterwards every CTA reads all the records (one load round), lists the 32-row chunks of the split units
// in record order, and merges chunks x, x + grid, ...; CTAs x < B also write the statuses of their requests and
// zero the outputs of failed ones.  A merge thread takes 16 dims of one row (8 threads per row, two 16-byte loads
// per partial) and loads a batch of four contributors at once, so a unit spanning up to four CTAs costs one more
// round of loads.
constexpr int kMergeRows = kMergeThreads / 8;          // 32
constexpr int kMergeBatch = 4;

__device__ __forceinline__ int request_status(const AttnArgs& a, int b, int* s_flag) {
    const int T = a.T, tid = threadIdx.x;
    if (tid == 0) *s_flag = 0;
    __syncthreads();
    const int L = __ldg(a.kv_len + b);
    if (tid < T) {
        const int p = __ldg(a.parent + (size_t)b * T + tid);
        if (tid == 0 ? p != -1 : (p < 0 || p >= tid)) *s_flag = 1;
    }
    __syncthreads();
    int st = *s_flag ? SV_ERR_BAD_TREE : SV_OK;
    if (st == SV_OK && (L < 0 || L + T > a.kv_cap)) st = SV_ERR_INVALID_ARG;
    if (st == SV_OK && a.page_table) {   // every page the request reads must name a page of the pool
        const int32_t* pt = a.page_table + (size_t)b * a.max_pages;
        for (int i = tid; i <= (L + T - 1) >> a.page_shift; i += blockDim.x)
            if (__ldg(pt + i) < 0 || __ldg(pt + i) >= a.num_pages) *s_flag = 2;
        __syncthreads();
        if (*s_flag) st = SV_ERR_INVALID_ARG;
    }
    __syncthreads();
    return st;
}

__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const __grid_constant__ AttnArgs a, int grid_main) {
    __shared__ int s_flag, s_to;
    __shared__ SplitRec s_rec[kMaxGrid];
    __shared__ int s_pfx[kMaxGrid + 1];   // chunks of the records before record c
    __shared__ long long s_scan[33];
    const int T = a.T, G = a.Hq / a.Hkv;
    const int tid = threadIdx.x, x = blockIdx.x;
    constexpr int kReqs = 4;              // requests checked before the wait (any further ones after it)
    int st_pre[kReqs];
#pragma unroll
    for (int k = 0; k < kReqs; ++k) {
        const int b = x + k * (int)gridDim.x;
        st_pre[k] = b < a.B ? request_status(a, b, &s_flag) : SV_OK;
    }
    pdl_wait_prior();   // the attention grid has completed and its results are visible from here on

    // the records (L2: written by the attention grid), with the time-out flags
    const SplitRec* recs = (const SplitRec*)((const uint8_t*)a.ws + rec_off());
    if (tid == 0) s_to = 0;
    int chunks = 0;
    if (tid < grid_main) {
        const int4 r0 = __ldcg((const int4*)(recs + tid)), r1 = __ldcg((const int4*)(recs + tid) + 1);
        SplitRec r;
        r.unit = r0.x; r.b = r0.y; r.hk = r0.z; r.row0 = r0.w;
        r.rows = r1.x; r.cf = r1.y; r.cf_slot = r1.z; r.err = r1.w;
        s_rec[tid] = r;
        chunks = r.unit >= 0 ? (r.rows + kMergeRows - 1) / kMergeRows : 0;
    }
    __syncthreads();
    if (tid < grid_main && s_rec[tid].err) s_to = 1;
    long long total;
    const int pfx = (int)block_scan(chunks, s_scan, &total);   // ends with __syncthreads
    if (tid < grid_main) s_pfx[tid] = pfx;
    if (tid == 0) s_pfx[grid_main] = (int)total;
    __syncthreads();

    // statuses (after a time-out every status says so: the outputs are garbage then)
    for (int k = 0, b = x; b < a.B; ++k, b += gridDim.x) {
        int st = k < kReqs ? st_pre[k] : request_status(a, b, &s_flag);
        if (s_to) st = SV_ERR_TIMEOUT;
        if (tid == 0 && a.status) a.status[b] = st;
        if (st != SV_OK && st != SV_ERR_TIMEOUT) {
            const size_t n = (size_t)T * a.Hq;
            uint16_t* o = (uint16_t*)a.out + (size_t)b * n * kD;
            for (size_t i = tid; i < n * kD / 8; i += blockDim.x) ((uint4*)o)[i] = make_uint4(0, 0, 0, 0);
            if (a.lse) for (size_t i = tid; i < n; i += blockDim.x) a.lse[(size_t)b * n + i] = 0.f;
        }
    }

    // merges (a request that fails its checks keeps the zero outputs of its status CTA: the record of a malformed
    // tree names no unit, and a bad page table is checked here)
    const uint8_t* slots = (const uint8_t*)a.ws + slots_off();
    for (int task = x; task < (int)total; task += gridDim.x) {
        int lo = 0, hi = grid_main - 1;   // the record holding chunk `task`: the last c with s_pfx[c] <= task
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pfx[mid] <= task) lo = mid;
            else hi = mid - 1;
        }
        const int ci = lo;
        const SplitRec rec = s_rec[ci];
        const int chunk = task - s_pfx[ci];
        if (a.page_table) {
            if (request_status(a, rec.b, &s_flag) != SV_OK) continue;
        }
        const int r = chunk * kMergeRows + (tid >> 3), d0 = (tid & 7) * 16;
        const int rr = min(r, rec.rows - 1);
        float M = -INFINITY, Ls = 0.f, acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        for (int c0 = rec.cf; c0 <= ci; c0 += kMergeBatch) {
            float m[kMergeBatch], l[kMergeBatch];
            uint4 v[kMergeBatch][2];
#pragma unroll
            for (int i = 0; i < kMergeBatch; ++i) {
                const int c = min(c0 + i, ci);
                const uint8_t* base = slots + (long long)(c == rec.cf ? rec.cf_slot : 2 * c) * slot_bytes();
                const float* ml = (const float*)(base + (size_t)kUnitRows * kD * 2);
                m[i] = c0 + i <= ci ? __ldcg(ml + rr) : -INFINITY;
                l[i] = __ldcg(ml + kUnitRows + rr);
                const uint4* src = (const uint4*)((const uint16_t*)base + (size_t)rr * kD + d0);
                v[i][0] = __ldcg(src);
                v[i][1] = __ldcg(src + 1);
            }
            float mn = M;
#pragma unroll
            for (int i = 0; i < kMergeBatch; ++i) mn = fmaxf(mn, m[i]);
            const float sc = M == -INFINITY ? 0.f : ex2(M - mn);   // rescale the running sums
            Ls *= sc;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] *= sc;
#pragma unroll
            for (int i = 0; i < kMergeBatch; ++i) {
                // a partial that saw no finite score (or a padding contributor) weighs nothing
                const float w = m[i] == -INFINITY ? 0.f : l[i] * ex2(m[i] - mn);
                Ls += w;
                const uint32_t wv[8] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w,
                                        v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    acc[2 * e] += __uint_as_float(wv[e] << 16) * w;
                    acc[2 * e + 1] += __uint_as_float(wv[e] & 0xffff0000u) * w;
                }
            }
            M = mn;
        }
        if (r < rec.rows) {
            const int qi = rec.row0 + r, t_node = qi / G, g_head = qi - t_node * G;
            const size_t out_row = ((size_t)rec.b * T + t_node) * a.Hq + (size_t)rec.hk * G + g_head;
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
            uint4* dst = (uint4*)((uint16_t*)a.out + out_row * kD + d0);
            dst[0] = make_uint4(pack2<false>(acc[0] * inv, acc[1] * inv), pack2<false>(acc[2] * inv, acc[3] * inv),
                                pack2<false>(acc[4] * inv, acc[5] * inv), pack2<false>(acc[6] * inv, acc[7] * inv));
            dst[1] = make_uint4(pack2<false>(acc[8] * inv, acc[9] * inv), pack2<false>(acc[10] * inv, acc[11] * inv),
                                pack2<false>(acc[12] * inv, acc[13] * inv), pack2<false>(acc[14] * inv, acc[15] * inv));
            if (a.lse && (tid & 7) == 0) a.lse[out_row] = (M + __log2f(Ls)) * 0.69314718055994531f;
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

// A 2D tensor map [rows][inner bytes or elements] with the given box and swizzle.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, unsigned long long inner,
               unsigned long long rows, unsigned long long row_bytes, unsigned box_inner, unsigned box_rows,
               CUtensorMapSwizzle swz) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

int kv_kind(const AttnArgs& a) { return a.kv_dt == SV_E4M3 ? KV_E4M3 : a.kv_dt == SV_E2M1 ? KV_E2M1 : KV_BF16; }

// rows of the cache view the K / V tensor maps cover: contiguous [B*Hkv*kv_cap], paged [num_pages*Hkv*page_size]
long long view_rows(const AttnArgs& a) {
    return a.page_table ? (long long)a.num_pages * a.Hkv << a.page_shift : (long long)a.B * a.Hkv * a.kv_cap;
}

// CTAs that fit on the device at once with this kernel's resources (cached per kernel); the persistent grid
// never exceeds it, so every CTA of the grid is resident from the start.
// merge CTAs resident at once (the merge grid never waits for a second wave)
int merge_ctas() {
    static int n = 0;
    if (!n) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_merge_kernel, kMergeThreads, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        n = per_sm * num_sms();
    }
    return n;
}

template <int KVK, int KS>
int resident_ctas() {
    static int n = 0;
    if (!n) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_tc_kernel<KVK, KS>, threads_of<KVK>(), kSmemAlloc) !=
                cudaSuccess || per_sm < 1)
            per_sm = 1;
        n = per_sm * num_sms();
    }
    return n;
}

template <int KVK, int KS>
cudaError_t launch_main(const AttnArgs& a, cudaStream_t s, float scale_log2, int* grid_out) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<KVK, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap tmK, tmV, tmQ, tmKs, tmVs;
    const long long rows = view_rows(a);
    const unsigned box_rows = a.page_table ? (unsigned)min(1 << a.page_shift, kTileN) : (unsigned)kTileN;
    bool ok;
    if (KVK == KV_BF16) {
        ok = encode_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.k, kD, rows, kD * 2, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B) &&
             encode_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.v, kD, rows, kD * 2, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        tmKs = tmK;
        tmVs = tmV;
    } else if (KVK == KV_E4M3) {
        ok = encode_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k, kD, rows, kD, kD, box_rows, CU_TENSOR_MAP_SWIZZLE_128B) &&
             encode_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v, kD, rows, kD, kD, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        tmKs = tmK;
        tmVs = tmV;
    } else {
        // codes [rows][64 B] with the 64-byte swizzle; block scales [rows / 2][16 B] (two cache rows per TMA row)
        ok = encode_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k, kD / 2, rows, kD / 2, kD / 2, kTileN, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v, kD / 2, rows, kD / 2, kD / 2, kTileN, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_2d(&tmKs, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_block, 16, rows / 2, 16, 16, kTileN / 2, CU_TENSOR_MAP_SWIZZLE_NONE) &&
             encode_2d(&tmVs, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v_block, 16, rows / 2, 16, 16, kTileN / 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return cudaErrorInvalidValue;
    // Q by TMA when the heads of a kv group tile the 128-row M tile; else the softmax warps write it
    const int q_tma = encode_q_map(&tmQ, a) ? 1 : 0;
    if (!q_tma) tmQ = tmK;
    int grid = resident_ctas<KVK, KS>();
    if (grid > kMaxGrid) grid = kMaxGrid;
    *grid_out = grid;
    AttnArgs la = a;
    la.wait_cycles = attn_wait_cycles();
    return launch_ex(attn_tc_kernel<KVK, KS>, dim3(grid), dim3(threads_of<KVK>()), (size_t)kSmemAlloc, s, 1, false, tmK,
                     tmV, tmQ, tmKs, tmVs, la, scale_log2, q_tma, (int)box_rows);
}

// every unit of the launch in split mode (at most 128 query rows per kv head): the 3-slot K ring
template <int KVK>
cudaError_t launch_kind(const AttnArgs& a, cudaStream_t s, float scale_log2, int* grid_out) {
    const bool split_only = (long long)a.T * (a.Hq / a.Hkv) <= kRows;
    return split_only ? launch_main<KVK, 3>(a, s, scale_log2, grid_out) : launch_main<KVK, 2>(a, s, scale_log2, grid_out);
}

}  // namespace

size_t attn_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap) {
    (void)B; (void)T; (void)kv_cap;
    if (D != kD || Hkv < 1 || Hq % Hkv) return 0;
    return (size_t)workspace_bytes();
}

bool attn_tc_supported(const AttnArgs& a) {
    const long long TG = (long long)a.T * (a.Hq / a.Hkv);
    const long long rows = view_rows(a);
    bool ok = a.q_dt == SV_BF16 && (a.kv_dt == SV_BF16 || a.kv_dt == SV_E4M3 || a.kv_dt == SV_E2M1) && a.D == kD &&
              a.B >= 1 && rows < (1LL << 31) - kTileN && TG < 65536 &&
              // tile indices of the whole call fit the kernel's 32-bit bookkeeping
              (long long)a.B * a.Hkv * ((TG + kUnitRows - 1) / kUnitRows) * ((a.kv_cap + kTileN - 1) / kTileN) < (1LL << 24) &&
              tensor_map_encoder() != nullptr;
    if (a.page_table) ok = ok && a.kv_dt != SV_E2M1 && a.page_shift >= 3;   // pages of at least one swizzle atom
    if (a.kv_dt == SV_E2M1) ok = ok && (rows & 1) == 0 && a.kv_cap % 2 == 0;
    return ok;
}

cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const float scale = a.sm_scale != 0.f ? a.sm_scale : (float)(1.0 / sqrt((double)a.D));
    const float sl2 = scale * 1.4426950408889634f;
    int grid = 0;
    switch (kv_kind(a)) {
    case KV_E4M3: e = launch_kind<KV_E4M3>(a, s, sl2, &grid); break;
    case KV_E2M1: e = launch_kind<KV_E2M1>(a, s, sl2, &grid); break;
    default: e = launch_kind<KV_BF16>(a, s, sl2, &grid); break;
    }
    if (e != cudaSuccess) return e;
    return launch_ex(attn_merge_kernel, dim3(merge_ctas()), dim3(kMergeThreads), 0, s, 1, true, a, grid);
}

}  // namespace sv
