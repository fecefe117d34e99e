// sv_internal.cuh -- device helpers and internal launchers of libsv.so (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sv.h"

#define SV_MAX_T 64

namespace sv {

// --------------------------------------------------------------------------------------------- scalars
__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }
__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// OCP E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, S.1111.111 = NaN.
__device__ __forceinline__ float e4m3_to_float(uint32_t c) {
    uint32_t e = (c >> 3) & 15u, m = c & 7u;
    float v;
    if (e == 0) v = (float)m * 0.001953125f;                       // m * 2^-9 (exact)
    else        v = __uint_as_float(((e + 120u) << 23) | (m << 20)); // (1 + m/8) * 2^(e - 7)
    if (e == 15 && m == 7) v = __uint_as_float(0x7fc00000u);
    return (c & 0x80u) ? -v : v;
}

template <int DT> struct Elem;
template <> struct Elem<SV_F32>  { using T = float;    __device__ static float get(const T* p, size_t i) { return p[i]; } };
template <> struct Elem<SV_BF16> { using T = uint16_t; __device__ static float get(const T* p, size_t i) { return bf16_bits_to_float(p[i]); } };
template <> struct Elem<SV_E4M3> { using T = uint8_t;  __device__ static float get(const T* p, size_t i) { return e4m3_to_float(p[i]); } };

// --------------------------------------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// --------------------------------------------------------------------------------------------- tree checks
// Parent array of one request in shared memory; returns SV_OK or SV_ERR_BAD_TREE (all threads agree).
__device__ __forceinline__ int block_tree_check(const int32_t* s_par, int T) {
    int bad = 0;
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
        int p = s_par[i];
        bad |= (i == 0) ? (p != -1) : (p < 0 || p >= i);
    }
    return __syncthreads_or(bad) ? SV_ERR_BAD_TREE : SV_OK;
}

// --------------------------------------------------------------------------------------------- launchers
struct AttnArgs {
    int B, T, Hq, Hkv, D, kv_cap;
    sv_dtype q_dt, kv_dt;
    const void* q;
    const void* k;
    const void* v;
    const float* k_scale;
    const float* v_scale;
    const int32_t* kv_len;
    const int32_t* parent;
    float sm_scale;
    void* out;
    float* lse;
    int32_t* status;
    void* ws;
    size_t ws_bytes;
    // FP4 (e2m1) caches: k / v hold the codes [B, Hkv, kv_cap, D/2]; these the e4m3 block scales [.., D/16]
    const void* k_block = nullptr;
    const void* v_block = nullptr;
    // paged caches: k / v are pools [num_pages, Hkv, page_size, D]; logical position j of request b lives in page
    // page_table[b * max_pages + j / page_size] at offset j % page_size
    const int32_t* page_table = nullptr;
    int page_shift = 0;   // log2(page_size)
    int max_pages = 0;
    int num_pages = 0;
    // SM clock cycles a bounded wait of the attention kernel tries before it gives up (sv_set_wait_limit)
    long long wait_cycles = 1LL << 31;
};

long long attn_wait_cycles();

size_t attn_workspace_size(int B, int T, int Hq, int Hkv, int D, int kv_cap);
bool attn_tc_supported(const AttnArgs& a);
cudaError_t launch_attn_simt(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnArgs& a, cudaStream_t s);

struct AcceptArgs {
    int B, T, V;
    sv_dtype logit_dt;
    const void* target;
    const void* draft;
    const int32_t* tokens;
    const int32_t* parent;
    float temperature;
    float invT;
    const uint32_t* uniforms;
    int32_t* accept_len;
    int32_t* path;
    int32_t* out_tokens;
    int32_t* bonus;
    int32_t* argmax;
    int32_t* status;
    void* ws;
};

size_t accept_workspace_size(int B, int T, int V);
cudaError_t launch_accept(const AcceptArgs& a, cudaStream_t s);
int accept_noalloc_max_rows();
void* accept_noalloc_scratch();

struct LossArgs {
    int N, T, V;
    const void* logits;
    const int32_t* tokens;
    const int32_t* parent;
    const int32_t* labels;
    float* row_loss;
    float* sums;
    void* grad;
    int32_t* status;
    void* ws;
};

size_t loss_workspace_size(int N, int T, int V);
cudaError_t launch_loss(const LossArgs& a, cudaStream_t s);

struct AttnBwdArgs {
    int B, T, Hq, Hkv, D, kv_cap;
    sv_dtype q_dt, kv_dt;
    const void* q;
    const void* k;
    const void* v;
    const int32_t* kv_len;
    const int32_t* parent;
    float sm_scale;
    const void* out;
    const float* lse;
    const void* dout;
    float* dq;
    float* dk;
    float* dv;
    float* delta;   // workspace [B, T, Hq]
    int32_t* status;
};

size_t attn_bwd_workspace_size(int B, int T, int Hq);
cudaError_t launch_attn_bwd(const AttnBwdArgs& a, cudaStream_t s);

struct CompactArgs {
    int B, T, Hkv, D, kv_cap;
    sv_dtype kv_dt;
    void* k;
    void* v;
    const int32_t* kv_len;
    const int32_t* parent;
    const int32_t* accept_len;
    const int32_t* path;
    int32_t* new_kv_len;
    int32_t* status;
};

cudaError_t launch_kv_compact(const CompactArgs& a, cudaStream_t s);

struct ExpandArgs {
    int B, n_front, V, k, n_keep;
    sv_dtype logit_dt;
    const void* logits;
    const float* front_score;
    int32_t* topk_token;
    float* topk_logprob;
    int32_t* child_parent;
    int32_t* child_token;
    float* child_score;
    int32_t* status;
};

#define SV_MAX_EXPAND_K 16
#define SV_MAX_EXPAND_CAND 1024

cudaError_t launch_tree_expand(const ExpandArgs& a, cudaStream_t s);

// Launch with an optional thread-block cluster and programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                      int cluster_x, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// PDL: let the next kernel in the stream start its prologue / wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace sv
