// sv_api.cu -- the C ABI of libsv.so: synchronous validation of host-visible arguments, then launches.
// Semantics, layouts and error behaviour are documented in include/sv.h.
#include <math.h>

#include <atomic>

#include "sv_internal.cuh"

using namespace sv;

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

constexpr long long kDefaultWaitCycles = 1LL << 31;   // about one second at the GB300's clocks
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

}  // namespace

long long sv::attn_wait_cycles() { return g_wait_cycles.load(); }

namespace {

// Most of the work is asynchronous; a failed launch surfaces here.
sv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

}  // namespace

extern "C" {

const char* sv_status_string(sv_status s) {
    switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_BAD_TREE: return "parent array is not a topological tree rooted at node 0";
    case SV_ERR_TREE_TOO_LARGE: return "tree has more than 64 nodes";
    case SV_ERR_UNSUPPORTED: return "unsupported dtype, shape or alignment";
    case SV_ERR_NONFINITE: return "non-finite logits";
    case SV_ERR_TIMEOUT: return "bounded device wait timed out";
    case SV_ERR_CUDA: return "CUDA launch failed";
    case SV_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

int sv_version(void) { return 100; }

sv_status sv_set_wait_limit(long long sm_cycles) {
    if (sm_cycles < 0) return SV_ERR_INVALID_ARG;
    g_wait_cycles.store(sm_cycles == 0 ? kDefaultWaitCycles : sm_cycles);
    return SV_OK;
}

size_t sv_workspace_size(sv_op op, int B, int T, int Hq, int Hkv, int D, int kv_cap, int V) {
    if (B < 0 || T < 1 || T > SV_MAX_T) return 0;
    switch (op) {
    case SV_OP_TREE_ATTN: return attn_workspace_size(B, T, Hq, Hkv, D, kv_cap);
    case SV_OP_ACCEPT: return accept_workspace_size(B, T, V);
    case SV_OP_LOSS: return loss_workspace_size(B, T, V);
    case SV_OP_TREE_ATTN_BWD: return attn_bwd_workspace_size(B, T, Hq);
    }
    return 0;
}

sv_status sv_tree_attn(int B, int T, int Hq, int Hkv, int D, int kv_cap, sv_dtype q_dt, sv_dtype kv_dt,
                       const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                       const float* v_scale, const int32_t* kv_len, const int32_t* parent, float sm_scale,
                       void* out, float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                       sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || B > 65535 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || kv_cap < T) return SV_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return SV_ERR_INVALID_ARG;
    if ((q_dt != SV_F32 && q_dt != SV_BF16) || (kv_dt != SV_F32 && kv_dt != SV_BF16 && kv_dt != SV_E4M3))
        return SV_ERR_UNSUPPORTED;
    if (B == 0) return SV_OK;
    if (!q || !k_cache || !v_cache || !kv_len || !parent || !out) return SV_ERR_INVALID_ARG;
    if (kv_dt == SV_E4M3 && (!k_scale || !v_scale)) return SV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(kv_len, 4) || !aligned(parent, 4) || !aligned(lse, 4) || !aligned(status, 4) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return SV_ERR_UNSUPPORTED;
    AttnArgs a{B, T, Hq, Hkv, D, kv_cap, q_dt, kv_dt, q, k_cache, v_cache, k_scale, v_scale, kv_len, parent,
               sm_scale, out, lse, status, workspace, ws_bytes};
    const bool tc = attn_tc_supported(a);
    if (!tc && (D > 256 || (size_t)(Hq / Hkv) * D > 4096)) return SV_ERR_UNSUPPORTED;
    const size_t need = tc ? attn_workspace_size(B, T, Hq, Hkv, D, kv_cap) : 0;
    if (need && (!workspace || ws_bytes < need || !aligned(workspace, 256))) return SV_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    return from_cuda(tc ? launch_attn_tc(a, s) : launch_attn_simt(a, s));
}

sv_status sv_tree_attn_fp4(int B, int T, int Hq, int Hkv, int D, int kv_cap, sv_dtype q_dt, const void* q,
                           const void* k_codes, const void* v_codes, const void* k_block, const void* v_block,
                           const float* k_scale, const float* v_scale, const int32_t* kv_len, const int32_t* parent,
                           float sm_scale, void* out, float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                           sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || B > 65535 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1 || kv_cap < T) return SV_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return SV_ERR_INVALID_ARG;
    if (q_dt != SV_BF16 || D != 128 || kv_cap % 2) return SV_ERR_UNSUPPORTED;
    if (B == 0) return SV_OK;
    if (!q || !k_codes || !v_codes || !k_block || !v_block || !k_scale || !v_scale || !kv_len || !parent || !out)
        return SV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_codes, 16) || !aligned(v_codes, 16) || !aligned(k_block, 16) ||
        !aligned(v_block, 16) || !aligned(out, 16) || !aligned(kv_len, 4) || !aligned(parent, 4) || !aligned(lse, 4) ||
        !aligned(status, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return SV_ERR_UNSUPPORTED;
    AttnArgs a{B, T, Hq, Hkv, D, kv_cap, q_dt, SV_E2M1, q, k_codes, v_codes, k_scale, v_scale, kv_len, parent,
               sm_scale, out, lse, status, workspace, ws_bytes};
    a.k_block = k_block;
    a.v_block = v_block;
    if (!attn_tc_supported(a)) return SV_ERR_UNSUPPORTED;
    const size_t need = attn_workspace_size(B, T, Hq, Hkv, D, kv_cap);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return SV_ERR_WORKSPACE;
    return from_cuda(launch_attn_tc(a, (cudaStream_t)stream));
}

sv_status sv_tree_attn_paged(int B, int T, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                             sv_dtype q_dt, sv_dtype kv_dt, const void* q, const void* k_pool, const void* v_pool,
                             const float* k_scale, const float* v_scale, const int32_t* page_table,
                             const int32_t* kv_len, const int32_t* parent, float sm_scale, void* out, float* lse,
                             int32_t* status, void* workspace, size_t ws_bytes, sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || B > 65535 || T < 1 || Hq < 1 || Hkv < 1 || Hkv > 65535 || Hq % Hkv || D < 1) return SV_ERR_INVALID_ARG;
    if (page_size < 1 || (page_size & (page_size - 1)) || max_pages < 1 || num_pages < 1) return SV_ERR_INVALID_ARG;
    if ((long long)page_size * max_pages > 0x7fffffffLL || (long long)page_size * max_pages < T) return SV_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return SV_ERR_INVALID_ARG;
    if ((q_dt != SV_F32 && q_dt != SV_BF16) || (kv_dt != SV_F32 && kv_dt != SV_BF16 && kv_dt != SV_E4M3))
        return SV_ERR_UNSUPPORTED;
    if (D > 256 || (size_t)(Hq / Hkv) * D > 4096) return SV_ERR_UNSUPPORTED;
    if (B == 0) return SV_OK;
    if (!q || !k_pool || !v_pool || !page_table || !kv_len || !parent || !out) return SV_ERR_INVALID_ARG;
    if (kv_dt == SV_E4M3 && (!k_scale || !v_scale)) return SV_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(k_pool, 4) || !aligned(v_pool, 4) || !aligned(out, 4) || !aligned(page_table, 4) ||
        !aligned(kv_len, 4) || !aligned(parent, 4) || !aligned(lse, 4) || !aligned(status, 4) ||
        !aligned(k_scale, 4) || !aligned(v_scale, 4))
        return SV_ERR_UNSUPPORTED;
    int shift = 0;
    while ((1 << shift) < page_size) ++shift;
    AttnArgs a{B, T, Hq, Hkv, D, page_size * max_pages, q_dt, kv_dt, q, k_pool, v_pool, k_scale, v_scale, kv_len,
               parent, sm_scale, out, lse, status, workspace, ws_bytes};
    a.page_table = page_table;
    a.page_shift = shift;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    // the tensor-core kernel reads whole 16-byte-aligned rows through TMA
    const bool tc = attn_tc_supported(a) && aligned(q, 16) && aligned(k_pool, 16) && aligned(v_pool, 16) &&
                    aligned(out, 16);
    if (tc) {
        const size_t need = attn_workspace_size(B, T, Hq, Hkv, D, page_size * max_pages);
        if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return SV_ERR_WORKSPACE;
    }
    cudaStream_t s = (cudaStream_t)stream;
    return from_cuda(tc ? launch_attn_tc(a, s) : launch_attn_simt(a, s));
}

sv_status sv_accept(int B, int T, int V, sv_dtype logit_dt, const void* target_logits,
                    const void* draft_logits, const int32_t* tokens, const int32_t* parent, float temperature,
                    const uint32_t* uniforms, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                    int32_t* bonus, int32_t* argmax, int32_t* status, void* workspace, size_t ws_bytes,
                    sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || T < 1 || V < 1) return SV_ERR_INVALID_ARG;
    if ((long long)B * T * 2 * 8 > 0x7fffffffLL) return SV_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_INVALID_ARG;
    if (logit_dt != SV_F32 && logit_dt != SV_BF16) return SV_ERR_UNSUPPORTED;
    const bool stoch = temperature > 0.f;
    if (stoch && !uniforms) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !tokens || !parent || !accept_len || !path || !out_tokens || !bonus)
        return SV_ERR_INVALID_ARG;
    if (!aligned(target_logits, 16) || !aligned(draft_logits, 16) || !aligned(tokens, 4) || !aligned(parent, 4) ||
        !aligned(uniforms, 4) || !aligned(accept_len, 4) || !aligned(path, 4) || !aligned(out_tokens, 4) ||
        !aligned(bonus, 4) || !aligned(argmax, 4) || !aligned(status, 4))
        return SV_ERR_UNSUPPORTED;
    const size_t need = accept_workspace_size(B, T, V);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return SV_ERR_WORKSPACE;
    AcceptArgs a{B, T, V, logit_dt, target_logits, stoch ? draft_logits : nullptr, tokens, parent, temperature,
                 stoch ? (float)(1.0 / (double)temperature) : 1.f, uniforms, accept_len, path, out_tokens,
                 bonus, argmax, status, workspace};
    return from_cuda(launch_accept(a, (cudaStream_t)stream));
}

sv_status sv_accept_noalloc(int B, int T, int V, sv_dtype logit_dt, const void* target_logits,
                            const void* draft_logits, const int32_t* tokens, const int32_t* parent,
                            float temperature, const uint32_t* uniforms, int32_t* accept_len, int32_t* path,
                            int32_t* out_tokens, int32_t* bonus, int32_t* argmax, int32_t* status,
                            sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || T < 1 || V < 1) return SV_ERR_INVALID_ARG;
    if ((long long)B * T > accept_noalloc_max_rows()) return SV_ERR_WORKSPACE;
    if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_INVALID_ARG;
    if (logit_dt != SV_F32 && logit_dt != SV_BF16) return SV_ERR_UNSUPPORTED;
    const bool stoch = temperature > 0.f;
    if (stoch && !uniforms) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!target_logits || !tokens || !parent || !accept_len || !path || !out_tokens || !bonus)
        return SV_ERR_INVALID_ARG;
    if (!aligned(target_logits, 16) || !aligned(draft_logits, 16) || !aligned(tokens, 4) || !aligned(parent, 4) ||
        !aligned(uniforms, 4) || !aligned(accept_len, 4) || !aligned(path, 4) || !aligned(out_tokens, 4) ||
        !aligned(bonus, 4) || !aligned(argmax, 4) || !aligned(status, 4))
        return SV_ERR_UNSUPPORTED;
    void* scratch = accept_noalloc_scratch();
    if (!scratch) return SV_ERR_CUDA;
    AcceptArgs a{B, T, V, logit_dt, target_logits, stoch ? draft_logits : nullptr, tokens, parent, temperature,
                 stoch ? (float)(1.0 / (double)temperature) : 1.f, uniforms, accept_len, path, out_tokens,
                 bonus, argmax, status, scratch};
    return from_cuda(launch_accept(a, (cudaStream_t)stream));
}

sv_status sv_loss(int N, int T, int V, const void* draft_logits, const int32_t* tokens,
                  const int32_t* parent, const int32_t* labels, float* row_loss, float* sums, void* grad,
                  int32_t* status, void* workspace, size_t ws_bytes, sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (N < 0 || T < 1 || V < 2) return SV_ERR_INVALID_ARG;
    if ((long long)N * T * 8 > 0x7fffffffLL) return SV_ERR_INVALID_ARG;
    if (!sums) return SV_ERR_INVALID_ARG;
    if (N > 0 && (!draft_logits || !tokens || !parent || !labels || !row_loss)) return SV_ERR_INVALID_ARG;
    if (!aligned(draft_logits, 16) || !aligned(grad, 16) || !aligned(tokens, 4) || !aligned(parent, 4) ||
        !aligned(labels, 4) || !aligned(row_loss, 4) || !aligned(sums, 4) || !aligned(status, 4))
        return SV_ERR_UNSUPPORTED;
    const size_t need = loss_workspace_size(N, T, V);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return SV_ERR_WORKSPACE;
    LossArgs a{N, T, V, draft_logits, tokens, parent, labels, row_loss, sums, grad, status, workspace};
    return from_cuda(launch_loss(a, (cudaStream_t)stream));
}

sv_status sv_tree_attn_bwd(int B, int T, int Hq, int Hkv, int D, int kv_cap, sv_dtype q_dt, sv_dtype kv_dt,
                           const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                           const int32_t* parent, float sm_scale, const void* out, const float* lse,
                           const void* dout, float* dq, float* dk, float* dv, int32_t* status, void* workspace,
                           size_t ws_bytes, sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || B > 65535 || T < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || kv_cap < T) return SV_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f) || isinf(sm_scale)) return SV_ERR_INVALID_ARG;
    if ((q_dt != SV_F32 && q_dt != SV_BF16) || (kv_dt != SV_F32 && kv_dt != SV_BF16)) return SV_ERR_UNSUPPORTED;
    if ((D != 32 && D != 64 && D != 128) || (size_t)(Hq / Hkv) * D > 2048) return SV_ERR_UNSUPPORTED;
    if (Hkv > 65535 || (kv_cap + 15) / 16 > 0x7fffffff) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!q || !k_cache || !v_cache || !kv_len || !parent || !out || !lse || !dout || !dq || !dk || !dv)
        return SV_ERR_INVALID_ARG;
    if (!aligned(q, 4) || !aligned(k_cache, 4) || !aligned(v_cache, 4) || !aligned(out, 4) || !aligned(dout, 4) ||
        !aligned(lse, 4) || !aligned(dq, 4) || !aligned(dk, 4) || !aligned(dv, 4) || !aligned(kv_len, 4) ||
        !aligned(parent, 4) || !aligned(status, 4))
        return SV_ERR_UNSUPPORTED;
    const size_t need = attn_bwd_workspace_size(B, T, Hq);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return SV_ERR_WORKSPACE;
    AttnBwdArgs a{B, T, Hq, Hkv, D, kv_cap, q_dt, kv_dt, q, k_cache, v_cache, kv_len, parent, sm_scale, out, lse,
                  dout, dq, dk, dv, (float*)workspace, status};
    return from_cuda(launch_attn_bwd(a, (cudaStream_t)stream));
}

sv_status sv_kv_compact(int B, int T, int Hkv, int D, int kv_cap, sv_dtype kv_dt, void* k_cache, void* v_cache,
                        const int32_t* kv_len, const int32_t* parent, const int32_t* accept_len,
                        const int32_t* path, int32_t* new_kv_len, int32_t* status, sv_stream_t stream) {
    if (T > SV_MAX_T) return SV_ERR_TREE_TOO_LARGE;
    if (B < 0 || B > 65535 || T < 1 || Hkv < 1 || D < 1 || kv_cap < T || (long long)B * Hkv > 0x7fffffffLL)
        return SV_ERR_INVALID_ARG;
    if (kv_dt != SV_F32 && kv_dt != SV_BF16 && kv_dt != SV_E4M3) return SV_ERR_UNSUPPORTED;
    const int esz = kv_dt == SV_F32 ? 4 : kv_dt == SV_BF16 ? 2 : 1;
    if ((D * esz) % 16 || D * esz > 8192) return SV_ERR_UNSUPPORTED;
    if (B == 0) return SV_OK;
    if (!k_cache || !v_cache || !kv_len || !parent || !accept_len || !path || !new_kv_len) return SV_ERR_INVALID_ARG;
    if ((const void*)new_kv_len == (const void*)kv_len) return SV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(kv_len, 4) || !aligned(parent, 4) ||
        !aligned(accept_len, 4) || !aligned(path, 4) || !aligned(new_kv_len, 4) || !aligned(status, 4))
        return SV_ERR_UNSUPPORTED;
    CompactArgs a{B, T, Hkv, D, kv_cap, kv_dt, k_cache, v_cache, kv_len, parent, accept_len, path, new_kv_len, status};
    return from_cuda(launch_kv_compact(a, (cudaStream_t)stream));
}

sv_status sv_tree_expand(int B, int n_front, int V, int k, int n_keep, sv_dtype logit_dt, const void* logits,
                         const float* front_score, int32_t* topk_token, float* topk_logprob, int32_t* child_parent,
                         int32_t* child_token, float* child_score, int32_t* status, sv_stream_t stream) {
    if (B < 0 || B > 65535 || n_front < 1 || V < 1 || k < 1 || k > V || n_keep < 0) return SV_ERR_INVALID_ARG;
    if (k > SV_MAX_EXPAND_K || n_front * k > SV_MAX_EXPAND_CAND || n_keep > n_front * k) return SV_ERR_INVALID_ARG;
    if ((long long)B * n_front * 8 > 0x7fffffffLL) return SV_ERR_INVALID_ARG;
    if (logit_dt != SV_F32 && logit_dt != SV_BF16) return SV_ERR_UNSUPPORTED;
    if (B == 0) return SV_OK;
    if (!logits || !front_score || !topk_token || !topk_logprob) return SV_ERR_INVALID_ARG;
    if (n_keep > 0 && (!child_parent || !child_token || !child_score)) return SV_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || !aligned(front_score, 4) || !aligned(topk_token, 4) || !aligned(topk_logprob, 4) ||
        !aligned(child_parent, 4) || !aligned(child_token, 4) || !aligned(child_score, 4) || !aligned(status, 4))
        return SV_ERR_UNSUPPORTED;
    ExpandArgs a{B, n_front, V, k, n_keep, logit_dt, logits, front_score, topk_token, topk_logprob, child_parent,
                 child_token, child_score, status};
    return from_cuda(launch_tree_expand(a, (cudaStream_t)stream));
}

}  // extern "C"
