/*
 * sv.h -- C ABI of libsv.so: speculative tree verification on one GB300 (sm_103a).
 *
 * Three hot-path calls sit under a speculative-decoding server's verify step and under its online draft
 * trainer:
 *   sv_tree_attn  tree-masked GQA attention of every draft-tree node over the request's KV prefix and its
 *                 own ancestors ("Aurora" post, section 2: a custom attention mask that follows the
 *                 speculative tree's causal structure so all branches go through one batched pass);
 *   sv_accept     the target's verification of the draft tree: greedy argmax matching or rejection
 *                 sampling, giving the acceptance length (TIDE evaluation section: draft tokens accepted
 *                 per verification step), the accepted path and the target's own next token;
 *   sv_loss       the draft-training signal from logged trees ("Aurora" post, section 2: cross-entropy on
 *                 accepted tokens plus a rejection loss on rejected branches), taken here as
 *                 -log q(accepted token) and -log(1 - q(rejected token)), with its gradient.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument except the host scalars is DEVICE memory owned by the caller.  The library
 *    allocates nothing, keeps no state between calls and never synchronises the stream.
 *  - Work is enqueued on `stream` and runs asynchronously; outputs are valid once the stream reaches the
 *    call.  Calls on different streams may overlap only if they use different workspaces and outputs.
 *  - A draft tree is a parent array int32 [T] per request: parent[0] = -1 (node 0 is the root, the last
 *    committed token) and 0 <= parent[i] < i for i >= 1 (topological order).  Siblings are ordered by
 *    node id, which is the draft's rank order.  T <= 64.
 *  - Errors in host-visible arguments (sizes, dtypes, NULL or misaligned pointers, a workspace that is
 *    too small) are returned synchronously and nothing is launched.  Errors in device data (a malformed
 *    parent array, a token >= V, kv_len + T > kv_cap, non-finite logits) are reported per request in the
 *    optional status array with the same codes; the call still returns SV_OK.  No kernel ever traps.
 *  - Alignment: tensors read with 128-bit loads (q, caches, logits, gradient) must be 16-byte aligned and
 *    their row lengths (D or V elements) must keep every row 16-byte aligned, otherwise SV_ERR_UNSUPPORTED.
 *    int32 / float arrays must be 4-byte aligned.
 *  - SV_ERR_CUDA means a launch failed; cudaGetLastError() holds the CUDA code.
 */
#ifndef SV_H
#define SV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sv_stream_t; /* == cudaStream_t; NULL is the legacy default stream */

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,      /* bad size, NULL pointer, or (per request) token/kv_len out of range  */
    SV_ERR_BAD_TREE = 2,         /* (per request) parent array is not a topological tree rooted at 0     */
    SV_ERR_TREE_TOO_LARGE = 3,   /* T > 64                                                               */
    SV_ERR_UNSUPPORTED = 4,      /* dtype / shape / alignment combination not provided                   */
    SV_ERR_NONFINITE = 5,        /* (per request) NaN or Inf in a logit row the call reads               */
    SV_ERR_TIMEOUT = 6,          /* (per request) a bounded device-side wait gave up                     */
    SV_ERR_CUDA = 7,             /* a CUDA launch failed                                                  */
    SV_ERR_WORKSPACE = 8         /* workspace NULL or smaller than sv_workspace_size()                   */
} sv_status;

/* SV_E2M1: FP4 caches in the NVFP4 layout, only through sv_tree_attn_fp4 (codes plus block scales). */
typedef enum { SV_F32 = 0, SV_BF16 = 1, SV_E4M3 = 2, SV_E2M1 = 3 } sv_dtype;

typedef enum { SV_OP_TREE_ATTN = 0, SV_OP_ACCEPT = 1, SV_OP_LOSS = 2, SV_OP_TREE_ATTN_BWD = 3 } sv_op;

/* Human-readable name of a status code (static storage). */
const char* sv_status_string(sv_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int sv_version(void);

/*
 * sv_set_wait_limit -- diagnostic: how long a bounded wait of the tensor-core attention kernels tries before it
 * gives up, in SM clock cycles (0 restores the default, 2^31: about one second).  No kernel of the library ever
 * waits without a bound: a lost arrival ends the wait, the kernel winds down (waiting with the full limit for its
 * own copies and MMAs) and every request of the call gets SV_ERR_TIMEOUT.  A tiny limit makes those waits give up
 * at once, so a test can drive the failure path without faulting or hanging the GPU.  Process-wide setting read
 * when a call is launched (a CUDA graph keeps the value it was captured with); negative values are rejected.
 */
sv_status sv_set_wait_limit(long long sm_cycles);

/*
 * Bytes of device workspace a call needs (0 if none).  Arguments that do not apply to `op` are ignored:
 *   SV_OP_TREE_ATTN: B, T, Hq, Hkv, D, kv_cap      SV_OP_ACCEPT: B (= rows/T), T, V      SV_OP_LOSS: B (= N), T, V
 *   SV_OP_TREE_ATTN_BWD: B, T, Hq
 * The result is an upper bound that does not depend on device data, so it can be computed once.
 */
size_t sv_workspace_size(sv_op op, int B, int T, int Hq, int Hkv, int D, int kv_cap, int V);

/*
 * sv_tree_attn -- tree-masked grouped-query attention for one verification step.
 *
 * For request b, node i (0 <= i < T) and query head h, with kv head hk = h / (Hq / Hkv):
 *     allowed(b, i) = { 0 .. kv_len[b]-1 }  U  { kv_len[b] + a : a is i, an ancestor of i, or the root }
 *     out[b,i,h,:]  = sum_{j in allowed} softmax_j( sm_scale * <q[b,i,h,:], K[b,hk,j,:]> ) * V[b,hk,j,:]
 *     lse[b,i,h]    = log sum_{j in allowed} exp( sm_scale * <q, K_j> )            (natural log)
 * The tree's own K/V (node a) sit in the cache at position kv_len[b] + a, already written by the caller.
 *
 *   q        [B, T, Hq, D]        q_dt  (SV_F32 or SV_BF16)
 *   k_cache  [B, Hkv, kv_cap, D]  kv_dt (SV_F32, SV_BF16, or SV_E4M3 with per-kv-head scales)
 *   v_cache  [B, Hkv, kv_cap, D]  kv_dt
 *   k_scale, v_scale  float [Hkv]: real value = decoded E4M3 * scale; required for SV_E4M3, else ignored
 *   kv_len   int32 [B]  prefix length L_b; requires 0 <= L_b and L_b + T <= kv_cap (else status 1)
 *   parent   int32 [B, T]
 *   sm_scale float; 0 selects 1/sqrt(D)
 *   out      [B, T, Hq, D] in q_dt
 *   lse      float [B, T, Hq] or NULL
 *   status   int32 [B] or NULL; a failed request's out/lse rows are zero
 *   workspace / ws_bytes: at least sv_workspace_size(SV_OP_TREE_ATTN, ...) bytes, 256-byte aligned; any
 *            content (every call writes what it reads back); never shared by two calls that may overlap
 * Cache positions >= kv_len[b] + T are never used, whatever they hold (NaN included).
 * Shapes: 1 <= T <= 64, Hq % Hkv == 0.  The tensor-core path takes bf16 Q with bf16 or E4M3 caches and
 * D = 128; everything else (f32 tensors, D up to 256 with Hq / Hkv * D <= 4096) runs on the CUDA-core path.
 */
sv_status sv_tree_attn(int B, int T, int Hq, int Hkv, int D, int kv_cap, sv_dtype q_dt, sv_dtype kv_dt,
                       const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                       const float* v_scale, const int32_t* kv_len, const int32_t* parent, float sm_scale,
                       void* out, float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                       sv_stream_t stream);

/*
 * sv_tree_attn_fp4 -- sv_tree_attn over FP4 KV caches.
 *
 * The pages name FP4 among the serving stack's precisions ("Aurora" post, section 1: production speed-up depends
 * on the kernels and their numerical precision, FP8/FP4) but fix no format.  This call reads the NVFP4 layout the
 * GB300 tensor cores use natively: OCP E2M1 codes, two per byte with the even element in the low nibble, one
 * E4M3 block scale per 16 consecutive elements of a cache row, and an fp32 scale per kv head:
 *     K[b, hk, j, d] = e2m1(code) * e4m3(k_block[b, hk, j, d / 16]) * k_scale[hk]      (V likewise)
 * The attention is exactly sv_tree_attn's ("Aurora" post, section 2) over those values.
 *   k_codes, v_codes   uint8 [B, Hkv, kv_cap, D/2]
 *   k_block, v_block   uint8 [B, Hkv, kv_cap, D/16] E4M3 codes
 *   k_scale, v_scale   float [Hkv]
 *   q, kv_len, parent, sm_scale, out, lse, status, workspace: as for sv_tree_attn
 * Shapes: q_dt SV_BF16, D = 128, kv_cap even, 1 <= T <= 64, Hq % Hkv == 0; all cache pointers 16-byte aligned.
 * Tensor cores: every decoded value (a 2-bit-mantissa code times a 4-bit-mantissa scale) is exactly an f16 value,
 * so the caches are expanded to f16 in shared memory and the MMAs run on f16 operands (Q rounded to f16), with
 * fp32 accumulation; the head scales fold into the softmax scale and the output.  Workspace: as sv_tree_attn's
 * (sv_workspace_size(SV_OP_TREE_ATTN, ...)).  Anything else returns SV_ERR_UNSUPPORTED.
 */
sv_status sv_tree_attn_fp4(int B, int T, int Hq, int Hkv, int D, int kv_cap, sv_dtype q_dt, const void* q,
                           const void* k_codes, const void* v_codes, const void* k_block, const void* v_block,
                           const float* k_scale, const float* v_scale, const int32_t* kv_len, const int32_t* parent,
                           float sm_scale, void* out, float* lse, int32_t* status, void* workspace, size_t ws_bytes,
                           sv_stream_t stream);

/*
 * sv_tree_attn_paged -- sv_tree_attn over a paged KV cache.
 *
 * Serving systems keep the KV cache in fixed-size pages shared by all requests and give each request a
 * page table.  The attention is exactly sv_tree_attn's ("Aurora" post, section 2) over each request's
 * logical cache, whose position j (0 <= j < max_pages * page_size) lives at
 *     pool[page_table[b, j / page_size], hk, j % page_size, :]
 * with the tree's own K/V at logical positions kv_len[b] .. kv_len[b] + T - 1, as in sv_tree_attn.
 *   k_pool, v_pool  [num_pages, Hkv, page_size, D] in kv_dt (SV_F32, SV_BF16, SV_E4M3 + per-head scales)
 *   page_table      int32 [B, max_pages]; entries past the pages a request reads are ignored
 *   page_size       a power of two
 *   q, out, lse, kv_len, parent, sm_scale, status: as for sv_tree_attn, with kv_cap = max_pages * page_size
 *   workspace / ws_bytes: at least sv_workspace_size(SV_OP_TREE_ATTN, B, T, Hq, Hkv, D, max_pages * page_size, 0)
 *                   bytes, 256-byte aligned, when that size is not 0 (else may be NULL)
 * A request whose kv_len + T exceeds max_pages * page_size, or that reads a page id outside
 * [0, num_pages), gets status SV_ERR_INVALID_ARG and zero outputs.  bf16 Q with bf16 or e4m3 pools, D = 128 and
 * pages of at least 8 rows run on the tensor-core kernel (the K/V tiles are gathered page by page by TMA);
 * everything else on the CUDA-core attention kernel (fp32 arithmetic, any D up to 256).
 */
sv_status sv_tree_attn_paged(int B, int T, int Hq, int Hkv, int D, int page_size, int max_pages, int num_pages,
                             sv_dtype q_dt, sv_dtype kv_dt, const void* q, const void* k_pool, const void* v_pool,
                             const float* k_scale, const float* v_scale, const int32_t* page_table,
                             const int32_t* kv_len, const int32_t* parent, float sm_scale, void* out, float* lse,
                             int32_t* status, void* workspace, size_t ws_bytes, sv_stream_t stream);

/*
 * sv_accept -- verify one batch of draft trees against the target's per-node logits.
 *
 * Row i of request b (target_logits[b, i, :]) is the target's next-token logits after node i.  The walk
 * starts at the root; at node `cur` its children are tried in ascending node id:
 *   greedy (temperature == 0): the first child whose token equals argmax(row cur) (lowest index on ties)
 *       is accepted; if none, the walk stops and bonus = argmax(row cur).
 *   stochastic (temperature > 0): standard speculative sampling, accept with probability min(1, p/q) and
 *       otherwise continue with the residual norm(max(0, p - q)), under an exact integer contract so
 *       results are reproducible bit for bit:
 *         y = fp32(z) * invT, invT = (float)(1 / (double)temperature); m = max y; t = (y - m) * log2(e);
 *         W = 0 if t < -24, else floor(P(t - n) * 2^(24 + n)), n = rint(t), P the degree-7 Horner
 *         polynomial with coefficients fp32((ln 2)^j / j!) evaluated with fma;  S = sum W  (p ~ W / S).
 *       child c with token x is accepted iff  U_c * Wq(x) * S'_p  <  2^32 * W'_p(x) * S_q   (128-bit),
 *       U_c = uniforms[b, c].  On rejection, W'_p(k) <- floor(max(0, W'_p(k) S_q - Wq(k) S'_p) / S_q).
 *       draft_logits == NULL means one-hot proposals (q = delta of the child's token: rejection zeroes
 *       that token).  When the walk stops, the bonus token is the smallest j whose prefix sum of the
 *       final weights exceeds floor(uniforms[b, 0] * R / 2^32), R = sum of the weights: the residual after
 *       rejections (or the row itself when it is empty) or, at a node with no children, the node's row.
 *   Outputs (for a failed request: accept_len = bonus = -1, path/out_tokens all -1):
 *   accept_len int32 [B]     number of accepted DRAFT tokens (root and bonus not counted)
 *   path       int32 [B, T]  accepted node ids in order, then -1
 *   out_tokens int32 [B, T]  tokens of the accepted nodes, then the bonus token, then -1
 *   bonus      int32 [B]
 *   argmax     int32 [B, T] or NULL: argmax of every target row (first index; -1 if the row is not finite)
 *   status     int32 [B] or NULL
 *   target_logits / draft_logits: [B, T, V] in logit_dt (SV_F32 or SV_BF16); the draft row of a node is
 *       its proposal distribution for the node's children.  tokens int32 [B, T] (tokens[b,0] unused).
 *   uniforms uint32 [B, T], raw 32-bit uniforms; required iff temperature > 0.
 *   workspace: at least sv_workspace_size(SV_OP_ACCEPT, B, T, 0, 0, 0, 0, V) bytes.
 */
sv_status sv_accept(int B, int T, int V, sv_dtype logit_dt, const void* target_logits,
                    const void* draft_logits, const int32_t* tokens, const int32_t* parent, float temperature,
                    const uint32_t* uniforms, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                    int32_t* bonus, int32_t* argmax, int32_t* status, void* workspace, size_t ws_bytes,
                    sv_stream_t stream);

/*
 * sv_accept_noalloc -- sv_accept for callers that cannot allocate device memory.
 *
 * The method's pages have no counterpart to this call; it is an interface convenience.  Some callers
 * cannot hand the library a workspace: code that runs where allocation is not allowed (a serving loop
 * whose allocator is owned by another framework, a plugin without access to an allocator, a real-time
 * path that must never call cudaMalloc).  This entry point takes the same arguments as sv_accept minus
 * the workspace and gives identical results; it allocates nothing.  Its scratch is a fixed 3 MiB array
 * of static device memory inside the library, which every GPU that loads the library keeps until the
 * process exits.
 *   Limit: B * T <= 65536 (target rows); larger calls return SV_ERR_WORKSPACE and launch nothing.
 *   The first call on each device looks up the array's device address on that device (with that device
 *   current); make that first call before any CUDA stream capture.
 *   Every call uses the same array: calls that overlap on the GPU (other streams, other host threads)
 *   race and corrupt each other's results, so the caller must serialise them.  Nothing in the array
 *   needs to start at zero.
 */
sv_status sv_accept_noalloc(int B, int T, int V, sv_dtype logit_dt, const void* target_logits,
                            const void* draft_logits, const int32_t* tokens, const int32_t* parent,
                            float temperature, const uint32_t* uniforms, int32_t* accept_len, int32_t* path,
                            int32_t* out_tokens, int32_t* bonus, int32_t* argmax, int32_t* status,
                            sv_stream_t stream);

/*
 * sv_loss -- acceptance + rejection loss of the draft over N logged trees, and its gradient.
 *
 * Row (n, p) of draft_logits ([N*T, V], bf16) is the draft's logits after node p of trace n; q_p is its
 * softmax.  For every non-root node j with parent p and token x = tokens[n, j]:
 *     accepted  (x == labels[n, p], the target's token after p):  term = -log q_p(x)
 *     rejected  (otherwise):                                       term = -log(1 - q_p(x)), q_p(x) <= 1 - 1e-6
 * loss = (sum of accepted terms + sum of rejected terms) / n_terms,  n_terms = N * (T - 1).
 *   row_loss  float [N*T]   sum of the terms of row p's children (0 for leaves)
 *   sums      float [3]     { sum accepted, sum rejected, n_terms } (fixed-order reduction: deterministic)
 *   grad      bf16 [N*T, V] d loss / d draft_logits (leaf rows are zero), or NULL to skip it
 *   status    int32 [N] or NULL; a failed trace contributes no terms and a zero gradient
 *   workspace: at least sv_workspace_size(SV_OP_LOSS, N, T, 0, 0, 0, 0, V) bytes.
 */
sv_status sv_loss(int N, int T, int V, const void* draft_logits, const int32_t* tokens,
                  const int32_t* parent, const int32_t* labels, float* row_loss, float* sums, void* grad,
                  int32_t* status, void* workspace, size_t ws_bytes, sv_stream_t stream);

/*
 * sv_tree_attn_bwd -- gradient of sv_tree_attn for training the draft on its trees.
 *
 * The draft is trained on every accepted and rejected branch of its logged trees in one batched forward
 * and backward pass ("Aurora" post, section 2), so the tree attention of that pass needs its gradient under
 * the same ancestor mask.  Given the forward's inputs, its output `out` and log-sum-exp `lse` (as written by
 * sv_tree_attn) and the upstream gradient dout = d loss / d out, with p_j = exp(s_j - lse),
 * s_j = sm_scale <q, k_j> over the allowed set of sv_tree_attn and delta = <dout, out> per query row:
 *     dq  = sm_scale * sum_j p_j (<dout, v_j> - delta) k_j
 *     dk_j = sm_scale * sum over query rows that see j of p_j (<dout, v_j> - delta) q
 *     dv_j = sum over query rows that see j of p_j dout
 *   q, out, dout  [B, T, Hq, D] in q_dt (SV_F32 or SV_BF16); k_cache, v_cache [B, Hkv, kv_cap, D] in kv_dt
 *                 (SV_F32 or SV_BF16); kv_len, parent, sm_scale as for sv_tree_attn
 *   lse           float [B, T, Hq] from the forward
 *   dq            float [B, T, Hq, D]
 *   dk, dv        float [B, Hkv, kv_cap, D]: positions [0, kv_len[b] + T) are written (a position no query row
 *                 sees gets 0); positions from kv_len[b] + T on are not touched
 *   status        int32 [B] or NULL; a failed request gets zero dq and untouched dk / dv
 *   workspace: at least sv_workspace_size(SV_OP_TREE_ATTN_BWD, B, T, Hq, ...) bytes (delta per query row)
 * Shapes: 1 <= T <= 64, Hq % Hkv == 0, D in {32, 64, 128}, (Hq / Hkv) * D <= 2048.  CUDA-core arithmetic in
 * fp32; results are deterministic (fixed reduction order, no atomics).
 */
sv_status sv_tree_attn_bwd(int B, int T, int Hq, int Hkv, int D, int kv_cap, sv_dtype q_dt, sv_dtype kv_dt,
                           const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_len,
                           const int32_t* parent, float sm_scale, const void* out, const float* lse,
                           const void* dout, float* dq, float* dk, float* dv, int32_t* status, void* workspace,
                           size_t ws_bytes, sv_stream_t stream);

/*
 * sv_kv_compact -- make the accepted path's K/V contiguous after verification.
 *
 * After sv_accept the committed tokens of request b are the root plus the accepted path ("Aurora" post,
 * section 2, and the TIDE overview: the target keeps the accepted continuation of the draft).  The root's
 * K/V are at cache position L = kv_len[b] (the first tree slot) and accepted node path[b, j] at
 * L + path[b, j]; this call moves them so that, for every kv head,
 *     K/V[b, :, L + 1 + j, :]  <-  K/V[b, :, L + path[b, j], :]      j = 0 .. accept_len[b] - 1
 * with every read seeing the cache as it was before the call, and writes new_kv_len[b] = L + 1 +
 * accept_len[b]: the next verification step sees a causal prefix.  Positions past the new length keep
 * whatever they held.  The copy is in place on the caches; it moves bytes, so the result is exact for
 * every kv_dt.
 *   k_cache, v_cache  [B, Hkv, kv_cap, D] in kv_dt (SV_F32, SV_BF16 or SV_E4M3 codes); D * element size
 *                     must be a multiple of 16 bytes and at most 8192
 *   kv_len     int32 [B]     the prefix length the tree was verified against
 *   parent     int32 [B, T]  the verified tree
 *   accept_len int32 [B], path int32 [B, T]: as written by sv_accept
 *   new_kv_len int32 [B]     output; must not alias kv_len
 *   status     int32 [B] or NULL: SV_ERR_BAD_TREE for a malformed parent array, SV_ERR_INVALID_ARG for
 *              accept_len < 0 (a failed verification) or > T - 1, a path that is not a walk down the tree
 *              from the root, or kv_len + T > kv_cap.  Such a request is left untouched and its
 *              new_kv_len is kv_len.
 * No workspace.  Requests and kv heads are independent CTAs; the call never reads positions below L.
 */
sv_status sv_kv_compact(int B, int T, int Hkv, int D, int kv_cap, sv_dtype kv_dt, void* k_cache, void* v_cache,
                        const int32_t* kv_len, const int32_t* parent, const int32_t* accept_len,
                        const int32_t* path, int32_t* new_kv_len, int32_t* status, sv_stream_t stream);

/*
 * sv_tree_expand -- one level of draft tree expansion, the step that builds the tree verified next.
 *
 * The draft proposes the tokens the target then verifies in one pass ("Aurora" post, section 2; TIDE
 * overview).  Row s of request b (logits[b, s, :]) is the draft's next-token logits after frontier node s,
 * whose path score front_score[b, s] is the sum of the draft's log-probabilities from the root (0 for the
 * root).  Each row proposes its k most likely tokens: larger logit first, lower token id first on equal
 * logits, with log-probability z - logsumexp(row) at temperature 1.  A candidate's score is its frontier
 * node's score plus its log-probability; the n_keep best candidates of the request survive (higher score
 * first, then lower slot, then lower rank) and are listed in (slot, rank) order, which is the breadth-first
 * numbering of the next level.  Calling this once per level with (n_front, k, n_keep) = (n_{d-1}, k_d, n_d)
 * builds a tree with a fixed node budget per level.
 *   logits       [B, n_front, V] in logit_dt (SV_F32 or SV_BF16)
 *   front_score  float [B, n_front]
 *   topk_token   int32 [B, n_front, k], topk_logprob float [B, n_front, k]   (outputs, required)
 *   child_parent int32 [B, n_keep] frontier slot of each survivor; child_token int32 [B, n_keep];
 *   child_score  float [B, n_keep] = front_score + log-probability, rounded to float32 once
 *   status       int32 [B] or NULL: SV_ERR_NONFINITE when a row of the request holds NaN/Inf or its
 *                front_score is not finite; that request's outputs are -1 (tokens, slots) and -inf.
 * Limits: 1 <= k <= min(16, V), n_front * k <= 1024, 0 <= n_keep <= n_front * k.  Log-probabilities are
 * computed in float32 (the scores of two candidates closer than about 1e-5 may rank differently from an
 * exact computation).  No workspace.
 */
sv_status sv_tree_expand(int B, int n_front, int V, int k, int n_keep, sv_dtype logit_dt, const void* logits,
                         const float* front_score, int32_t* topk_token, float* topk_logprob, int32_t* child_parent,
                         int32_t* child_token, float* child_score, int32_t* status, sv_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SV_H */
