/*
 * oracle.h -- plain CPU reference for speculative tree verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * call it.  It shares no code, header, table or constant generator with the CUDA library; both sides
 * implement the same written definitions independently.
 *
 * Status codes mirror the library's so tests can compare them:
 *   0 ok, 1 invalid argument, 2 bad tree, 3 tree too large (T > 64), 4 unsupported, 5 non-finite input.
 * Dtype codes: 0 = float32, 1 = bfloat16 bits (uint16), 2 = OCP FP8 E4M3 codes (uint8).
 */
#ifndef SV_ORACLE_H
#define SV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tree metadata: depth[i] and ancestor lists by explicit parent walks.  Returns 0 or 2 (bad tree). */
int or_tree_check(int T, const int32_t* parent);
int or_tree_depth(int T, const int32_t* parent, int32_t* depth);

/* Tree-masked GQA attention in float64.  Node i of request b, query head h (kv head h / (Hq/Hkv)),
 * attends to prefix positions [0, kv_len[b]) plus the cache positions kv_len[b] + a of every ancestor a
 * of i (i itself and the root included).  out [B,T,Hq,D] and lse [B,T,Hq] (natural log) are float64.
 * If rows != NULL only the n_rows listed (b, i, h) triples are computed (out/lse indexed as usual).
 * status[b] receives a per-request code.  Returns 0 or an argument error. */
int or_tree_attn(int B, int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, int kv_dt,
                 const void* q, const void* k, const void* v, const float* k_scale, const float* v_scale,
                 const int32_t* kv_len, const int32_t* parent, double sm_scale,
                 const int32_t* rows, int n_rows, double* out, double* lse, int32_t* status);

/* Fixed-point softmax weight of the acceptance contract: W = floor(2^24 * 2^{(y-m)*log2 e}) with the
 * contract's own exp2 (range reduction + degree-7 Horner polynomial in fp32 fma). */
uint32_t or_fx_weight(float y, float m);
float or_fx_exp2(float f); /* the polynomial on [-1/2, 1/2] */
void or_fx_exp2_batch(const float* f, float* out, long n);
void or_fx_weight_batch(const float* y, float m, uint32_t* out, long n);

/* Acceptance.  temperature == 0: greedy argmax walk.  temperature > 0: rejection sampling under the
 * integer contract; draft_logits == NULL selects one-hot proposals.  Outputs as in the library header. */
int or_accept(int B, int T, int V, int logit_dt, const void* target_logits, const void* draft_logits,
              const int32_t* tokens, const int32_t* parent, float temperature, const uint32_t* uniforms,
              int32_t* accept_len, int32_t* path, int32_t* out_tokens, int32_t* bonus, int32_t* argmax,
              int32_t* status);

/* Loss over logged traces, float64.  logits [N*T, V] float64 (or bf16 bits for or_loss).
 * row_loss/row_acc/row_rej [N*T]; sums[3] = {sum acc, sum rej, n_terms}; grad [N*T, V] (may be NULL)
 * = d(loss)/d(logits) with loss = (sum acc + sum rej) / n_terms, n_terms = N * (T - 1). */
int or_loss_f64(int N, int T, int V, const double* logits, const int32_t* tokens, const int32_t* parent,
                const int32_t* labels, double* row_loss, double* row_acc, double* row_rej, double* sums,
                double* grad, int32_t* status);
int or_loss(int N, int T, int V, const uint16_t* logits_bf16, const int32_t* tokens, const int32_t* parent,
            const int32_t* labels, double* row_loss, double* row_acc, double* row_rej, double* sums,
            double* grad, int32_t* status);

/* KV compaction after acceptance: position kv_len[b] + 1 + j of every kv head receives what was at
 * kv_len[b] + path[b, j] (j < accept_len[b]); new_kv_len[b] = kv_len[b] + 1 + accept_len[b].  In place on
 * k_cache / v_cache ([B, Hkv, kv_cap, D] in kv_dt), read-before-write semantics.  status[b]: 0, 1 (bad
 * length or path), 2 (bad tree).  Returns 0 or an argument error. */
int or_kv_compact(int B, int T, int Hkv, int D, int kv_cap, int kv_dt, void* k_cache, void* v_cache,
                  const int32_t* kv_len, const int32_t* parent, const int32_t* accept_len, const int32_t* path,
                  int32_t* new_kv_len, int32_t* status);

/* One level of draft tree expansion: per frontier row the top-k tokens with log-probabilities (float64),
 * then the n_keep best candidates of each request by path score, listed in (slot, rank) order. */
int or_tree_expand(int B, int n_front, int V, int k, int n_keep, int logit_dt, const void* logits,
                   const float* front_score, int32_t* topk_token, double* topk_logprob, int32_t* child_parent,
                   int32_t* child_token, double* child_score, int32_t* status);

/* Backward of the tree-masked attention, float64: dq [B,T,Hq,D], dk / dv [B,Hkv,kv_cap,D] (zero outside
 * [0, kv_len + T)) for the upstream gradient dout [B,T,Hq,D] (in q_dt).  kv_dt f32 or bf16. */
int or_tree_attn_bwd(int B, int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, int kv_dt, const void* q,
                     const void* k, const void* v, const int32_t* kv_len, const int32_t* parent, double sm_scale,
                     const void* dout, double* dq, double* dk, double* dv, int32_t* status);

/* Tree attention over FP4 caches (OCP E2M1 codes, two per byte, even element in the low nibble), one E4M3
 * block scale per 16 elements of a row and an fp32 scale per kv head: value = code * block * head scale.
 * k / v [B, Hkv, kv_cap, D/2] bytes, k_block / v_block [B, Hkv, kv_cap, D/16], k_scale / v_scale [Hkv].
 * rows: NULL (every row) or n_rows (b, i, h) triples.  Returns 9 if memory for one request's decoded
 * caches cannot be allocated. */
int or_tree_attn_e2m1(int B, int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, const void* q,
                      const uint8_t* k, const uint8_t* v, const uint8_t* k_block, const uint8_t* v_block,
                      const float* k_scale, const float* v_scale, const int32_t* kv_len, const int32_t* parent,
                      double sm_scale, const int32_t* rows, int n_rows, double* out, double* lse, int32_t* status);

/* Number of OpenMP threads the oracle will use (1 when built without OpenMP). */
int or_num_threads(void);

/* Set the number of OpenMP threads of later calls (no effect without OpenMP or for n < 1). */
void or_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
