/*
 * oracle.c -- plain, slow, obviously-correct CPU reference for speculative tree verification.
 *
 * TEST INFRASTRUCTURE ONLY: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg load
 * this library.  It shares nothing with the CUDA path.
 *
 * What it follows (page titles and sections of the method's public descriptions):
 *  - "Aurora" blog post, section 2 (core idea): the target verifies the draft's proposals in parallel;
 *    a tree-attention mask built from the speculative tree's causal structure lets every accepted and
 *    rejected branch be processed in one batched pass; the draft is trained with an acceptance loss
 *    (cross-entropy on accepted tokens) and a rejection loss on rejected branches.
 *  - "TIDE" (moreh.io) overview and evaluation: drafts are verified in one target pass; the acceptance
 *    length is the number of draft tokens the target accepts per verification step.
 *  The pages give no formulas.  The attention is the plain masked-softmax definition; the stochastic
 *  rule is standard speculative sampling (accept with min(1, p/q), resample from norm(max(0, p - q)));
 *  the rejection term is -log(1 - q(token)).  The integer contract that makes acceptance reproducible
 *  bit for bit is stated next to each function.
 *
 * Floating point: every accumulation is float64.  The acceptance contract is fp32 + integers by
 * definition (see or_fx_weight) and must be compiled with -ffp-contract=off.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef unsigned __int128 u128;

enum { OK = 0, E_ARG = 1, E_TREE = 2, E_BIG = 3, E_UNSUP = 4, E_NONFINITE = 5, E_NOMEM = 9 };
enum { DT_F32 = 0, DT_BF16 = 1, DT_E4M3 = 2, DT_F64_DECODED = 9 /* internal: caches decoded to float64 */ };

int or_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------------------------------------- */
/* element decoding                                                                                 */
/* ---------------------------------------------------------------------------------------------- */
static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* OCP 8-bit floating point E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite magnitude 448. */
static double e4m3_to_double(uint8_t c) {
    int e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* subnormal: m/8 * 2^(1-7) */
    else        v = ldexp((double)(8 + m), e - 10);  /* (1 + m/8) * 2^(e-7) */
    return (c & 0x80) ? -v : v;
}

static double load_elem(const void* base, size_t i, int dt) {
    switch (dt) {
    case DT_F32:  return (double)((const float*)base)[i];
    case DT_BF16: return (double)bf16_to_float(((const uint16_t*)base)[i]);
    case DT_F64_DECODED: return ((const double*)base)[i];
    default:      return e4m3_to_double(((const uint8_t*)base)[i]);
    }
}

/* float32 view of a logit (f32 or bf16 only) */
static float load_logit(const void* base, size_t i, int dt) {
    return dt == DT_F32 ? ((const float*)base)[i] : bf16_to_float(((const uint16_t*)base)[i]);
}

/* ---------------------------------------------------------------------------------------------- */
/* tree                                                                                             */
/* ---------------------------------------------------------------------------------------------- */
/* A draft tree is a parent array: node 0 is the root (the last committed token, parent -1); every other
 * node names an earlier node as its parent, so parent[i] < i and the array is topologically ordered. */
int or_tree_check(int T, const int32_t* parent) {
    if (T < 1) return E_ARG;
    if (parent[0] != -1) return E_TREE;
    for (int i = 1; i < T; ++i)
        if (parent[i] < 0 || parent[i] >= i) return E_TREE;
    return OK;
}

int or_tree_depth(int T, const int32_t* parent, int32_t* depth) {
    int st = or_tree_check(T, parent);
    if (st) return st;
    for (int i = 0; i < T; ++i) {
        int d = 0;
        for (int a = i; parent[a] >= 0; a = parent[a]) ++d;   /* explicit walk to the root */
        depth[i] = d;
    }
    return OK;
}

/* ---------------------------------------------------------------------------------------------- */
/* tree-masked attention (plain definition, float64)                                               */
/* ---------------------------------------------------------------------------------------------- */
static void attn_row(int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, int kv_dt, const void* q,
                     const void* k, const void* v, const float* k_scale, const float* v_scale, int L,
                     const int32_t* par, double scale, int b, int i, int h, double* o, double* lse_out) {
    int G = Hq / Hkv, hk = h / G;                       /* contiguous GQA groups */
    int on[64];
    memset(on, 0, sizeof on);
    for (int a = i; a >= 0; a = par[a]) on[a] = 1;       /* ancestors of i, itself and the root included */
    double ks = (kv_dt == DT_E4M3) ? (double)k_scale[hk] : 1.0;
    double vs = (kv_dt == DT_E4M3) ? (double)v_scale[hk] : 1.0;
    size_t qoff = (((size_t)b * T + i) * Hq + h) * D;
    size_t kvbase = ((size_t)b * Hkv + hk) * (size_t)kv_cap * D;
    int npos = L + T;
    double* s = (double*)malloc(sizeof(double) * (size_t)npos);
    double m = -INFINITY;
    for (int j = 0; j < npos; ++j) {
        int allowed = j < L || on[j - L];
        if (!allowed) { s[j] = -INFINITY; continue; }
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += load_elem(q, qoff + d, q_dt) * (load_elem(k, kvbase + (size_t)j * D + d, kv_dt) * ks);
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double sum = 0.0;
    double* acc = (double*)calloc((size_t)D, sizeof(double));   /* private accumulator, stored once */
    for (int j = 0; j < npos; ++j) {
        if (s[j] == -INFINITY) continue;
        double w = exp(s[j] - m);
        sum += w;
        for (int d = 0; d < D; ++d) acc[d] += w * (load_elem(v, kvbase + (size_t)j * D + d, kv_dt) * vs);
    }
    for (int d = 0; d < D; ++d) o[d] = acc[d] / sum;
    *lse_out = m + log(sum);
    free(acc);
    free(s);
}

int or_tree_attn(int B, int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, int kv_dt,
                 const void* q, const void* k, const void* v, const float* k_scale, const float* v_scale,
                 const int32_t* kv_len, const int32_t* parent, double sm_scale,
                 const int32_t* rows, int n_rows, double* out, double* lse, int32_t* status) {
    if (B < 0 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || kv_cap < 0) return E_ARG;
    if (T > 64) return E_BIG;
    if (Hq % Hkv) return E_ARG;
    if (q_dt == DT_E4M3 || q_dt < 0 || q_dt > 2 || kv_dt < 0 || kv_dt > 2) return E_UNSUP;
    if (kv_dt == DT_E4M3 && (!k_scale || !v_scale)) return E_ARG;
    double scale = sm_scale != 0.0 ? sm_scale : 1.0 / sqrt((double)D);
    for (int b = 0; b < B; ++b) {
        int st = or_tree_check(T, parent + (size_t)b * T);
        if (!st && (kv_len[b] < 0 || kv_len[b] + T > kv_cap)) st = E_ARG;
        status[b] = st;
    }
    long total = rows ? n_rows : (long)B * T * Hq;
#pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < total; ++r) {
        int b, i, h;
        if (rows) { b = rows[3 * r]; i = rows[3 * r + 1]; h = rows[3 * r + 2]; }
        else { h = (int)(r % Hq); i = (int)((r / Hq) % T); b = (int)(r / ((long)Hq * T)); }
        if (status[b]) continue;
        size_t idx = ((size_t)b * T + i) * Hq + h;
        attn_row(T, Hq, Hkv, D, kv_cap, q_dt, kv_dt, q, k, v, k_scale, v_scale, kv_len[b],
                 parent + (size_t)b * T, scale, b, i, h, out + idx * D, lse + idx);
    }
    return OK;
}

/* ---------------------------------------------------------------------------------------------- */
/* acceptance: the integer contract                                                                 */
/* ---------------------------------------------------------------------------------------------- */
/* Contract (both the oracle and the device implement it from this text):
 *   y_k = fp32(z_k) * invT with invT = (float)(1/(double)temperature);  m = max_k y_k
 *   d = y_k - m;  t = d * log2(e)  (fp32, each op rounded to nearest even)
 *   t < -24  ->  W_k = 0
 *   else n = rint(t), f = t - n,  P(f) = Horner over c7..c0 with fmaf, c_j = fp32((ln 2)^j / j!)
 *        W_k = floor(P(f) * 2^(24 + n))           (so W at the row maximum is exactly 2^24)
 *   S = sum_k W_k (64-bit).  p(k) is read as W_k / S. */
static const float C_LOG2E = 0x1.715476p+0f;
static const float C_P0 = 1.0f;
static const float C_P1 = 0x1.62e430p-1f;
static const float C_P2 = 0x1.ebfbe0p-3f;
static const float C_P3 = 0x1.c6b08ep-5f;
static const float C_P4 = 0x1.3b2ab6p-7f;
static const float C_P5 = 0x1.5d87fep-10f;
static const float C_P6 = 0x1.430912p-13f;
static const float C_P7 = 0x1.ffcbfcp-17f;

float or_fx_exp2(float f) {
    float p = C_P7;
    p = fmaf(p, f, C_P6);
    p = fmaf(p, f, C_P5);
    p = fmaf(p, f, C_P4);
    p = fmaf(p, f, C_P3);
    p = fmaf(p, f, C_P2);
    p = fmaf(p, f, C_P1);
    p = fmaf(p, f, C_P0);
    return p;
}

uint32_t or_fx_weight(float y, float m) {
    float d = y - m;
    float t = d * C_LOG2E;
    if (!(t >= -24.0f)) return 0u;
    float n = rintf(t);
    float f = t - n;
    float w = ldexpf(or_fx_exp2(f), 24 + (int)n);
    return (uint32_t)floorf(w);
}

void or_fx_exp2_batch(const float* f, float* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = or_fx_exp2(f[i]);
}

void or_fx_weight_batch(const float* y, float m, uint32_t* out, long n) {
    for (long i = 0; i < n; ++i) out[i] = or_fx_weight(y[i], m);
}

typedef struct {
    float m;       /* max of y over the row */
    uint64_t S;    /* sum of W */
    int finite;    /* all y finite */
} row_stats;

static row_stats row_fx_stats(const void* logits, size_t row, int V, int dt, float invT) {
    row_stats r;
    r.m = -INFINITY; r.S = 0; r.finite = 1;
    size_t base = row * (size_t)V;
    for (int k = 0; k < V; ++k) {
        float y = load_logit(logits, base + k, dt) * invT;
        if (!isfinite(y)) r.finite = 0;
        if (y > r.m) r.m = y;
    }
    if (!r.finite) return r;
    for (int k = 0; k < V; ++k) r.S += or_fx_weight(load_logit(logits, base + k, dt) * invT, r.m);
    return r;
}

static void row_fx_weights(const void* logits, size_t row, int V, int dt, float invT, float m, uint64_t* w) {
    size_t base = row * (size_t)V;
    for (int k = 0; k < V; ++k) w[k] = or_fx_weight(load_logit(logits, base + k, dt) * invT, m);
}

/* first index of the maximum; -1 if the row holds a non-finite value */
static int row_argmax(const void* logits, size_t row, int V, int dt) {
    size_t base = row * (size_t)V;
    int best = -1;
    float bv = -INFINITY;
    for (int k = 0; k < V; ++k) {
        float z = load_logit(logits, base + k, dt);
        if (!isfinite(z)) return -1;
        if (best < 0 || z > bv) { bv = z; best = k; }
    }
    return best;
}

/* smallest j whose inclusive prefix sum of w exceeds floor(u * R / 2^32), R = sum of w > 0 */
static int sample_index(const uint64_t* w, int V, uint64_t R, uint32_t u) {
    u128 thr = ((u128)u * R) >> 32;
    u128 run = 0;
    for (int j = 0; j < V; ++j) {
        run += w[j];
        if (run > thr) return j;
    }
    return V - 1; /* unreachable when R = sum(w) */
}

int or_accept(int B, int T, int V, int logit_dt, const void* target, const void* draft,
              const int32_t* tokens, const int32_t* parent, float temperature, const uint32_t* uniforms,
              int32_t* accept_len, int32_t* path, int32_t* out_tokens, int32_t* bonus, int32_t* argmax,
              int32_t* status) {
    if (B < 0 || T < 1 || V < 1) return E_ARG;
    if (T > 64) return E_BIG;
    if (logit_dt != DT_F32 && logit_dt != DT_BF16) return E_UNSUP;
    if (!(temperature >= 0.0f) || isinf(temperature)) return E_ARG;
    int greedy = temperature == 0.0f;
    if (!greedy && !uniforms) return E_ARG;
    float invT = greedy ? 1.0f : (float)(1.0 / (double)temperature);

    /* argmax of every target row, independent of the walk */
    if (argmax) {
#pragma omp parallel for schedule(dynamic, 8)
        for (long r = 0; r < (long)B * T; ++r) argmax[r] = row_argmax(target, (size_t)r, V, logit_dt);
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int32_t* par = parent + (size_t)b * T;
        const int32_t* tok = tokens + (size_t)b * T;
        int32_t* pth = path + (size_t)b * T;
        int32_t* otk = out_tokens + (size_t)b * T;
        for (int j = 0; j < T; ++j) { pth[j] = -1; otk[j] = -1; }
        accept_len[b] = -1;
        bonus[b] = -1;
        int st = or_tree_check(T, par);
        for (int c = 1; !st && c < T; ++c)
            if (tok[c] < 0 || tok[c] >= V) st = E_ARG;
        if (!st) {   /* every row of the request is scanned on the device, so all must be finite */
            for (int r = 0; r < T && !st; ++r) {
                size_t row = (size_t)b * T + r;
                if (greedy) {
                    if (row_argmax(target, row, V, logit_dt) < 0) st = E_NONFINITE;
                } else {
                    if (!row_fx_stats(target, row, V, logit_dt, invT).finite) st = E_NONFINITE;
                    if (draft && !row_fx_stats(draft, row, V, logit_dt, invT).finite) st = E_NONFINITE;
                }
            }
        }
        if (status) status[b] = st;
        if (st) continue;

        int n = 0, cur = 0;
        if (greedy) {
            /* greedy: descend to the first child (ascending node id) whose token is the target argmax */
            for (;;) {
                int am = row_argmax(target, (size_t)b * T + cur, V, logit_dt);
                int next = -1;
                for (int c = cur + 1; c < T; ++c)
                    if (par[c] == cur && tok[c] == am) { next = c; break; }
                if (next < 0) { bonus[b] = am; break; }
                pth[n++] = next;
                cur = next;
            }
        } else {
            uint64_t* wres = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
            uint64_t* wq = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)V);
            for (;;) {
                size_t row = (size_t)b * T + cur;
                row_stats ps = row_fx_stats(target, row, V, logit_dt, invT);
                int has_child = 0;
                for (int c = cur + 1; c < T; ++c) if (par[c] == cur) { has_child = 1; break; }
                row_fx_weights(target, row, V, logit_dt, invT, ps.m, wres);
                uint64_t Sres = ps.S;
                if (!has_child) {
                    bonus[b] = sample_index(wres, V, Sres, uniforms[(size_t)b * T]);
                    break;
                }
                uint64_t Sq = 1;
                if (draft) {
                    row_stats qs = row_fx_stats(draft, row, V, logit_dt, invT);
                    row_fx_weights(draft, row, V, logit_dt, invT, qs.m, wq);
                    Sq = qs.S;
                }
                int next = -1;
                for (int c = cur + 1; c < T; ++c) {
                    if (par[c] != cur) continue;
                    int x = tok[c];
                    uint64_t wqx = draft ? wq[x] : 1u;   /* one-hot proposal: q = delta_x, Sq = 1 */
                    u128 lhs = (u128)uniforms[(size_t)b * T + c] * wqx * Sres;
                    u128 rhs = ((u128)wres[x] * Sq) << 32;
                    if (lhs < rhs) { next = c; break; }
                    /* rejected: p' <- floor(max(0, p'*Sq - q*S') / Sq), taken per token */
                    uint64_t S2 = 0;
                    for (int kk = 0; kk < V; ++kk) {
                        uint64_t qk = draft ? wq[kk] : (uint64_t)(kk == x);
                        u128 a = (u128)wres[kk] * Sq, s = (u128)qk * Sres;
                        wres[kk] = a > s ? (uint64_t)((a - s) / Sq) : 0u;
                        S2 += wres[kk];
                    }
                    Sres = S2;
                }
                if (next >= 0) { pth[n++] = next; cur = next; continue; }
                if (Sres == 0) {   /* residual vanished: fall back to the target row itself */
                    row_fx_weights(target, row, V, logit_dt, invT, ps.m, wres);
                    Sres = ps.S;
                }
                bonus[b] = sample_index(wres, V, Sres, uniforms[(size_t)b * T]);
                break;
            }
            free(wres);
            free(wq);
        }
        accept_len[b] = n;
        for (int j = 0; j < n; ++j) otk[j] = tok[pth[j]];
        otk[n] = bonus[b];
    }
    return OK;
}

/* ---------------------------------------------------------------------------------------------- */
/* training loss                                                                                    */
/* ---------------------------------------------------------------------------------------------- */
/* log(1 - e^{-a}) for a > 0, in the two-branch form that keeps full relative accuracy
 * (log(-expm1(-a)) up to ln 2, log1p(-e^{-a}) beyond). */
static double log1mexp(double a) {
    return a <= M_LN2 ? log(-expm1(-a)) : log1p(-exp(-a));
}

static int loss_core(int N, int T, int V, const void* logits, int is_bf16, const int32_t* tokens,
                     const int32_t* parent, const int32_t* labels, double* row_loss, double* row_acc,
                     double* row_rej, double* sums, double* grad, int32_t* status) {
    if (N < 0 || T < 1 || V < 2) return E_ARG;
    if (T > 64) return E_BIG;
    double n_terms = (double)N * (double)(T - 1);
    double inv_n = n_terms > 0 ? 1.0 / n_terms : 0.0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int n = 0; n < N; ++n) {
        const int32_t* par = parent + (size_t)n * T;
        const int32_t* tok = tokens + (size_t)n * T;
        const int32_t* lab = labels + (size_t)n * T;
        int st = or_tree_check(T, par);
        for (int c = 1; !st && c < T; ++c)
            if (tok[c] < 0 || tok[c] >= V || lab[par[c]] < 0 || lab[par[c]] >= V) st = E_ARG;
        double* z = (double*)malloc(sizeof(double) * (size_t)V);
        for (int p = 0; p < T; ++p) {
            size_t row = (size_t)n * T + p;
            row_loss[row] = row_acc[row] = row_rej[row] = 0.0;
            int nch = 0;
            for (int c = p + 1; c < T && !st; ++c) if (par[c] == p) ++nch;
            if (st || nch == 0) {
                if (grad) memset(grad + row * V, 0, sizeof(double) * (size_t)V);
                continue;
            }
            for (int k = 0; k < V; ++k)
                z[k] = is_bf16 ? (double)bf16_to_float(((const uint16_t*)logits)[row * V + k])
                               : ((const double*)logits)[row * V + k];
            double m = -INFINITY;
            for (int k = 0; k < V; ++k) if (z[k] > m) m = z[k];
            double s = 0.0;
            for (int k = 0; k < V; ++k) s += exp(z[k] - m);
            double lse = m + log(s);
            double A = 0.0, C = 0.0, acc = 0.0, rej = 0.0;
            for (int c = p + 1; c < T; ++c) {
                if (par[c] != p) continue;
                int x = tok[c];
                if (x == lab[p]) {          /* accepted: cross-entropy -log q(x) */
                    A += 1.0;
                    acc += lse - z[x];
                } else {                    /* rejected: -log(1 - q(x)), q clamped to <= 1 - 1e-6 */
                    double a = lse - z[x];
                    if (a < 1e-6) a = 1e-6;
                    rej += -log1mexp(a);
                    C += 1.0 / expm1(a);    /* q/(1-q) */
                }
            }
            row_acc[row] = acc;
            row_rej[row] = rej;
            row_loss[row] = acc + rej;
            if (grad) {
                double* g = grad + row * V;
                for (int k = 0; k < V; ++k) g[k] = exp(z[k] - lse) * (A - C);
                g[lab[p]] -= A;
                for (int c = p + 1; c < T; ++c) {
                    if (par[c] != p || tok[c] == lab[p]) continue;
                    double a = lse - z[tok[c]];
                    if (a < 1e-6) a = 1e-6;
                    g[tok[c]] += 1.0 / expm1(a);
                }
                for (int k = 0; k < V; ++k) g[k] *= inv_n;
            }
        }
        free(z);
        if (status) status[n] = st;
    }
    double sa = 0.0, sr = 0.0;
    for (long r = 0; r < (long)N * T; ++r) { sa += row_acc[r]; sr += row_rej[r]; }
    sums[0] = sa;
    sums[1] = sr;
    sums[2] = n_terms;
    return OK;
}

int or_loss_f64(int N, int T, int V, const double* logits, const int32_t* tokens, const int32_t* parent,
                const int32_t* labels, double* row_loss, double* row_acc, double* row_rej, double* sums,
                double* grad, int32_t* status) {
    return loss_core(N, T, V, logits, 0, tokens, parent, labels, row_loss, row_acc, row_rej, sums, grad,
                     status);
}

int or_loss(int N, int T, int V, const uint16_t* logits_bf16, const int32_t* tokens, const int32_t* parent,
            const int32_t* labels, double* row_loss, double* row_acc, double* row_rej, double* sums,
            double* grad, int32_t* status) {
    return loss_core(N, T, V, logits_bf16, 1, tokens, parent, labels, row_loss, row_acc, row_rej, sums,
                     grad, status);
}

/* ---------------------------------------------------------------------------------------------- */
/* KV compaction after acceptance (plain definition)                                                */
/* ---------------------------------------------------------------------------------------------- */
/* After verification the request's committed tokens are the root plus the accepted path.  The root's K/V
 * already sit at cache position L (the first tree slot) and the accepted node path[j] sits at L + path[j];
 * compaction makes the committed tokens contiguous, so position L + 1 + j receives what was at
 * L + path[j] ("Aurora" post, section 2: verification keeps the accepted continuation; TIDE overview:
 * the target keeps the accepted draft tokens).  The new prefix length is L + 1 + accept_len; positions
 * past it keep whatever they held.  This is the out-of-place definition: every read sees the cache as it
 * was before the call.  A request whose accept_len is negative (a failed verification) or whose path is
 * not a root path of its tree is left untouched (new length = old length) with a status code. */
int or_kv_compact(int B, int T, int Hkv, int D, int kv_cap, int kv_dt, void* k_cache, void* v_cache,
                  const int32_t* kv_len, const int32_t* parent, const int32_t* accept_len, const int32_t* path,
                  int32_t* new_kv_len, int32_t* status) {
    if (B < 0 || T < 1 || Hkv < 1 || D < 1 || kv_cap < T) return E_ARG;
    if (T > 64) return E_BIG;
    if (kv_dt != DT_F32 && kv_dt != DT_BF16 && kv_dt != DT_E4M3) return E_UNSUP;
    size_t esz = kv_dt == DT_F32 ? 4 : kv_dt == DT_BF16 ? 2 : 1;
    size_t row = (size_t)D * esz;
    unsigned char* old = (unsigned char*)malloc(row * (size_t)T);
    for (int b = 0; b < B; ++b) {
        const int32_t* par = parent + (size_t)b * T;
        const int32_t* pth = path + (size_t)b * T;
        int L = kv_len[b], n = accept_len[b];
        int st = or_tree_check(T, par);
        if (!st && (L < 0 || (long)L + T > kv_cap)) st = E_ARG;
        if (!st && (n < 0 || n > T - 1)) st = E_ARG;
        /* the path must walk down the tree from the root: path[0] a child of 0, path[j] a child of path[j-1] */
        for (int j = 0; !st && j < n; ++j) {
            int node = pth[j], up = j == 0 ? 0 : pth[j - 1];
            if (node < 1 || node >= T || par[node] != up) st = E_ARG;
        }
        status[b] = st;
        new_kv_len[b] = st ? L : L + 1 + n;
        if (st) continue;
        for (int h = 0; h < Hkv; ++h) {
            for (int c = 0; c < 2; ++c) {
                unsigned char* cache = (unsigned char*)(c == 0 ? k_cache : v_cache);
                unsigned char* base = cache + (((size_t)b * Hkv + h) * (size_t)kv_cap + (size_t)L) * row;
                memcpy(old, base, row * (size_t)T);             /* the tree block as it was */
                for (int j = 0; j < n; ++j) memcpy(base + (size_t)(1 + j) * row, old + (size_t)pth[j] * row, row);
            }
        }
    }
    free(old);
    return OK;
}

/* ---------------------------------------------------------------------------------------------- */
/* Draft tree expansion, one level (plain definition, float64)                                      */
/* ---------------------------------------------------------------------------------------------- */
/* The draft proposes the next level of its tree from the logits of the current frontier ("Aurora" post,
 * section 2, and the TIDE overview: the draft proposes tokens that the target then verifies in one pass).
 * Row s of a request is the draft's next-token logits after frontier node s, whose path score (the sum of
 * the draft's log-probabilities along the path from the root) is front_score[s].  Each row proposes its
 * k most likely tokens (largest logit first, lower token id first on equal logits), with log-probability
 * z - logsumexp(row) at temperature 1.  A candidate's score is its parent's score plus its log-probability;
 * the n_keep best candidates of the request survive (higher score first, then lower frontier slot, then
 * lower rank), and they are listed in (frontier slot, rank) order, the breadth-first numbering of the next
 * level.  Outputs per request: topk_token / topk_logprob [n_front, k], child_parent (frontier slot) /
 * child_token / child_score [n_keep].  A request with a non-finite logit or score gets status 5 and -1 /
 * -inf outputs. */
typedef struct { double score; int slot, rank; } or_cand;

static int cand_cmp(const void* a, const void* b) {
    const or_cand* x = (const or_cand*)a;
    const or_cand* y = (const or_cand*)b;
    if (x->score != y->score) return x->score > y->score ? -1 : 1;
    if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;
    return x->rank < y->rank ? -1 : (x->rank > y->rank);
}

static int cand_bfs_cmp(const void* a, const void* b) {
    const or_cand* x = (const or_cand*)a;
    const or_cand* y = (const or_cand*)b;
    if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;
    return x->rank < y->rank ? -1 : (x->rank > y->rank);
}

int or_tree_expand(int B, int n_front, int V, int k, int n_keep, int logit_dt, const void* logits,
                   const float* front_score, int32_t* topk_token, double* topk_logprob, int32_t* child_parent,
                   int32_t* child_token, double* child_score, int32_t* status) {
    if (B < 0 || n_front < 1 || V < 1 || k < 1 || k > V || n_keep < 0 || n_keep > n_front * k) return E_ARG;
    if (logit_dt != DT_F32 && logit_dt != DT_BF16) return E_UNSUP;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        int st = OK;
        or_cand* cand = (or_cand*)malloc(sizeof(or_cand) * (size_t)n_front * k);
        char* taken = (char*)malloc((size_t)V);
        for (int s = 0; s < n_front && !st; ++s) {
            size_t r = (size_t)b * n_front + s;
            if (!isfinite(front_score[r])) { st = E_NONFINITE; break; }
            double m = -INFINITY;
            for (int j = 0; j < V; ++j) {
                float z = load_logit(logits, r * V + j, logit_dt);
                if (!isfinite(z)) { st = E_NONFINITE; break; }
                if (z > m) m = z;
            }
            if (st) break;
            double sum = 0.0;
            for (int j = 0; j < V; ++j) sum += exp((double)load_logit(logits, r * V + j, logit_dt) - m);
            double lse = m + log(sum);
            /* k rounds of "largest remaining logit, lowest id on ties" */
            memset(taken, 0, (size_t)V);
            for (int q = 0; q < k; ++q) {
                int best = -1;
                float bz = 0.f;
                for (int j = 0; j < V; ++j) {
                    if (taken[j]) continue;
                    float z = load_logit(logits, r * V + j, logit_dt);
                    if (best < 0 || z > bz) { best = j; bz = z; }
                }
                taken[best] = 1;
                topk_token[r * k + q] = best;
                topk_logprob[r * k + q] = (double)bz - lse;
                cand[s * k + q].score = (double)front_score[r] + ((double)bz - lse);
                cand[s * k + q].slot = s;
                cand[s * k + q].rank = q;
            }
        }
        if (st) {
            for (int i = 0; i < n_front * k; ++i) {
                topk_token[(size_t)b * n_front * k + i] = -1;
                topk_logprob[(size_t)b * n_front * k + i] = -INFINITY;
            }
            for (int i = 0; i < n_keep; ++i) {
                child_parent[(size_t)b * n_keep + i] = -1;
                child_token[(size_t)b * n_keep + i] = -1;
                child_score[(size_t)b * n_keep + i] = -INFINITY;
            }
        } else {
            qsort(cand, (size_t)n_front * k, sizeof(or_cand), cand_cmp);   /* best first */
            qsort(cand, (size_t)n_keep, sizeof(or_cand), cand_bfs_cmp);    /* survivors in BFS order */
            for (int i = 0; i < n_keep; ++i) {
                size_t r = (size_t)b * n_front + cand[i].slot;
                child_parent[(size_t)b * n_keep + i] = cand[i].slot;
                child_token[(size_t)b * n_keep + i] = topk_token[r * k + cand[i].rank];
                child_score[(size_t)b * n_keep + i] = cand[i].score;
            }
        }
        status[b] = st;
        free(cand);
        free(taken);
    }
    return OK;
}

/* ---------------------------------------------------------------------------------------------- */
/* tree-masked attention backward (plain definition, float64)                                      */
/* ---------------------------------------------------------------------------------------------- */
/* The draft is trained on every accepted and rejected branch of its trees in one batched forward and
 * backward pass ("Aurora" post, section 2), so the attention of that pass needs its gradient under the
 * same tree mask.  With p = softmax(s), s_j = scale * <q, k_j> over the allowed set A(b, i) of the forward
 * (prefix plus the node's ancestors), o = sum_j p_j v_j and an upstream gradient dO = d loss / d o:
 *     dv_j += p_j dO                      dp_j = <dO, v_j>        delta = <dO, o> = sum_j p_j dp_j
 *     ds_j  = p_j (dp_j - delta)          dq    = scale * sum_j ds_j k_j
 *     dk_j += scale * ds_j q
 * summed over every (node, query head) whose allowed set holds position j.  This is the chain rule of the
 * softmax written out; the forward (p, o) is recomputed here in float64 from q, k, v.  dq is [B,T,Hq,D];
 * dk and dv are [B,Hkv,kv_cap,D] with every position outside [0, kv_len + T) left at zero.  E4M3 caches
 * are not taken (the backward trains a draft whose cache is bf16 or fp32). */
static void attn_row_bwd(int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, int kv_dt, const void* q,
                         const void* k, const void* v, const void* dout, int L, const int32_t* par,
                         double scale, int b, int i, int h, double* dq, double* dk, double* dv) {
    const int G = Hq / Hkv;
    const int hk = h / G;                               /* contiguous GQA groups, as in the forward */
    int on[64];
    memset(on, 0, sizeof on);
    for (int x = i; x >= 0; x = par[x]) on[x] = 1;   /* the node, its ancestors and the root */
    size_t qoff = (((size_t)b * T + i) * Hq + h) * D;
    size_t kvbase = ((size_t)b * Hkv + hk) * (size_t)kv_cap * D;
    int npos = L + T;
    double* s = (double*)malloc(sizeof(double) * (size_t)npos);
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    double* g = (double*)malloc(sizeof(double) * (size_t)D);
    double* o = (double*)calloc((size_t)D, sizeof(double));
    for (int d = 0; d < D; ++d) { qv[d] = load_elem(q, qoff + d, q_dt); g[d] = load_elem(dout, qoff + d, q_dt); }
    double m = -INFINITY;
    for (int j = 0; j < npos; ++j) {
        if (!(j < L || on[j - L])) { s[j] = -INFINITY; continue; }
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qv[d] * load_elem(k, kvbase + (size_t)j * D + d, kv_dt);
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    double sum = 0.0;
    for (int j = 0; j < npos; ++j) if (s[j] != -INFINITY) sum += exp(s[j] - m);
    for (int j = 0; j < npos; ++j) {                     /* s becomes p */
        s[j] = s[j] == -INFINITY ? 0.0 : exp(s[j] - m) / sum;
        if (s[j] == 0.0) continue;
        for (int d = 0; d < D; ++d) o[d] += s[j] * load_elem(v, kvbase + (size_t)j * D + d, kv_dt);
    }
    double delta = 0.0;
    for (int d = 0; d < D; ++d) delta += g[d] * o[d];
    for (int d = 0; d < D; ++d) dq[d] = 0.0;
    for (int j = 0; j < npos; ++j) {
        if (!(j < L || on[j - L])) continue;
        double p = s[j], dp = 0.0;
        for (int d = 0; d < D; ++d) dp += g[d] * load_elem(v, kvbase + (size_t)j * D + d, kv_dt);
        double ds = p * (dp - delta);
        size_t row = ((size_t)b * Hkv + hk) * (size_t)kv_cap + (size_t)j;
        for (int d = 0; d < D; ++d) {
            dq[d] += scale * ds * load_elem(k, kvbase + (size_t)j * D + d, kv_dt);
            dk[row * D + d] += scale * ds * qv[d];
            dv[row * D + d] += p * g[d];
        }
    }
    free(o); free(g); free(qv); free(s);
}

int or_tree_attn_bwd(int B, int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, int kv_dt, const void* q,
                     const void* k, const void* v, const int32_t* kv_len, const int32_t* parent, double sm_scale,
                     const void* dout, double* dq, double* dk, double* dv, int32_t* status) {
    if (B < 0 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || kv_cap < 0) return E_ARG;
    if (T > 64) return E_BIG;
    if (Hq % Hkv) return E_ARG;
    if (q_dt == DT_E4M3 || q_dt < 0 || q_dt > 2 || kv_dt < 0 || kv_dt > 1) return E_UNSUP;
    double scale = sm_scale != 0.0 ? sm_scale : 1.0 / sqrt((double)D);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * kv_cap * D);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * kv_cap * D);
    for (int b = 0; b < B; ++b) {
        int st = or_tree_check(T, parent + (size_t)b * T);
        if (!st && (kv_len[b] < 0 || kv_len[b] + T > kv_cap)) st = E_ARG;
        status[b] = st;
    }
    /* one thread per request: dk / dv of different requests never overlap */
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < T; ++i)
            for (int h = 0; h < Hq; ++h) {
                double* dqr = dq + (((size_t)b * T + i) * Hq + h) * D;
                if (status[b]) { for (int d = 0; d < D; ++d) dqr[d] = 0.0; continue; }
                attn_row_bwd(T, Hq, Hkv, D, kv_cap, q_dt, kv_dt, q, k, v, dout, kv_len[b], parent + (size_t)b * T,
                             scale, b, i, h, dqr, dk, dv);
            }
    }
    return OK;
}


/* ---------------------------------------------------------------------------------------------- */
/* FP4 (e2m1) KV caches                                                                             */
/* ---------------------------------------------------------------------------------------------- */
/* OCP 4-bit floating point E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no infinities or NaN:
 * magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.  A cache element is code * block scale * head scale, with one
 * E4M3 block scale per 16 consecutive elements of a row (the NVFP4 layout) and the fp32 per-kv-head scale of
 * the E4M3 caches.  Codes are packed two per byte, the even element in the low nibble. */
static double e2m1_to_double(unsigned c) {
    int e = (c >> 1) & 3, m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (c & 8) ? -v : v;
}

/* Tree attention over FP4 caches: k / v codes [B, Hkv, kv_cap, D/2] bytes, block scales [B, Hkv, kv_cap,
 * D/16] E4M3 codes, head scales [Hkv] fp32.  Each request's caches are decoded to float64 (one request at a
 * time, so memory stays at one request's worth) and the plain definition above runs on them.  rows, if
 * given, lists the (b, i, h) triples to compute (n_rows of them, grouped by b in any order); other outputs
 * are left untouched.  D must be a multiple of 16.  Returns E_NOMEM if the decode buffers cannot be had. */
int or_tree_attn_e2m1(int B, int T, int Hq, int Hkv, int D, int kv_cap, int q_dt, const void* q,
                      const uint8_t* k, const uint8_t* v, const uint8_t* k_block, const uint8_t* v_block,
                      const float* k_scale, const float* v_scale, const int32_t* kv_len, const int32_t* parent,
                      double sm_scale, const int32_t* rows, int n_rows, double* out, double* lse, int32_t* status) {
    if (B < 0 || T < 1 || Hq < 1 || Hkv < 1 || D < 16 || D % 16 || kv_cap < 0) return E_ARG;
    if (T > 64) return E_BIG;
    if (Hq % Hkv) return E_ARG;
    if (q_dt != DT_F32 && q_dt != DT_BF16) return E_UNSUP;
    double scale = sm_scale != 0.0 ? sm_scale : 1.0 / sqrt((double)D);
    for (int b = 0; b < B; ++b) {
        int st = or_tree_check(T, parent + (size_t)b * T);
        if (!st && (kv_len[b] < 0 || kv_len[b] + T > kv_cap)) st = E_ARG;
        status[b] = st;
    }
    size_t n = (size_t)Hkv * kv_cap * D;                 /* one request's elements per cache */
    double* kd = (double*)malloc(sizeof(double) * (n ? n : 1));
    double* vd = (double*)malloc(sizeof(double) * (n ? n : 1));
    if (!kd || !vd) {
        free(kd);
        free(vd);
        return E_NOMEM;
    }
    size_t qsz = q_dt == DT_F32 ? 4 : 2;
    for (int b = 0; b < B; ++b) {
        if (status[b]) continue;
        int wanted = rows == NULL;
        for (int r = 0; r < n_rows && !wanted; ++r) wanted = rows[3 * r] == b;
        if (!wanted) continue;
        size_t base = (size_t)b * n;
        for (size_t i = 0; i < n; ++i) {
            size_t row = i / (size_t)D;                  /* (kv head, position) row inside the request */
            int h = (int)(row / (size_t)kv_cap);
            size_t blk = (base + i) / 16;                /* 16 consecutive elements of a row share a scale */
            unsigned kc = (k[(base + i) / 2] >> (4 * (i & 1))) & 15, vc = (v[(base + i) / 2] >> (4 * (i & 1))) & 15;
            kd[i] = e2m1_to_double(kc) * e4m3_to_double(k_block[blk]) * (double)k_scale[h];
            vd[i] = e2m1_to_double(vc) * e4m3_to_double(v_block[blk]) * (double)v_scale[h];
        }
        const void* qb = (const char*)q + (size_t)b * T * Hq * D * qsz;
        long total = (long)T * Hq;
#pragma omp parallel for schedule(dynamic, 4)
        for (long r = 0; r < total; ++r) {
            int h = (int)(r % Hq), i = (int)(r / Hq);
            if (rows) {
                int hit = 0;
                for (int x = 0; x < n_rows && !hit; ++x) hit = rows[3 * x] == b && rows[3 * x + 1] == i && rows[3 * x + 2] == h;
                if (!hit) continue;
            }
            size_t idx = ((size_t)b * T + i) * Hq + h;
            attn_row(T, Hq, Hkv, D, kv_cap, q_dt, DT_F64_DECODED, qb, kd, vd, NULL, NULL, kv_len[b],
                     parent + (size_t)b * T, scale, 0, i, h, out + idx * D, lse + idx);
        }
    }
    free(kd);
    free(vd);
    return OK;
}
