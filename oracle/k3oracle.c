/*
 * k3oracle.c -- CPU ORACLE for the Kimi-K3-style MXFP4 MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg may load this library. The CUDA library never links,
 * includes or calls it, and it shares no code with the CUDA path.
 *
 * Plain, slow, obviously correct: every quantity is computed in IEEE double by
 * plain sequential loops, in the order the method states it. Sources, cited by
 * page title and section:
 *  - "kimi-k3-in-c" review (blog.123qwe.co.kr, "한눈에 보는 kimi-k3-in-c" table and
 *    "KDA·MLA·MoE" table): 896 routed experts per MoE layer, top-16, 2 shared
 *    experts; routed experts stored as MXFP4 and multiplied directly from the
 *    nibbles ("디퀀트 없이 니블 직접 곱"), 17,547,264 B per expert.
 *  - kimi-k3-in-c README (rosettalens.com, "shard census"): 33,030,144 params
 *    per expert at 0.53125 B/weight = 0.5 B per nibble + 1/32 B for the shared
 *    E8M0 scale.
 *  - OCP Microscaling Formats (MX) v1.0: E2M1 element values and E8M0 scale
 *    2^(b-127), b = 0xFF is NaN.
 *  - Router, score 0 (softmax): softmax over the E expert logits, top-k, gates
 *    renormalised over the k selected (the routing bias, if any, is added to the
 *    logits). Score 1 (sigmoid + bias): the review's list of public-header
 *    invariants states that the routing bias skews only the selection and that
 *    the combine weights come from the unbiased sigmoid score: s_e =
 *    sigmoid(x . W_e), selection by s_e + b_e, gates s_e / sum over the k of s.
 *  - Expert FFN: h = SiLU(W_gate x) * (W_up x), o = W_down h (SiLU-gated GLU,
 *    the stand-in for the pages' unspecified "SiTU-GLU").
 *  - Combine: y = sum_i w_i o_i + sum_s o_s (shared experts weight 1).
 *  - Shared experts in bf16 (a variant): the kimi-k3-in-c README's parameter
 *    budget (after the shard census) counts every non-routed parameter in
 *    bfloat16. A bf16 shared record is [gate f x d][up f x d][down d x f] bf16,
 *    row-major; its weights are the exact values of the bf16 bit patterns and
 *    the FFN is the same.
 *
 * Readings where the pages are silent (layout of a record, block axis, nibble
 * order, tie order): blocks of 32 run along the reduction axis; the even
 * element is the low nibble; a record is gate, up, down, each codes then
 * scales; equal logits put the lower expert index first.
 *
 * Parity: pinned by tests/test_oracle.py (OCP table, byte counts printed by
 * the pages, brute force, closed forms and invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Test hook: deliberately wrong variants, so tests can show the pins catch them. */
static int g_fault = 0;
void k3o_set_fault(int f) { g_fault = f; }
enum {
    FAULT_NONE = 0,
    FAULT_NIBBLE_ORDER = 1,  /* even element read from the high nibble          */
    FAULT_SCALE_BIAS = 2,    /* E8M0 decoded as 2^(b-126)                        */
    FAULT_DROP_SHARED = 3,   /* shared experts left out of the combine           */
    FAULT_NO_RENORM = 4,     /* gate = full-softmax probability, not renormalised */
    FAULT_TIE_HIGH = 5,      /* equal logits -> higher index first               */
    FAULT_DOWN_T = 6,        /* down projection read transposed                  */
    FAULT_GLU_ON_UP = 7,     /* SiLU applied to the up branch instead of the gate */
    FAULT_BIAS_IN_GATE = 8,  /* sigmoid score: gates from the biased score          */
    FAULT_NO_BIAS_SELECT = 9,/* sigmoid score: selection ignores the bias           */
    FAULT_SILU_SIGN = 10,    /* SiLU(z) as z / (1 + e^z)                            */
    FAULT_E2M1_TABLE = 11,   /* one wrong table entry: code 5 read as 2.5           */
    FAULT_SHARED_GATED = 12, /* shared experts weighted by the first gate, not 1    */
    FAULT_SELECT_LOWEST = 13,/* the k lowest logits selected                        */
    FAULT_RENORM_SHORT = 14, /* renormalising sum over k - 1 of the k gates         */
    FAULT_RMS_SUM = 15,      /* RMSNorm over the sum of squares, not their mean     */
    FAULT_SCALE_BLOCK = 16,  /* weight scaled by the next block's scale byte        */
};

/* OCP MX v1.0, FP4 E2M1: magnitudes of the 8 positive codes. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double k3o_e2m1(int code) {
    double v = E2M1_MAG[code & 7];
    if (g_fault == FAULT_E2M1_TABLE && (code & 7) == 5) v = 2.5;
    return (code & 8) ? -v : v; /* code 8 is -0.0 */
}

/* E8M0 scale: 2^(b-127); returns -1 for the NaN encoding 0xFF. */
int k3o_e8m0(int b, double* out) {
    if (b < 0 || b > 255) return -1;
    if (b == 255) return -1;
    *out = ldexp(1.0, b - (g_fault == FAULT_SCALE_BIAS ? 126 : 127));
    return 0;
}

/* Bytes of one expert record: three d x f MXFP4 matrices at 0.53125 B/weight. */
int64_t k3o_record_bytes(int64_t d, int64_t f) { return 3 * (d * f / 2 + d * f / 32); }

/* Weight (r, c) of a rows x cols MXFP4 matrix: codes[rows][cols/2], scales[rows][cols/32]. */
static int weight(const uint8_t* codes, const uint8_t* scales, int64_t cols, int64_t r, int64_t c,
                  double* w) {
    uint8_t byte = codes[r * (cols / 2) + c / 2];
    int even_low = (g_fault == FAULT_NIBBLE_ORDER) ? 0 : 1;
    int nib = ((c % 2 == 0) == even_low) ? (byte & 0xF) : (byte >> 4);
    double s;
    int64_t blk = c / 32;
    if (g_fault == FAULT_SCALE_BLOCK) blk = (blk + 1) % (cols / 32);
    if (k3o_e8m0(scales[r * (cols / 32) + blk], &s)) return -1;
    *w = k3o_e2m1(nib) * s;
    return 0;
}

/* Dense dequantisation of a whole matrix into out[rows][cols] (used by the pins). */
int k3o_decode_matrix(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                      double* out) {
    if (cols % 32) return -1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            if (weight(codes, scales, cols, r, c, &out[r * cols + c])) return -1;
    return 0;
}

/* bf16 bit pattern -> exact double. */
double k3o_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------ router */
typedef struct {
    double l;
    int32_t e;
} scored;

static int cmp_desc(const void* a, const void* b) {
    const scored* x = (const scored*)a;
    const scored* y = (const scored*)b;
    const int lowest = g_fault == FAULT_SELECT_LOWEST;
    if (x->l > y->l) return lowest ? 1 : -1;
    if (x->l < y->l) return lowest ? -1 : 1;
    if (g_fault == FAULT_TIE_HIGH) return (x->e > y->e) ? -1 : (x->e < y->e);
    return (x->e < y->e) ? -1 : (x->e > y->e); /* equal logits: lower index first */
}

/*
 * Route one token. x[d] (exact input values), W[E][d] fp32, bias[E] or NULL.
 * logits_out[E] (may be NULL), idx_out[k], w_out[k].
 * score 0 (softmax): logits l_e = sum_j x_j W_ej (+ b_e); full softmax over E;
 * top-k by logit (a full sort, ties to the lower index); gates renormalised
 * over the k. score 1 (sigmoid + bias): logits l_e = sum_j x_j W_ej (no bias);
 * s_e = 1 / (1 + exp(-l_e)); top-k by s_e + b_e (a full sort, ties to the lower
 * index); gates s_e / sum over the k of s.
 */
static int route_sigmoid(int32_t E, int32_t d, int32_t k, const double* x, const float* W, const float* bias,
                         double* logits_out, int32_t* idx_out, double* w_out) {
    scored* s = (scored*)malloc(sizeof(scored) * (size_t)E);
    double* sg = (double*)malloc(sizeof(double) * (size_t)E);
    if (!s || !sg) { free(s); free(sg); return -2; }
    for (int32_t e = 0; e < E; ++e) {
        double l = 0.0;
        for (int32_t j = 0; j < d; ++j) l += x[j] * (double)W[(int64_t)e * d + j];
        if (logits_out) logits_out[e] = l;
        sg[e] = 1.0 / (1.0 + exp(-l));
        s[e].l = sg[e] + ((bias && g_fault != FAULT_NO_BIAS_SELECT) ? (double)bias[e] : 0.0);
        s[e].e = e;
    }
    qsort(s, (size_t)E, sizeof(scored), cmp_desc);
    double zk = 0.0;
    for (int32_t i = 0; i < k; ++i) zk += (g_fault == FAULT_BIAS_IN_GATE) ? s[i].l : sg[s[i].e];
    for (int32_t i = 0; i < k; ++i) {
        idx_out[i] = s[i].e;
        w_out[i] = ((g_fault == FAULT_BIAS_IN_GATE) ? s[i].l : sg[s[i].e]) / zk;
    }
    free(s);
    free(sg);
    return 0;
}

int k3o_route_token(int32_t E, int32_t d, int32_t k, const double* x, const float* W,
                    const float* bias, double* logits_out, int32_t* idx_out, double* w_out, int32_t score) {
    if (k < 1 || k > E) return -1;
    if (score == 1) return route_sigmoid(E, d, k, x, W, bias, logits_out, idx_out, w_out);
    if (score != 0) return -1;
    scored* s = (scored*)malloc(sizeof(scored) * (size_t)E);
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    if (!s || !p) { free(s); free(p); return -2; }
    double lmax = -INFINITY;
    for (int32_t e = 0; e < E; ++e) {
        double l = 0.0;
        for (int32_t j = 0; j < d; ++j) l += x[j] * (double)W[(int64_t)e * d + j];
        if (bias) l += (double)bias[e];
        s[e].l = l;
        s[e].e = e;
        if (logits_out) logits_out[e] = l;
        if (l > lmax) lmax = l;
    }
    double z = 0.0;
    for (int32_t e = 0; e < E; ++e) { p[e] = exp(s[e].l - lmax); z += p[e]; }
    for (int32_t e = 0; e < E; ++e) p[e] /= z;
    qsort(s, (size_t)E, sizeof(scored), cmp_desc);
    double zk = 0.0;
    for (int32_t i = 0; i < k - (g_fault == FAULT_RENORM_SHORT ? 1 : 0); ++i) zk += p[s[i].e];
    for (int32_t i = 0; i < k; ++i) {
        idx_out[i] = s[i].e;
        w_out[i] = (g_fault == FAULT_NO_RENORM) ? p[s[i].e] : p[s[i].e] / zk;
    }
    free(s);
    free(p);
    return 0;
}

/*
 * Route T tokens (the per-token routine above, tokens in parallel): x is T x d,
 * bf16 bit patterns (x_is_bf16 = 1) or fp32 (0); logits_out[T][E] (may be NULL),
 * idx_out[T][k], w_out[T][k]. Used by the tests to check every token's selection
 * at prefill sizes, where the expert FFN of every token would take too long.
 */
int k3o_route_tokens(int32_t E, int32_t d, int32_t k, const void* x, int32_t x_is_bf16, int64_t T,
                     const float* W, const float* bias, double* logits_out, int32_t* idx_out,
                     double* w_out, int32_t score) {
    int status = 0;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        double* xt = (double*)malloc(sizeof(double) * (size_t)d);
        int st = xt ? 0 : -2;
        if (!st) {
            for (int32_t j = 0; j < d; ++j)
                xt[j] = x_is_bf16 ? k3o_bf16(((const uint16_t*)x)[t * d + j])
                                  : (double)((const float*)x)[t * d + j];
            st = k3o_route_token(E, d, k, xt, W, bias, logits_out ? logits_out + t * E : NULL,
                                 idx_out + t * k, w_out + t * k, score);
        }
        if (st) {
#pragma omp critical
            if (!status) status = st;
        }
        free(xt);
    }
    return status;
}

/* ------------------------------------------------------------------ expert FFN */
static double silu(double z) { return z / (1.0 + exp(g_fault == FAULT_SILU_SIGN ? z : -z)); }

/*
 * One expert on one token: record = [gate codes][gate scales][up codes][up scales]
 * [down codes][down scales]; gate/up are d_ff x d_model (reduction over d_model),
 * down is d_model x d_ff (reduction over d_ff). out[d] = W_down (SiLU(W_gate x) * (W_up x)).
 * h_out[f] (may be NULL) receives the GLU output.
 */
int k3o_expert_token(int32_t d, int32_t f, const uint8_t* record, const double* x, double* out,
                     double* h_out) {
    const int64_t nc = (int64_t)d * f / 2, ns = (int64_t)d * f / 32;
    const uint8_t* gc = record;
    const uint8_t* gs = gc + nc;
    const uint8_t* uc = gs + ns;
    const uint8_t* us = uc + nc;
    const uint8_t* dc = us + ns;
    const uint8_t* ds = dc + nc;
    double* h = (double*)malloc(sizeof(double) * (size_t)f);
    if (!h) return -2;
    for (int32_t r = 0; r < f; ++r) {
        double g = 0.0, u = 0.0, w;
        for (int32_t c = 0; c < d; ++c) {
            if (weight(gc, gs, d, r, c, &w)) { free(h); return -1; }
            g += w * x[c];
            if (weight(uc, us, d, r, c, &w)) { free(h); return -1; }
            u += w * x[c];
        }
        h[r] = (g_fault == FAULT_GLU_ON_UP) ? silu(u) * g : silu(g) * u;
        if (h_out) h_out[r] = h[r];
    }
    for (int32_t i = 0; i < d; ++i) {
        double o = 0.0, w;
        for (int32_t r = 0; r < f; ++r) {
            if (g_fault == FAULT_DOWN_T) {
                /* read the d x f matrix as if it were stored f x d (a transposed-operand slip) */
                int64_t flat = (int64_t)r * d + i;
                if (weight(dc, ds, f, flat / f, flat % f, &w)) { free(h); return -1; }
            } else if (weight(dc, ds, f, i, r, &w)) { free(h); return -1; }
            o += w * h[r];
        }
        out[i] = o;
    }
    free(h);
    return 0;
}

/*
 * One expert with bf16 weights on one token: record = [gate f x d][up f x d][down d x f] bf16 bit
 * patterns, row-major. out[d] = W_down (SiLU(W_gate x) * (W_up x)), the same loops as above with
 * each weight the exact value of its bf16 pattern.
 */
int k3o_expert_token_bf16(int32_t d, int32_t f, const uint16_t* record, const double* x, double* out,
                          double* h_out) {
    const uint16_t* gw = record;
    const uint16_t* uw = gw + (int64_t)f * d;
    const uint16_t* dw = uw + (int64_t)f * d;
    double* h = (double*)malloc(sizeof(double) * (size_t)f);
    if (!h) return -2;
    for (int32_t r = 0; r < f; ++r) {
        double g = 0.0, u = 0.0;
        for (int32_t c = 0; c < d; ++c) {
            g += k3o_bf16(gw[(int64_t)r * d + c]) * x[c];
            u += k3o_bf16(uw[(int64_t)r * d + c]) * x[c];
        }
        h[r] = (g_fault == FAULT_GLU_ON_UP) ? silu(u) * g : silu(g) * u;
        if (h_out) h_out[r] = h[r];
    }
    for (int32_t i = 0; i < d; ++i) {
        double o = 0.0;
        for (int32_t r = 0; r < f; ++r) o += k3o_bf16(dw[(int64_t)i * f + r]) * h[r];
        out[i] = o;
    }
    free(h);
    return 0;
}

/* ------------------------------------------------------------------ layer */
/*
 * One MoE layer over T tokens.
 *   x: T x d, bf16 bit patterns (x_is_bf16 = 1) or fp32 (x_is_bf16 = 0)
 *   W: E x d fp32 router weights; bias: E fp32 or NULL
 *   routed: E record pointers (a NULL entry is an error only if that expert is selected)
 *   shared: S record pointers
 *   y: T x d doubles (overwritten); idx/w: T x k (may be NULL); logits: T x E (may be NULL)
 *   score: 0 softmax, 1 sigmoid + selection-only bias (k3o_route_token)
 *   shared_bf16: 0 shared records are MXFP4 like the routed ones, 1 they are bf16 records
 * Returns 0, -1 on bad data (NaN scale byte, missing record), -2 on allocation failure.
 */
int k3o_layer(int32_t d, int32_t f, int32_t E, int32_t k, int32_t S, const void* x, int32_t x_is_bf16,
              int64_t T, const float* W, const float* bias, const uint8_t* const* routed,
              const uint8_t* const* shared, double* y, int32_t* idx, double* w, double* logits, int32_t score,
              int32_t shared_bf16) {
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        double* xt = (double*)malloc(sizeof(double) * (size_t)d);
        double* o = (double*)malloc(sizeof(double) * (size_t)d);
        int32_t* it = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
        double* wt = (double*)malloc(sizeof(double) * (size_t)k);
        int st = 0;
        if (!xt || !o || !it || !wt) st = -2;
        if (!st) {
            for (int32_t j = 0; j < d; ++j)
                xt[j] = x_is_bf16 ? k3o_bf16(((const uint16_t*)x)[t * d + j])
                                  : (double)((const float*)x)[t * d + j];
            st = k3o_route_token(E, d, k, xt, W, bias, logits ? logits + t * E : NULL, it, wt, score);
        }
        double* yt = y + t * d;
        if (!st) for (int32_t j = 0; j < d; ++j) yt[j] = 0.0;
        for (int32_t i = 0; i < k && !st; ++i) {
            if (!routed[it[i]]) { st = -1; break; }
            st = k3o_expert_token(d, f, routed[it[i]], xt, o, NULL);
            if (!st) for (int32_t j = 0; j < d; ++j) yt[j] += wt[i] * o[j];
        }
        for (int32_t s = 0; s < S && !st && g_fault != FAULT_DROP_SHARED; ++s) {
            st = shared_bf16 ? k3o_expert_token_bf16(d, f, (const uint16_t*)shared[s], xt, o, NULL)
                             : k3o_expert_token(d, f, shared[s], xt, o, NULL);
            const double ws = g_fault == FAULT_SHARED_GATED ? wt[0] : 1.0;
            if (!st) for (int32_t j = 0; j < d; ++j) yt[j] += ws * o[j];
        }
        if (!st) {
            if (idx) memcpy(idx + t * k, it, sizeof(int32_t) * (size_t)k);
            if (w) memcpy(w + t * k, wt, sizeof(double) * (size_t)k);
        }
        if (st) {
#pragma omp critical
            if (!status) status = st;
        }
        free(xt); free(o); free(it); free(wt);
    }
    return status;
}

/* RMSNorm with unit weight: out_j = x_j / sqrt(mean(x^2) + eps) (pre-norm of the stack harness). */
void k3o_rmsnorm(const double* x, int64_t T, int32_t d, double eps, double* out) {
    for (int64_t t = 0; t < T; ++t) {
        double ss = 0.0;
        for (int32_t j = 0; j < d; ++j) ss += x[t * d + j] * x[t * d + j];
        double r = 1.0 / sqrt((g_fault == FAULT_RMS_SUM ? ss : ss / d) + eps);
        for (int32_t j = 0; j < d; ++j) out[t * d + j] = x[t * d + j] * r;
    }
}
