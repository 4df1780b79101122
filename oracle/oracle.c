/*
 * oracle.c -- plain fp64 CPU statement of the recurrent linear-attention
 * decode step over a paged fp32 state pool.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file: only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header or constant with the CUDA path.
 *
 * Notation (state S is K x V, as the recurrence is written):
 *   B batch entries, T tokens per entry, H q/k heads, HV v-heads (HV % H == 0),
 *   K key dim, V value dim, P pool slots.
 *   The pool stores S transposed: pool[p][hv][v][k] = S[k][v], K fastest.
 *
 * Sources followed (web pages, cited by title and section):
 *  - ROCm/aiter PR #4584 "Fused Gluon KDA decode path", advisory review:
 *    the per-token recurrence, in this order:
 *        S <- exp(g_t) * S                  (per-key-channel exp(g_t) for KDA)
 *        S <- S + beta_t * k_t (x) (v_t - S^T k_t)
 *        o_t = S^T q_t
 *    and the in-kernel gate / l2norm / sigmoid fusion; its wrapper review
 *    names A_log, dt_bias and use_gate_in_kernel.
 *  - flashinfer PR "fp32 sibling of #3268" (4D pool + output_state_indices):
 *    read slot initial_state_indices[b], write slot output_state_indices[b]
 *    (defaults to the read slot; a negative entry skips the writeback), pool
 *    written in place through its own strides, optional per-token
 *    intermediate-state cache.
 *  - cuLA PR #75 "wire h0_indices into Lightning Attention decode": the LA
 *    state of (entry n, head h) lives at flat row h0_indices[n] * H + h of a
 *    [pool * H, V, K] tensor.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - GQA map: q/k head of v-head hv is hv / (HV / H).
 *  - l2norm: x / sqrt(sum(x^2) + 1e-6) over K.
 *  - Gate chain: g = -exp(A_log[hv]) * softplus(g_raw + dt_bias), softplus with
 *    torch's default threshold (x > 20 -> x); beta = 1 / (1 + exp(-b_raw)).
 *  - LA update: S <- lambda_h * S + k (x) v, o = S^T q (no delta term).
 *  - A negative read index means a zero initial state; an index >= P is
 *    treated the same way on the read side, skipped on the write side, and
 *    counted in the return value.
 *  - The intermediate cache holds the state after token t, t = 0..T-1.
 *  - T = 0 is a step of no tokens: the recurrence is applied zero times, so
 *    the state as read is what goes to the write slot (the empty spans of the
 *    variable-length mode).
 *  - o is multiplied by `scale` (1.0 unless a caller asks otherwise).
 *
 * Every input except the pool arrives as a contiguous fp64 array (the Python
 * wrapper widens bf16/fp32 exactly).  The pool is fp32 or bfloat16 (flag
 * pool_bf16; values are widened exactly on read and rounded to nearest even
 * on write), read and written in place through four element strides (slot,
 * hv, v, k), so strided views of a
 * larger backing buffer are handled the way the pages require.  All reads of
 * the pool happen before any write (phase 1 / phase 2), so every entry sees
 * the pool as it was when the call started.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * bfloat16: the upper 16 bits of an IEEE fp32 (sign, 8 exponent bits, 7 stored
 * fraction bits, i.e. 8 significant bits).  oracle_round_bf16 rounds an fp64
 * value straight to the nearest bfloat16, ties to even (one rounding, not via
 * fp32), and returns its bit pattern.
 */
uint16_t oracle_round_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double ax = fabs(x);
    double q;                               /* spacing of bfloat16 values around ax */
    if (ax >= 0x1p-126) {
        int e;
        frexp(ax, &e);                      /* ax = m 2^e, m in [0.5, 1) */
        q = ldexp(1.0, e - 8);
    } else {
        q = 0x1p-133;                       /* subnormal spacing: 2^-126 / 2^7 */
    }
    const double r = nearbyint(ax / q) * q; /* ax / q is exact; ties to even */
    if (r >= 0x1p128) return sign | 0x7F80; /* overflow to infinity */
    const float f = (float)r;               /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

static double bf16_value(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Pool element at element offset `off`, widened; pool_bf16 selects the storage type. */
static double elem_get(const void* pool, int pool_bf16, int64_t off) {
    if (pool_bf16) return bf16_value(((const uint16_t*)pool)[off]);
    return (double)((const float*)pool)[off];
}

/* Store x rounded to the pool's type (nearest, ties to even). */
static void elem_put(void* pool, int pool_bf16, int64_t off, double x) {
    if (pool_bf16) ((uint16_t*)pool)[off] = oracle_round_bf16(x);
    else ((float*)pool)[off] = (float)x;    /* fp64 -> fp32 rounds to nearest even */
}

/* Widened pool element S[k][v] of slot p, head hv. */
static double pool_get(const void* pool, int pool_bf16, const int64_t* st, int64_t p, int64_t hv,
                       int64_t vv, int64_t kk) {
    return elem_get(pool, pool_bf16, p * st[0] + hv * st[1] + vv * st[2] + kk * st[3]);
}

static void pool_put(void* pool, int pool_bf16, const int64_t* st, int64_t p, int64_t hv,
                     int64_t vv, int64_t kk, double x) {
    elem_put(pool, pool_bf16, p * st[0] + hv * st[1] + vv * st[2] + kk * st[3], x);
}

/*
 * Gated delta rule decode, GDN (per_channel = 0) or KDA (per_channel = 1).
 *
 *   q, k    [B,T,H,K]
 *   v       [B,T,HV,V]
 *   g       GDN [B,T,HV]; KDA [B,T,HV,K]   (log-decay, or raw gate input if gate_raw)
 *   beta    [B,T,HV]                       (or raw logit if beta_raw)
 *   A_log   [HV]            required when gate_raw
 *   dt_bias GDN [HV]; KDA [HV*K]; may be NULL (zero) when gate_raw
 *   pool    fp32 or bf16 (pool_bf16), strides st[4] in elements over (slot, hv, v, k), P slots
 *   read_idx, write_idx [B] (write_idx NULL: write to the read slot)
 *   out     [B,T,HV,V]
 *   final_state [B,HV,V,K] or NULL: the state after the last token (storage order)
 *   inter   [B,T,HV,V,K] or NULL: the state after each token (storage order)
 *
 * Returns the number of slot indices >= P that were seen, or -1 on a bad argument.
 */
static long delta_rule(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                       int per_channel, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, const double* A_log,
                       const double* dt_bias, int qk_l2norm, int gate_raw, int beta_raw,
                       double scale, void* pool, int pool_bf16, int64_t P, const int64_t* st,
                       const int64_t* read_idx, const int64_t* write_idx,
                       const int64_t* num_accepted, const int64_t* state_idx, double* out,
                       double* final_state, double* inter) {
    if (B < 0 || T < 0 || H < 1 || HV < 1 || K < 1 || V < 1 || HV % H != 0) return -1;
    if (gate_raw && !A_log) return -1;
    if (num_accepted && !state_idx) return -1;
    if (!num_accepted && !read_idx) return -1;
    /* per-token slots need every token's state: keep them even if the caller did not ask */
    double* tok = inter;
    if (state_idx && !tok) {
        tok = (double*)malloc(sizeof(double) * (size_t)(B * T * HV * V * K));
        if (!tok && B > 0) return -1;
    }
    const int64_t group = HV / H;
    long bad = 0;

    double* fin = final_state;
    if (!fin) {
        fin = (double*)malloc(sizeof(double) * (size_t)(B * HV * V * K));
        if (!fin && B > 0) return -1;
    }
    double* S = (double*)malloc(sizeof(double) * (size_t)(K * V)); /* S[kk*V + vv] */
    double* qh = (double*)malloc(sizeof(double) * (size_t)K);
    double* kh = (double*)malloc(sizeof(double) * (size_t)K);
    double* gk = (double*)malloc(sizeof(double) * (size_t)K);
    double* u = (double*)malloc(sizeof(double) * (size_t)V);

    /* phase 1: every state is read and advanced before anything is written */
    for (int64_t b = 0; b < B; ++b) {
        int64_t r;
        if (num_accepted) {
            /* the seed is the state stored after the last accepted token: slot
               state_idx[b][num_accepted[b] - 1]; a count outside [1, T] has no
               such slot and is counted, with a zero seed */
            const int64_t a = num_accepted[b];
            if (a >= 1 && a <= T) {
                r = state_idx[b * T + a - 1];
            } else {
                r = -1;
                ++bad;
            }
        } else {
            r = read_idx[b];
        }
        if (r >= P) ++bad;
        for (int64_t hv = 0; hv < HV; ++hv) {
            const int64_t h = hv / group;

            for (int64_t kk = 0; kk < K; ++kk)
                for (int64_t vv = 0; vv < V; ++vv)
                    S[kk * V + vv] = (r >= 0 && r < P) ? pool_get(pool, pool_bf16, st, r, hv, vv, kk) : 0.0;

            for (int64_t t = 0; t < T; ++t) {
                const double* qt = q + ((b * T + t) * H + h) * K;
                const double* kt = k + ((b * T + t) * H + h) * K;
                const double* vt = v + ((b * T + t) * HV + hv) * V;

                for (int64_t kk = 0; kk < K; ++kk) { qh[kk] = qt[kk]; kh[kk] = kt[kk]; }
                if (qk_l2norm) {
                    double sq = 0.0, sk = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) { sq += qh[kk] * qh[kk]; sk += kh[kk] * kh[kk]; }
                    const double nq = sqrt(sq + 1e-6), nk = sqrt(sk + 1e-6);
                    for (int64_t kk = 0; kk < K; ++kk) { qh[kk] /= nq; kh[kk] /= nk; }
                }

                double bt = beta[(b * T + t) * HV + hv];
                if (beta_raw) bt = sigmoid(bt);

                for (int64_t kk = 0; kk < K; ++kk) {
                    double x = per_channel ? g[((b * T + t) * HV + hv) * K + kk]
                                           : g[(b * T + t) * HV + hv];
                    if (gate_raw) {
                        double bias = 0.0;
                        if (dt_bias) bias = per_channel ? dt_bias[hv * K + kk] : dt_bias[hv];
                        x = -exp(A_log[hv]) * softplus(x + bias);
                    }
                    gk[kk] = x;
                }

                /* S <- exp(g) * S, row kk scaled by exp(g_kk) */
                for (int64_t kk = 0; kk < K; ++kk) {
                    const double d = exp(gk[kk]);
                    for (int64_t vv = 0; vv < V; ++vv) S[kk * V + vv] *= d;
                }
                /* u = S^T k */
                for (int64_t vv = 0; vv < V; ++vv) {
                    double acc = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) acc += S[kk * V + vv] * kh[kk];
                    u[vv] = acc;
                }
                /* S <- S + beta * k (x) (v - u) */
                for (int64_t kk = 0; kk < K; ++kk)
                    for (int64_t vv = 0; vv < V; ++vv)
                        S[kk * V + vv] += kh[kk] * (bt * (vt[vv] - u[vv]));
                /* o = scale * S^T q */
                for (int64_t vv = 0; vv < V; ++vv) {
                    double acc = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) acc += S[kk * V + vv] * qh[kk];
                    out[((b * T + t) * HV + hv) * V + vv] = scale * acc;
                }
                if (tok) {
                    double* it = tok + (((b * T + t) * HV + hv) * V) * K;
                    for (int64_t vv = 0; vv < V; ++vv)
                        for (int64_t kk = 0; kk < K; ++kk) it[vv * K + kk] = S[kk * V + vv];
                }
            }

            double* f = fin + ((b * HV + hv) * V) * K;
            for (int64_t vv = 0; vv < V; ++vv)
                for (int64_t kk = 0; kk < K; ++kk) f[vv * K + kk] = S[kk * V + vv];
        }
    }

    /* phase 2, per-token slots: the state after token t goes to slot state_idx[b][t]
       (in token order); negative skips, >= P is counted and skipped */
    if (state_idx) {
        for (int64_t b = 0; b < B; ++b)
            for (int64_t t = 0; t < T; ++t) {
                const int64_t w = state_idx[b * T + t];
                if (w < 0) continue;
                if (w >= P) { ++bad; continue; }
                for (int64_t hv = 0; hv < HV; ++hv) {
                    const double* f = tok + (((b * T + t) * HV + hv) * V) * K;
                    for (int64_t vv = 0; vv < V; ++vv)
                        for (int64_t kk = 0; kk < K; ++kk)
                            pool_put(pool, pool_bf16, st, w, hv, vv, kk, f[vv * K + kk]);
                }
            }
        if (tok != inter) free(tok);
        free(S); free(qh); free(kh); free(gk); free(u);
        if (fin != final_state) free(fin);
        return bad;
    }

    /* phase 2: writeback to the write slot; negative skips, >= P is counted and skipped */
    for (int64_t b = 0; b < B; ++b) {
        const int64_t w = write_idx ? write_idx[b] : read_idx[b];
        if (w < 0) continue;
        if (w >= P) { ++bad; continue; }
        for (int64_t hv = 0; hv < HV; ++hv) {
            const double* f = fin + ((b * HV + hv) * V) * K;
            for (int64_t vv = 0; vv < V; ++vv)
                for (int64_t kk = 0; kk < K; ++kk) pool_put(pool, pool_bf16, st, w, hv, vv, kk, f[vv * K + kk]);
        }
    }

    free(S); free(qh); free(kh); free(gk); free(u);
    if (fin != final_state) free(fin);
    return bad;
}

long oracle_gdn_decode(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                       const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* A_log, const double* dt_bias,
                       int qk_l2norm, int gate_raw, int beta_raw, double scale, void* pool,
                       int pool_bf16, int64_t P, const int64_t* pool_strides, const int64_t* read_idx,
                       const int64_t* write_idx, double* out, double* final_state,
                       double* inter) {
    return delta_rule(B, T, H, HV, K, V, 0, q, k, v, g, beta, A_log, dt_bias, qk_l2norm,
                      gate_raw, beta_raw, scale, pool, pool_bf16, P, pool_strides, read_idx, write_idx,
                      NULL, NULL, out, final_state, inter);
}

long oracle_kda_decode(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                       const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* A_log, const double* dt_bias,
                       int qk_l2norm, int gate_raw, int beta_raw, double scale, void* pool,
                       int pool_bf16, int64_t P, const int64_t* pool_strides, const int64_t* read_idx,
                       const int64_t* write_idx, double* out, double* final_state,
                       double* inter) {
    return delta_rule(B, T, H, HV, K, V, 1, q, k, v, g, beta, A_log, dt_bias, qk_l2norm,
                      gate_raw, beta_raw, scale, pool, pool_bf16, P, pool_strides, read_idx, write_idx,
                      NULL, NULL, out, final_state, inter);
}

/*
 * Multi-token decode with per-token pool slots (the aiter review's paged
 * per-token state slots and speculative seed):
 *   state_idx    [B, T]: slot that receives the state after token t of entry b
 *   num_accepted [B] or NULL: when given, the seed state is read from slot
 *                state_idx[b][num_accepted[b] - 1] (the state after the last
 *                accepted token of the previous step); otherwise from read_idx[b].
 * Everything else as oracle_gdn_decode / oracle_kda_decode (no write_idx).
 */
long oracle_gdn_decode_tokens(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                              const double* q, const double* k, const double* v, const double* g,
                              const double* beta, const double* A_log, const double* dt_bias,
                              int qk_l2norm, int gate_raw, int beta_raw, double scale, void* pool,
                              int pool_bf16, int64_t P, const int64_t* pool_strides,
                              const int64_t* read_idx, const int64_t* num_accepted,
                              const int64_t* state_idx, double* out, double* final_state,
                              double* inter) {
    if (!state_idx) return -1;
    return delta_rule(B, T, H, HV, K, V, 0, q, k, v, g, beta, A_log, dt_bias, qk_l2norm,
                      gate_raw, beta_raw, scale, pool, pool_bf16, P, pool_strides, read_idx, NULL,
                      num_accepted, state_idx, out, final_state, inter);
}

long oracle_kda_decode_tokens(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                              const double* q, const double* k, const double* v, const double* g,
                              const double* beta, const double* A_log, const double* dt_bias,
                              int qk_l2norm, int gate_raw, int beta_raw, double scale, void* pool,
                              int pool_bf16, int64_t P, const int64_t* pool_strides,
                              const int64_t* read_idx, const int64_t* num_accepted,
                              const int64_t* state_idx, double* out, double* final_state,
                              double* inter) {
    if (!state_idx) return -1;
    return delta_rule(B, T, H, HV, K, V, 1, q, k, v, g, beta, A_log, dt_bias, qk_l2norm,
                      gate_raw, beta_raw, scale, pool, pool_bf16, P, pool_strides, read_idx, NULL,
                      num_accepted, state_idx, out, final_state, inter);
}

/*
 * Lightning-Attention decode (no delta term), cuLA PR #75 layout.
 *
 *   q, k   [B,T,H,K];  v [B,T,H,V];  decay [H] = lambda_h
 *   pool   fp32 or bf16 (pool_bf16) [P*H, V, K], element strides st[3] over (row, v, k);
 *          the state of (entry b, head h) is row read_idx[b] * H + h.
 *   out    [B,T,H,V];  final_state [B,H,V,K] or NULL;  inter [B,T,H,V,K] or NULL
 *
 * Per token: S <- lambda_h * S + k (x) v;  o = scale * S^T q.
 * Returns the number of slot indices >= P seen, or -1 on a bad argument.
 */
long oracle_la_decode(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, const double* q,
                      const double* k, const double* v, const double* decay, double scale,
                      void* pool, int pool_bf16, int64_t pool_rows, const int64_t* st,
                      const int64_t* read_idx, const int64_t* write_idx, double* out,
                      double* final_state, double* inter) {
    if (B < 0 || T < 0 || H < 1 || K < 1 || V < 1 || pool_rows % H != 0) return -1;
    const int64_t P = pool_rows / H;
    long bad = 0;
    double* fin = final_state;
    if (!fin) {
        fin = (double*)malloc(sizeof(double) * (size_t)(B * H * V * K));
        if (!fin && B > 0) return -1;
    }
    double* S = (double*)malloc(sizeof(double) * (size_t)(K * V));

    for (int64_t b = 0; b < B; ++b) {
        const int64_t r = read_idx[b];
        if (r >= P) ++bad;
        for (int64_t h = 0; h < H; ++h) {
            const int64_t row = r * H + h;
            for (int64_t kk = 0; kk < K; ++kk)
                for (int64_t vv = 0; vv < V; ++vv)
                    S[kk * V + vv] = (r >= 0 && r < P)
                        ? elem_get(pool, pool_bf16, row * st[0] + vv * st[1] + kk * st[2]) : 0.0;

            const double lam = decay[h];
            for (int64_t t = 0; t < T; ++t) {
                const double* qt = q + ((b * T + t) * H + h) * K;
                const double* kt = k + ((b * T + t) * H + h) * K;
                const double* vt = v + ((b * T + t) * H + h) * V;
                for (int64_t kk = 0; kk < K; ++kk)
                    for (int64_t vv = 0; vv < V; ++vv)
                        S[kk * V + vv] = lam * S[kk * V + vv] + kt[kk] * vt[vv];
                for (int64_t vv = 0; vv < V; ++vv) {
                    double acc = 0.0;
                    for (int64_t kk = 0; kk < K; ++kk) acc += S[kk * V + vv] * qt[kk];
                    out[((b * T + t) * H + h) * V + vv] = scale * acc;
                }
                if (inter) {
                    double* it = inter + (((b * T + t) * H + h) * V) * K;
                    for (int64_t vv = 0; vv < V; ++vv)
                        for (int64_t kk = 0; kk < K; ++kk) it[vv * K + kk] = S[kk * V + vv];
                }
            }
            double* f = fin + ((b * H + h) * V) * K;
            for (int64_t vv = 0; vv < V; ++vv)
                for (int64_t kk = 0; kk < K; ++kk) f[vv * K + kk] = S[kk * V + vv];
        }
    }

    for (int64_t b = 0; b < B; ++b) {
        const int64_t w = write_idx ? write_idx[b] : read_idx[b];
        if (w < 0) continue;
        if (w >= P) { ++bad; continue; }
        for (int64_t h = 0; h < H; ++h) {
            const int64_t row = w * H + h;
            const double* f = fin + ((b * H + h) * V) * K;
            for (int64_t vv = 0; vv < V; ++vv)
                for (int64_t kk = 0; kk < K; ++kk)
                    elem_put(pool, pool_bf16, row * st[0] + vv * st[1] + kk * st[2], f[vv * K + kk]);
        }
    }
    free(S);
    if (fin != final_state) free(fin);
    return bad;
}
