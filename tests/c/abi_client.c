/* A plain C client of the decode library: no Python, no torch.  It builds a
 * small gated-delta-rule decode case on the host, runs it through the C ABI
 * (gdn_decode on device buffers it allocates itself, then gdn_decode_varlen on
 * the same tokens packed as spans), runs the same inputs through the fp64
 * oracle, and compares.  It also checks that a host-side
 * argument error comes back as a status before any launch.
 *
 * Exit status 0 on success; prints the first mismatch otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "lar.h"

/* the oracle's entry point (oracle/oracle.c) */
long oracle_gdn_decode(int64_t B, int64_t T, int64_t H, int64_t HV, int64_t K, int64_t V,
                       const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* A_log, const double* dt_bias,
                       int qk_l2norm, int gate_raw, int beta_raw, double scale, void* pool,
                       int pool_bf16, int64_t P, const int64_t* pool_strides, const int64_t* read_idx,
                       const int64_t* write_idx, double* out, double* final_state, double* inter);

enum { B = 3, T = 2, H = 1, HV = 2, K = 32, V = 40, P = 5 };

/* inputs: a 64-bit linear congruential sequence mapped to [-1, 1) */
static uint64_t lcg_state = 12345u;
static float uniform_pm1(void) {
    lcg_state = lcg_state * 6364136223846793005ull + 1442695040888963407ull;
    return (float)((double)(lcg_state >> 11) / 9007199254740992.0 * 2.0 - 1.0);
}

#define CHECK_CUDA(x)                                                                   \
    do {                                                                                \
        cudaError_t e_ = (x);                                                           \
        if (e_ != cudaSuccess) {                                                        \
            fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            return 2;                                                                   \
        }                                                                               \
    } while (0)

static lar_tensor desc(void* data, int32_t dtype, int ndim, const int64_t* shape) {
    lar_tensor t;
    memset(&t, 0, sizeof t);
    t.data = data;
    t.dtype = dtype;
    t.ndim = ndim;
    int64_t s = 1;
    for (int i = ndim - 1; i >= 0; --i) {  /* contiguous, row-major element strides */
        t.shape[i] = shape[i];
        t.stride[i] = s;
        s *= shape[i];
    }
    return t;
}

int main(void) {
    const size_t nq = (size_t)B * T * H * K, nv = (size_t)B * T * HV * V, ng = (size_t)B * T * HV;
    const size_t npool = (size_t)P * HV * V * K;
    float *q = malloc(nq * 4), *k = malloc(nq * 4), *v = malloc(nv * 4), *g = malloc(ng * 4);
    float *beta = malloc(ng * 4), *pool = malloc(npool * 4), *pool_ref = malloc(npool * 4);
    float* out = malloc(nv * 4);
    float* pool0 = malloc(npool * 4);
    for (size_t i = 0; i < nq; ++i) q[i] = uniform_pm1() * 0.3f;
    for (size_t i = 0; i < nq; ++i) k[i] = uniform_pm1() * 0.3f;
    for (size_t i = 0; i < nv; ++i) v[i] = uniform_pm1();
    for (size_t i = 0; i < ng; ++i) g[i] = -0.5f * (uniform_pm1() + 1.0f);   /* log decay in (-1, 0] */
    for (size_t i = 0; i < ng; ++i) beta[i] = 0.5f * (uniform_pm1() + 1.0f);
    for (size_t i = 0; i < npool; ++i) pool[i] = 0.1f * uniform_pm1();
    memcpy(pool_ref, pool, npool * 4);
    memcpy(pool0, pool, npool * 4);
    const int32_t ridx[B] = {4, 0, 2}, widx[B] = {1, -1, 3};

    /* ---- device side through the C ABI */
    float *dq, *dk, *dv, *dg, *dbeta, *dpool, *dout;
    int32_t *dridx, *dwidx, *derr;
    CHECK_CUDA(cudaMalloc((void**)&dq, nq * 4));
    CHECK_CUDA(cudaMalloc((void**)&dk, nq * 4));
    CHECK_CUDA(cudaMalloc((void**)&dv, nv * 4));
    CHECK_CUDA(cudaMalloc((void**)&dg, ng * 4));
    CHECK_CUDA(cudaMalloc((void**)&dbeta, ng * 4));
    CHECK_CUDA(cudaMalloc((void**)&dpool, npool * 4));
    CHECK_CUDA(cudaMalloc((void**)&dout, nv * 4));
    CHECK_CUDA(cudaMalloc((void**)&dridx, sizeof ridx));
    CHECK_CUDA(cudaMalloc((void**)&dwidx, sizeof widx));
    CHECK_CUDA(cudaMalloc((void**)&derr, 4));
    CHECK_CUDA(cudaMemcpy(dq, q, nq * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dk, k, nq * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, v, nv * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dg, g, ng * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dbeta, beta, ng * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dpool, pool, npool * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dridx, ridx, sizeof ridx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dwidx, widx, sizeof widx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(derr, 0, 4));

    const int64_t sq[4] = {B, T, H, K}, sv[4] = {B, T, HV, V}, sg[3] = {B, T, HV};
    const int64_t sp[4] = {P, HV, V, K}, si[1] = {B};
    lar_tensor tq = desc(dq, LAR_F32, 4, sq), tk = desc(dk, LAR_F32, 4, sq), tv = desc(dv, LAR_F32, 4, sv);
    lar_tensor tg = desc(dg, LAR_F32, 3, sg), tb = desc(dbeta, LAR_F32, 3, sg);
    lar_tensor tp = desc(dpool, LAR_F32, 4, sp), tr = desc(dridx, LAR_I32, 1, si);
    lar_tensor tw = desc(dwidx, LAR_I32, 1, si), to = desc(dout, LAR_F32, 4, sv);
    const float scale = 0.5f;

    /* a host-detectable error: no q at all */
    lar_status st = gdn_decode(NULL, &tk, &tv, &tg, &tb, NULL, NULL, &tp, &tr, &tw, &to, NULL, scale, 0, derr, NULL);
    if (st != LAR_ERR_NULL || lar_status_string(st) == NULL) {
        fprintf(stderr, "NULL q: expected LAR_ERR_NULL, got %d\n", (int)st);
        return 1;
    }
    st = gdn_decode(&tq, &tk, &tv, &tg, &tb, NULL, NULL, &tp, &tr, &tw, &to, NULL, scale, 0, derr, NULL);
    if (st != LAR_OK) {
        fprintf(stderr, "gdn_decode: %s\n", lar_status_string(st));
        return 1;
    }
    int32_t err = -1;
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_CUDA(cudaMemcpy(out, dout, nv * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(pool, dpool, npool * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(&err, derr, 4, cudaMemcpyDeviceToHost));
    if (err != 0) {
        fprintf(stderr, "dev_err = %d\n", err);
        return 1;
    }

    /* ---- the oracle on the same inputs */
    double *q64 = malloc(nq * 8), *k64 = malloc(nq * 8), *v64 = malloc(nv * 8), *g64 = malloc(ng * 8);
    double *b64 = malloc(ng * 8), *out64 = malloc(nv * 8), *fin64 = malloc((size_t)B * HV * V * K * 8);
    for (size_t i = 0; i < nq; ++i) { q64[i] = q[i]; k64[i] = k[i]; }
    for (size_t i = 0; i < nv; ++i) v64[i] = v[i];
    for (size_t i = 0; i < ng; ++i) { g64[i] = g[i]; b64[i] = beta[i]; }
    const int64_t pst[4] = {(int64_t)HV * V * K, (int64_t)V * K, K, 1};
    const int64_t r64[B] = {ridx[0], ridx[1], ridx[2]}, w64[B] = {widx[0], widx[1], widx[2]};
    long bad = oracle_gdn_decode(B, T, H, HV, K, V, q64, k64, v64, g64, b64, NULL, NULL, 0, 0, 0, scale,
                                 pool_ref, 0, P, pst, r64, w64, out64, fin64, NULL);
    if (bad != 0) {
        fprintf(stderr, "oracle reported %ld bad slots\n", bad);
        return 1;
    }

    /* ---- compare: outputs and every pool element (written slots and untouched ones) */
    for (size_t i = 0; i < nv; ++i) {
        const double d = fabs((double)out[i] - out64[i]);
        if (d > 1e-4 * fabs(out64[i]) + 1e-5) {
            fprintf(stderr, "out[%zu]: lib %.9g oracle %.9g\n", i, (double)out[i], out64[i]);
            return 1;
        }
    }
    for (size_t i = 0; i < npool; ++i) {
        const double d = fabs((double)pool[i] - (double)pool_ref[i]);
        if (d > 1e-4 * fabs((double)pool_ref[i]) + 1e-6) {
            fprintf(stderr, "pool[%zu]: lib %.9g oracle %.9g\n", i, (double)pool[i], (double)pool_ref[i]);
            return 1;
        }
    }

    /* ---- the same tokens as variable-length spans: B sequences of T tokens, token-major */
    int32_t* dcu;
    const int32_t cu[B + 1] = {0, T, 2 * T, 3 * T};
    CHECK_CUDA(cudaMalloc((void**)&dcu, sizeof cu));
    CHECK_CUDA(cudaMemcpy(dcu, cu, sizeof cu, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dpool, pool0, npool * 4, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(dout, 0, nv * 4));
    const int64_t vq[3] = {B * T, H, K}, vv[3] = {B * T, HV, V}, vg[2] = {B * T, HV}, vc[1] = {B + 1};
    lar_tensor uq = desc(dq, LAR_F32, 3, vq), uk = desc(dk, LAR_F32, 3, vq), uv = desc(dv, LAR_F32, 3, vv);
    lar_tensor ug = desc(dg, LAR_F32, 2, vg), ub = desc(dbeta, LAR_F32, 2, vg), uo = desc(dout, LAR_F32, 3, vv);
    lar_tensor uc = desc(dcu, LAR_I32, 1, vc);
    st = gdn_decode_varlen(&uq, &uk, &uv, &ug, &ub, NULL, NULL, &tp, &uc, &tr, &tw, &uo, NULL, scale, 0, derr, NULL);
    if (st != LAR_OK) {
        fprintf(stderr, "gdn_decode_varlen: %s\n", lar_status_string(st));
        return 1;
    }
    CHECK_CUDA(cudaDeviceSynchronize());
    CHECK_CUDA(cudaMemcpy(out, dout, nv * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(pool, dpool, npool * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(&err, derr, 4, cudaMemcpyDeviceToHost));
    if (err != 0) {
        fprintf(stderr, "varlen dev_err = %d\n", err);
        return 1;
    }
    for (size_t i = 0; i < nv; ++i) {
        const double d = fabs((double)out[i] - out64[i]);
        if (d > 1e-4 * fabs(out64[i]) + 1e-5) {
            fprintf(stderr, "varlen out[%zu]: lib %.9g oracle %.9g\n", i, (double)out[i], out64[i]);
            return 1;
        }
    }
    for (size_t i = 0; i < npool; ++i) {
        const double d = fabs((double)pool[i] - (double)pool_ref[i]);
        if (d > 1e-4 * fabs((double)pool_ref[i]) + 1e-6) {
            fprintf(stderr, "varlen pool[%zu]: lib %.9g oracle %.9g\n", i, (double)pool[i], (double)pool_ref[i]);
            return 1;
        }
    }
    printf("C ABI client: gdn_decode and gdn_decode_varlen match the oracle (%zu outputs, %zu pool elements)\n",
           nv, npool);
    return 0;
}
