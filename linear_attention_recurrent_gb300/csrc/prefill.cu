// prefill.cu -- chunked form of the gated delta rule (scalar decay, GDN) and of
// Lightning Attention (LA) over variable-length spans: the prefill path for long
// spans, at K = V = 128.
//
// Math.  Take one chunk of C tokens of a span, S0 the state entering it, a_t the
// per-token decay factor (GDN e^{g_t}, LA lambda) and P[t][s] = a_{s+1} ... a_t
// the decay from token s to token t (P[t][t] = 1), E_t = a_0 ... a_t.  Unrolling
// the per-token recurrence (decay, read-out S^T k on the decayed state, rank-1
// update, o = S^T q on the updated state; the aiter KDA review's order) over the
// chunk, the corrections d_t = beta_t (v_t - (a_t S_{t-1})^T k_t) solve the unit
// lower-triangular system
//     d_t + sum_{s<t} beta_t P[t][s] (k_t . k_s) d_s = beta_t (v_t - E_t S0^T k_t),
// the outputs are
//     o_t = E_t S0^T q_t + sum_{s<=t} P[t][s] (q_t . k_s) d_s,
// and the state leaving the chunk is
//     S = E_{C-1} S0 + sum_s P[C-1][s] k_s d_s^T.
// LA is the case d_t = v_t (no read-out correction).  The decay table is built
// from products of the per-token factors, as the recurrence applies them, not
// from differences of log-decay prefix sums (which lose precision for large
// decays and break down for a factor of 0).
//
// KDA (a decay factor a_t[c] per key channel c) is the same unrolling with the
// decay inside the dot products: P[t][s][c] = a_{s+1}[c] ... a_t[c],
// E_t[c] = a_0[c] ... a_t[c], and
//     A[t][s] = beta_t sum_c k_t[c] k_s[c] P[t][s][c]            (s < t)
//     d + A d = beta (v - (E o K) S0),
//     o_t = (E_t o q_t)^T S0 + sum_{s<=t} (sum_c q_t[c] k_s[c] P[t][s][c]) d_s,
//     S = diag(E_{C-1}) S0 + sum_s (P[C-1][s] o k_s) d_s^T.
// P[t][s][c] is a running product over t for each (s, c): every factor is at
// most 1, so nothing overflows, and a product that underflows is negligible
// next to the terms it is added to.
//
// Work.  A CTA of 256 threads per (sequence, v-head, block of VB value
// columns) keeps its columns of S (K x VB, fp32) in shared memory for the
// whole span and walks the span a chunk at a time: load the chunk (q, k
// l2-normalised when asked; v; decays; betas), the products K S0 and Q S0
// (4 rows x VB/32 columns per thread), K K^T and Q K^T, the triangular solve
// (one value column per thread), the outputs, and the state update (VB/16
// rows x 8 columns per thread).  Everything is fp32 on the CUDA
// cores with packed fp32x2 multiply-adds: the state must stay within 1e-4
// relative of the fp64 recurrence, which the tensor cores' tf32 and bf16 input
// formats do not give.  A tail chunk is padded with zero tokens (k = q = v = 0,
// beta = 0, decay factor 1), which change nothing.
#include "decode_kernel.cuh"

namespace lar {
namespace {

constexpr int PK = 128;        // key channels
constexpr int PV = 128;        // value channels
constexpr int PC = 32;         // tokens per chunk
constexpr int PTH = 256;       // threads per CTA
constexpr int KROW = PK + 4;   // padded q / k row
constexpr int TROW = PC + 1;   // padded row of the chunk's C x C tables
// value columns per CTA: each (sequence, head) pair is split over PV / VB CTAs,
// one per column block (the triangular solve, the outputs and the state update
// are independent per value column; K K^T and Q K^T are recomputed by each).
// 64 columns halve the shared memory (86 KB) and the registers (126), so two
// CTAs share an SM: 5-13 % faster than one 128-column CTA per pair.
#ifndef LAR_PF_VB
#define LAR_PF_VB 64
#endif

// shared-memory layout for VB value columns per CTA, in floats (KDA adds the
// per-channel decay rows)
template <int VB, bool KDA = false>
struct PfLayout {
    static constexpr int SROW = VB + 4;                  // padded state row
    static constexpr int OFF_S = 0;                      // S [K][SROW]
    static constexpr int OFF_K = OFF_S + PK * SROW;      // k rows [C][KROW]
    static constexpr int OFF_Q = OFF_K + PC * KROW;      // q rows [C][KROW]
    static constexpr int OFF_D = OFF_Q + PC * KROW;      // v rows, then right-hand sides, then d [C][VB]
    static constexpr int OFF_A = OFF_D + PC * VB;        // beta_t P[t][s] (k_t . k_s), s < t  [C][TROW]
    static constexpr int OFF_M = OFF_A + PC * TROW;      // decay table, then P[t][s] (q_t . k_s)  [C][TROW]
    static constexpr int OFF_AF = OFF_M + PC * TROW;     // a_t
    static constexpr int OFF_E = OFF_AF + PC;            // E_t
    static constexpr int OFF_W = OFF_E + PC;             // P[C-1][s]
    static constexpr int OFF_B = OFF_W + PC;             // beta_t
    static constexpr int OFF_AD = OFF_B + PC;            // KDA: a_t[c] [C][K]
    static constexpr int OFF_X = OFF_AD + (KDA ? PC * PK : 0);   // KDA: P[C-1][s][c] k_s[c] [C][K]
    static constexpr int OFF_EC = OFF_X + (KDA ? PC * PK : 0);   // KDA: E_{C-1}[c] [K]
    static constexpr int FLOATS = OFF_EC + (KDA ? PK : 0);
    static constexpr size_t BYTES = static_cast<size_t>(FLOATS) * sizeof(float);
    static_assert(OFF_K % 4 == 0 && OFF_Q % 4 == 0 && OFF_D % 4 == 0 && OFF_A % 4 == 0 && OFF_AD % 4 == 0 &&
                      OFF_X % 4 == 0,
                  "16-byte aligned blocks");
    static_assert(BYTES <= 227 * 1024, "fits one CTA's shared memory");
};

__device__ __forceinline__ float comp(const float4& x, int i) {
    return i == 0 ? x.x : (i == 1 ? x.y : (i == 2 ? x.z : x.w));
}

__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }

template <int FORM, int SB, int VB>
__global__ void __launch_bounds__(PTH, (VB == 128 || FORM == FORM_KDA) ? 1 : 2) prefill_kernel(const DecodeParams p) {
    constexpr bool KDA = FORM == FORM_KDA;
    using LY = PfLayout<VB, KDA>;
    constexpr int SROW = LY::SROW;
    extern __shared__ __align__(16) float sm[];
    float* S = sm + LY::OFF_S;
    float* Kc = sm + LY::OFF_K;
    float* Qc = sm + LY::OFF_Q;
    float* D = sm + LY::OFF_D;
    float* A = sm + LY::OFF_A;
    float* M = sm + LY::OFF_M;
    float* Af = sm + LY::OFF_AF;
    float* E = sm + LY::OFF_E;
    float* Wd = sm + LY::OFF_W;
    float* Bt = sm + LY::OFF_B;
    float* Ad = sm + LY::OFF_AD;     // KDA only
    float* X = sm + LY::OFF_X;       // KDA only
    float* EC = sm + LY::OFF_EC;     // KDA only

    constexpr int NSPLIT = PV / VB;        // CTAs per (sequence, head) pair, one per column block
    constexpr int CP = VB / 32;            // columns per thread in the products and outputs (2 or 4)
    constexpr int CP2 = CP / 2;            // ... as float pairs
    constexpr int RK = VB / 16;            // state rows per thread in the update (8 columns each)
    constexpr int VX = VB / 8;             // threads across the columns in the update
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int hv = blockIdx.x / NSPLIT;
    const int v0 = (blockIdx.x % NSPLIT) * VB;
    const int n = blockIdx.y;
    const int h = hv / p.group;
    constexpr int EPC = 16 / SB;     // pool elements per 16-byte chunk
    constexpr int NCHK = PK / EPC;   // chunks per state row

#if LAR_PDL
    // programmatic dependent launch: everything below may read what the
    // previous kernel on the stream wrote
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif
    // ---- span and slots (a span that is reversed or runs past the token
    // arrays is run as empty and flagged, as in the decode kernel; one CTA of
    // the sequence reports)
    const int64_t lo = ld_idx(p.cu, n * p.cu_s, p.cu_dt);
    const int64_t hi = ld_idx(p.cu, (n + 1) * p.cu_s, p.cu_dt);
    const bool span_ok = lo >= 0 && hi >= lo && hi <= p.ntok;
    const int64_t tb = span_ok ? lo : 0;
    const int64_t L = span_ok ? hi - lo : 0;
    // a variable-length call sends only its long spans here (the rest run token
    // by token), and none when some span is reversed (the token-by-token kernel
    // then takes them all)
    if (p.split_len > 0) {
        if (L < p.split_len) return;
        bool rev = false;
        for (int i = tid; i < p.B; i += PTH)
            rev |= ld_idx(p.cu, (i + 1) * p.cu_s, p.cu_dt) < ld_idx(p.cu, i * p.cu_s, p.cu_dt);
        if (__syncthreads_or(rev)) return;
    }
    const int64_t r = ld_idx(p.ridx, n * p.ri_s, p.ri_dt);
    const int64_t w = p.widx ? ld_idx(p.widx, n * p.wi_s, p.wi_dt) : r;
    const bool rd = r >= 0 && r < p.P;
    const bool wr = w >= 0 && w < p.P;
    if (tid == 0 && blockIdx.x == 0 && p.dev_err) {
        const int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0) |
                      (span_ok ? 0 : LAR_DEVERR_SEQLEN);
        if (e) atomicOr(p.dev_err, e);
    }

    // ---- S[k][v] = pool[r][hv][v0 + v][k] for the CTA's VB columns
    {
        const unsigned char* base =
            static_cast<const unsigned char*>(p.pool) + ((rd ? r : 0) * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1]) * SB;
        constexpr int TOT = VB * NCHK;
        constexpr int NB = TOT / PTH < 8 ? TOT / PTH : 8;   // chunks in flight per thread
        static_assert(TOT % (NB * PTH) == 0, "whole batches");
#pragma unroll 1
        for (int i0 = tid; i0 < TOT; i0 += NB * PTH) {
            uint4 raw[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int i = i0 + j * PTH;
                raw[j] = make_uint4(0u, 0u, 0u, 0u);
                if (rd)
                    raw[j] = __ldg(reinterpret_cast<const uint4*>(base + static_cast<int64_t>(v0 + i % VB) * p.ps[2] * SB) +
                                   i / VB);
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int i = i0 + j * PTH;
                const int v = i % VB;
                const int c = i / VB;
                const unsigned wd[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
                if constexpr (SB == 4) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) S[(c * 4 + e) * SROW + v] = __uint_as_float(wd[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        S[(c * 8 + 2 * e) * SROW + v] = __uint_as_float(wd[e] << 16);
                        S[(c * 8 + 2 * e + 1) * SROW + v] = __uint_as_float(wd[e] & 0xffff0000u);
                    }
                }
            }
        }
    }
    __syncthreads();

    const bool l2 = FORM != FORM_LA && (p.flags & LAR_QK_L2NORM) != 0;
    const bool gate_raw = (p.flags & LAR_GATE_RAW) != 0;
    const bool beta_raw = (p.flags & LAR_BETA_RAW) != 0;
    const int ty = tid >> 5, tx = tid & 31;   // products and outputs: rows 4ty.., columns CP tx..

    // A chunk's q, k, v, gate and beta values are loaded into registers, every
    // load of a thread issued before any is used.  q, k: one warp per row
    // (rows warp, warp + 8, ...), 4 channels per lane; v: the CTA's columns,
    // VB / 8 values per thread; gates and betas: lane t of warp 0.  (Loading
    // the next chunk's values during the current chunk's arithmetic measured
    // no faster.)
    constexpr int RPW = PC / (PTH / 32);   // q / k rows per warp
    constexpr int VPT = PC * VB / PTH;     // v values per thread
    float qx[RPW][4], kx[RPW][4], vx[VPT], gx = 0.f, bx = 0.f;
    float gk[KDA ? RPW : 1][4];      // KDA: the gate inputs of a q / k row's channels
    auto fetch = [&](int64_t c0) {
        const int Lc = static_cast<int>(L - c0 < PC ? L - c0 : PC);
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const int t = warp + j * (PTH / 32);
            const bool ok = t < Lc;
            const int64_t gt = tb + c0 + t;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = lane * 4 + e;
                qx[j][e] = ok ? ld_in(p.q, gt * p.qs[1] + h * p.qs[2] + c * p.qs[3], p.q_dt) : 0.f;
                kx[j][e] = ok ? ld_in(p.k, gt * p.ks[1] + h * p.ks[2] + c * p.ks[3], p.k_dt) : 0.f;
                if constexpr (KDA)
                    gk[j][e] = ok ? ld_in(p.g, gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2] + c * p.gs[3], p.g_dt)
                                  : 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int i = tid + j * PTH;
            const int t = i / VB;
            const int v = i - t * VB;
            vx[j] = t < Lc ? ld_in(p.v, (tb + c0 + t) * p.vs[1] + static_cast<int64_t>(hv) * p.vs[2] +
                                           (v0 + v) * p.vs[3], p.v_dt)
                           : 0.f;
        }
        if constexpr (FORM != FORM_LA) {
            if (warp == 0 && lane < Lc) {
                const int64_t gt = tb + c0 + lane;
                if constexpr (!KDA) gx = ld_in(p.g, gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2], p.g_dt);
                bx = ld_in(p.beta, gt * p.bs[1] + static_cast<int64_t>(hv) * p.bs[2], p.beta_dt);
            }
        }
    };

#pragma unroll 1
    for (int64_t c0 = 0; c0 < L; c0 += PC) {
        const int Lc = static_cast<int>(L - c0 < PC ? L - c0 : PC);
        fetch(c0);
        // ---- the chunk's q, k (l2-normalised when asked) and v rows into shared memory
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const int t = warp + j * (PTH / 32);
            float iq = 1.f, ik = 1.f;
            if (l2) {
                float sq = 0.f, sk = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sq = fmaf(qx[j][e], qx[j][e], sq);
                    sk = fmaf(kx[j][e], kx[j][e], sk);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    sq += __shfl_xor_sync(0xffffffffu, sq, off);
                    sk += __shfl_xor_sync(0xffffffffu, sk, off);
                }
                iq = 1.f / sqrtf(sq + 1e-6f);
                ik = 1.f / sqrtf(sk + 1e-6f);
            }
            *reinterpret_cast<float4*>(Qc + t * KROW + lane * 4) =
                make_float4(qx[j][0] * iq, qx[j][1] * iq, qx[j][2] * iq, qx[j][3] * iq);
            *reinterpret_cast<float4*>(Kc + t * KROW + lane * 4) =
                make_float4(kx[j][0] * ik, kx[j][1] * ik, kx[j][2] * ik, kx[j][3] * ik);
            if constexpr (KDA) {
                // per-channel decay factors a_t[c] (gate chain included); padding tokens: 1
                float a4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x = gk[j][e];
                    if (gate_raw) {
                        const int c = lane * 4 + e;
                        const float bias = p.dt_bias ? p.dt_bias[(static_cast<int64_t>(hv) * PK + c) * p.dtb_s] : 0.f;
                        x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
                    }
                    a4[e] = t < Lc ? expf(x) : 1.f;
                }
                *reinterpret_cast<float4*>(Ad + t * PK + lane * 4) = make_float4(a4[0], a4[1], a4[2], a4[3]);
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) D[tid + j * PTH] = vx[j];
        // ---- per-token decay factors and betas (warp 0, lane t), then the decay table
        if (warp == 0) {
            const int t = lane;
            float a = 1.f, bt = 0.f;   // padding tokens: no decay, no update
            if (t < Lc) {
                if constexpr (FORM == FORM_LA) {
                    a = p.decay[h * p.dec_s];
                    bt = 1.f;
                } else {
                    if constexpr (!KDA) {
                        float x = gx;
                        if (gate_raw) {
                            const float bias = p.dt_bias ? p.dt_bias[hv * p.dtb_s] : 0.f;
                            x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
                        }
                        a = expf(x);
                    }
                    bt = beta_raw ? 1.f / (1.f + expf(-bx)) : bx;
                }
            }
            Af[t] = a;
            Bt[t] = bt;
            __syncwarp();
            if constexpr (!KDA) {
                // row t: P[t][s] = a_{s+1} ... a_t for s <= t, 0 above
                float f = 1.f;
#pragma unroll 1
                for (int s = PC - 1; s >= 0; --s) {
                    if (s <= t) {
                        M[t * TROW + s] = f;
                        f *= Af[s];
                    } else {
                        M[t * TROW + s] = 0.f;
                    }
                }
                E[t] = f;   // a_0 ... a_t
                if (t == PC - 1) {
#pragma unroll 1
                    for (int s = 0; s < PC; ++s) Wd[s] = M[t * TROW + s];
                }
            }
        }
        __syncthreads();

        if constexpr (KDA) {
            // ---- A[t][s] = beta_t sum_c k_t[c] k_s[c] P[t][s][c] (s < t) and
            // M[t][s] = sum_c q_t[c] k_s[c] P[t][s][c] (s <= t).  Warp w takes
            // s = w, w + 8, ...; lane l channels 4l .. 4l + 3, with the products
            // P[t][s][c] kept as a running product over t.  Each lane's 32
            // partial sums (one per t) are reduced across the warp by recursive
            // halving, which leaves lane l holding the sums for t = l.
            static_assert(PC == 32, "one token per lane after the reduction");
#pragma unroll 1
            for (int s = warp; s < PC; s += PTH / 32) {
                const float4 ks = *reinterpret_cast<const float4*>(Kc + s * KROW + 4 * lane);
                float4 pr = make_float4(1.f, 1.f, 1.f, 1.f);
                float va[PC], vm[PC];
#pragma unroll
                for (int t = 0; t < PC; ++t) {
                    va[t] = 0.f;
                    vm[t] = 0.f;
                    if (t >= s) {
                        if (t > s) {
                            const float4 a4 = *reinterpret_cast<const float4*>(Ad + t * PK + 4 * lane);
                            pr = make_float4(pr.x * a4.x, pr.y * a4.y, pr.z * a4.z, pr.w * a4.w);
                        }
                        const float4 kt = *reinterpret_cast<const float4*>(Kc + t * KROW + 4 * lane);
                        const float4 qt = *reinterpret_cast<const float4*>(Qc + t * KROW + 4 * lane);
                        const float wx = ks.x * pr.x, wy = ks.y * pr.y, wz = ks.z * pr.z, ww = ks.w * pr.w;
                        va[t] = fmaf(kt.w, ww, fmaf(kt.z, wz, fmaf(kt.y, wy, kt.x * wx)));
                        vm[t] = fmaf(qt.w, ww, fmaf(qt.z, wz, fmaf(qt.y, wy, qt.x * wx)));
                    }
                }
#pragma unroll
                for (int n = PC / 2; n >= 1; n >>= 1) {
                    const bool up = (lane & n) != 0;
#pragma unroll
                    for (int i = 0; i < n; ++i) {
                        const float sa = up ? va[i] : va[i + n];
                        const float sq = up ? vm[i] : vm[i + n];
                        const float ka = up ? va[i + n] : va[i];
                        const float kq = up ? vm[i + n] : vm[i];
                        va[i] = ka + __shfl_xor_sync(0xffffffffu, sa, n);
                        vm[i] = kq + __shfl_xor_sync(0xffffffffu, sq, n);
                    }
                }
                const int t = lane;
                A[t * TROW + s] = t > s ? Bt[t] * va[0] : 0.f;
                M[t * TROW + s] = t >= s ? vm[0] : 0.f;
            }
            __syncthreads();
            // ---- per channel c: X[s][c] = P[C-1][s][c] k_s[c] (a running product
            // from the chunk's end), then k_t and q_t scaled by E_t[c] in place, and
            // E_{C-1}[c]
            if (tid < PK) {
                const int c = tid;
                float w = 1.f;
#pragma unroll 4
                for (int s = PC - 1; s >= 0; --s) {
                    X[s * PK + c] = Kc[s * KROW + c] * w;
                    w *= Ad[s * PK + c];
                }
                float e = 1.f;
#pragma unroll 4
                for (int t = 0; t < PC; ++t) {
                    e *= Ad[t * PK + c];
                    Kc[t * KROW + c] *= e;
                    Qc[t * KROW + c] *= e;
                }
                EC[c] = e;
            }
            __syncthreads();
        }

        // ---- K S0 and Q S0: rows 4ty..4ty+3, columns CP tx .. CP tx + CP - 1
        float2 oq[4][CP2];
        {
            float2 ak[4][CP2], aq[4][CP2];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < CP2; ++c) ak[i][c] = aq[i][c] = make_float2(0.f, 0.f);
#pragma unroll 2
            for (int k = 0; k < PK; k += 4) {
                float4 kr[4], qr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    kr[i] = *reinterpret_cast<const float4*>(Kc + (4 * ty + i) * KROW + k);
                    qr[i] = *reinterpret_cast<const float4*>(Qc + (4 * ty + i) * KROW + k);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    float2 sv[CP2];
                    if constexpr (CP == 4) {
                        const float4 s4 = *reinterpret_cast<const float4*>(S + (k + kk) * SROW + 4 * tx);
                        sv[0] = make_float2(s4.x, s4.y);
                        sv[CP2 - 1] = make_float2(s4.z, s4.w);
                    } else {
                        sv[0] = *reinterpret_cast<const float2*>(S + (k + kk) * SROW + 2 * tx);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if constexpr (FORM != FORM_LA) {
                            const float2 kv = dup(comp(kr[i], kk));
#pragma unroll
                            for (int c = 0; c < CP2; ++c) ak[i][c] = __ffma2_rn(kv, sv[c], ak[i][c]);
                        }
                        const float2 qv = dup(comp(qr[i], kk));
#pragma unroll
                        for (int c = 0; c < CP2; ++c) aq[i][c] = __ffma2_rn(qv, sv[c], aq[i][c]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * ty + i;
                // KDA: the per-channel E_t is already inside the scaled q and k rows
                const float2 et = dup(KDA ? 1.f : E[t]);
#pragma unroll
                for (int c = 0; c < CP2; ++c) oq[i][c] = __fmul2_rn(et, aq[i][c]);
                if constexpr (FORM != FORM_LA) {
                    // right-hand side beta_t (v_t - E_t (S0^T k_t)), in place of v_t
                    const float b = Bt[t], e = KDA ? 1.f : E[t];
#pragma unroll
                    for (int c = 0; c < CP2; ++c) {
                        float2* dp = reinterpret_cast<float2*>(D + t * VB + CP * tx + 2 * c);
                        const float2 d2 = *dp;
                        *dp = make_float2(b * fmaf(-e, ak[i][c].x, d2.x), b * fmaf(-e, ak[i][c].y, d2.y));
                    }
                }
            }
        }

        // ---- K K^T and Q K^T: row t, columns s = sg, sg + 8, sg + 16, sg + 24
        // (KDA built its decayed forms above)
        if constexpr (!KDA) {
            const int t = tid >> 3, sg = tid & 7;
            float kk[4] = {0.f, 0.f, 0.f, 0.f}, qk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int k = 0; k < PK; k += 4) {
                const float4 kt = *reinterpret_cast<const float4*>(Kc + t * KROW + k);
                const float4 qt = *reinterpret_cast<const float4*>(Qc + t * KROW + k);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 ks = *reinterpret_cast<const float4*>(Kc + (sg + 8 * j) * KROW + k);
                    if constexpr (FORM != FORM_LA)
                        kk[j] = fmaf(kt.w, ks.w, fmaf(kt.z, ks.z, fmaf(kt.y, ks.y, fmaf(kt.x, ks.x, kk[j]))));
                    qk[j] = fmaf(qt.w, ks.w, fmaf(qt.z, ks.z, fmaf(qt.y, ks.y, fmaf(qt.x, ks.x, qk[j]))));
                }
            }
            const float bt = Bt[t];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int s = sg + 8 * j;
                const float pd = M[t * TROW + s];   // decay table entry (0 above the diagonal)
                if constexpr (FORM != FORM_LA) A[t * TROW + s] = s < t ? bt * pd * kk[j] : 0.f;
                M[t * TROW + s] = pd * qk[j];
            }
        }
        __syncthreads();

        // ---- triangular solve, one value column per thread
        if constexpr (FORM != FORM_LA) {
            if (tid < VB) {
                float d[PC];
#pragma unroll
                for (int t = 0; t < PC; ++t) {
                    // two partial sums halve the dependent chain
                    float acc0 = D[t * VB + tid], acc1 = 0.f;
#pragma unroll
                    for (int s = 0; s + 1 < t; s += 2) {
                        acc0 = fmaf(-A[t * TROW + s], d[s], acc0);
                        acc1 = fmaf(-A[t * TROW + s + 1], d[s + 1], acc1);
                    }
                    if (t & 1) acc0 = fmaf(-A[t * TROW + t - 1], d[t - 1], acc0);
                    d[t] = acc0 + acc1;
                }
#pragma unroll
                for (int t = 0; t < PC; ++t) D[t * VB + tid] = d[t];
            }
            __syncthreads();
        }

        // ---- outputs o_t = E_t S0^T q_t + sum_{s<=t} P[t][s] (q_t . k_s) d_s
        {
#pragma unroll 4
            for (int s = 0; s < PC; ++s) {
                float2 dv[CP2];
#pragma unroll
                for (int c = 0; c < CP2; ++c) dv[c] = *reinterpret_cast<const float2*>(D + s * VB + CP * tx + 2 * c);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 m = dup(M[(4 * ty + i) * TROW + s]);
#pragma unroll
                    for (int c = 0; c < CP2; ++c) oq[i][c] = __ffma2_rn(m, dv[c], oq[i][c]);
                }
            }
            const bool obf = p.out_dt == LAR_BF16;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * ty + i;
                if (t < Lc) {
                    const int64_t base = (tb + c0 + t) * p.os[1] + static_cast<int64_t>(hv) * p.os[2];
#pragma unroll
                    for (int c = 0; c < CP2; ++c) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float o = e == 0 ? oq[i][c].x : oq[i][c].y;
                            const int64_t off = base + (v0 + CP * tx + 2 * c + e) * p.os[3];
                            if (obf) static_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(o * p.scale);
                            else static_cast<float*>(p.out)[off] = o * p.scale;
                        }
                    }
                }
            }
        }

        // ---- state update S = E_{C-1} S0 + sum_s P[C-1][s] k_s d_s^T: rows RK ky ..,
        // 8 columns 8 vx8 .. per thread
        {
            const int ky = tid / VX, vx8 = tid % VX;
            float2 acc[RK][4];
#pragma unroll
            for (int i = 0; i < RK; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
#pragma unroll 2
            for (int s = 0; s < PC; ++s) {
                // KDA: X holds P[C-1][s] o k_s, the scalar factor is 1
                const float2 ws = dup(KDA ? 1.f : Wd[s]);
                const float* krow = KDA ? X + s * PK : Kc + s * KROW;
                float kv[RK];
#pragma unroll
                for (int i4 = 0; i4 < RK / 4; ++i4) {
                    const float4 k4 = *reinterpret_cast<const float4*>(krow + RK * ky + 4 * i4);
                    kv[4 * i4] = k4.x;
                    kv[4 * i4 + 1] = k4.y;
                    kv[4 * i4 + 2] = k4.z;
                    kv[4 * i4 + 3] = k4.w;
                }
                const float4 d0 = *reinterpret_cast<const float4*>(D + s * VB + 8 * vx8);
                const float4 d1 = *reinterpret_cast<const float4*>(D + s * VB + 8 * vx8 + 4);
                const float2 dd[4] = {__fmul2_rn(ws, make_float2(d0.x, d0.y)), __fmul2_rn(ws, make_float2(d0.z, d0.w)),
                                      __fmul2_rn(ws, make_float2(d1.x, d1.y)), __fmul2_rn(ws, make_float2(d1.z, d1.w))};
#pragma unroll
                for (int i = 0; i < RK; ++i) {
                    const float2 k2 = dup(kv[i]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(k2, dd[j], acc[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < RK; ++i) {
                const float2 ec = dup(KDA ? EC[RK * ky + i] : E[PC - 1]);
                float4* sp = reinterpret_cast<float4*>(S + (RK * ky + i) * SROW + 8 * vx8);
                const float4 s0 = sp[0], s1 = sp[1];
                const float2 n0 = __ffma2_rn(ec, make_float2(s0.x, s0.y), acc[i][0]);
                const float2 n1 = __ffma2_rn(ec, make_float2(s0.z, s0.w), acc[i][1]);
                const float2 n2 = __ffma2_rn(ec, make_float2(s1.x, s1.y), acc[i][2]);
                const float2 n3 = __ffma2_rn(ec, make_float2(s1.z, s1.w), acc[i][3]);
                sp[0] = make_float4(n0.x, n0.y, n1.x, n1.y);
                sp[1] = make_float4(n2.x, n2.y, n3.x, n3.y);
            }
        }
        __syncthreads();
    }

    // ---- pool[w][hv][v0 + v][k] = S[k][v] (skipped for a negative or out-of-range slot)
    if (wr) {
        unsigned char* base =
            static_cast<unsigned char*>(p.pool) + (w * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1]) * SB;
        for (int i = tid; i < VB * NCHK; i += PTH) {
            const int v = i % VB;
            const int c = i / VB;
            uint4* dst = reinterpret_cast<uint4*>(base + static_cast<int64_t>(v0 + v) * p.ps[2] * SB) + c;
            if constexpr (SB == 4) {
                __stcs(dst, make_uint4(__float_as_uint(S[(c * 4) * SROW + v]), __float_as_uint(S[(c * 4 + 1) * SROW + v]),
                                       __float_as_uint(S[(c * 4 + 2) * SROW + v]),
                                       __float_as_uint(S[(c * 4 + 3) * SROW + v])));
            } else {
                unsigned wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 b2 =
                        __floats2bfloat162_rn(S[(c * 8 + 2 * e) * SROW + v], S[(c * 8 + 2 * e + 1) * SROW + v]);
                    wd[e] = *reinterpret_cast<const unsigned*>(&b2);
                }
                __stcs(dst, make_uint4(wd[0], wd[1], wd[2], wd[3]));
            }
        }
    }
}

template <int FORM, int SB>
lar_status launch_prefill_form(const DecodeParams& p, cudaStream_t stream) {
    constexpr int VB = LAR_PF_VB;
    auto kern = prefill_kernel<FORM, SB, VB>;
    constexpr size_t smem = PfLayout<VB, FORM == FORM_KDA>::BYTES;
    // the shared-memory opt-in is a per-device function attribute; setting it on
    // every call keeps it right on whichever device is current (a host-side
    // call, small next to a prefill launch)
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return LAR_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.HV) * (PV / VB), static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(PTH);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
#if LAR_PDL
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#endif
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? LAR_OK : LAR_ERR_LAUNCH;
}

}  // namespace

// 1: chunk products on the tensor cores (prefill_tc.cu, the default: 1.85x
// (GDN) and 2.2x (KDA) faster on 16 spans of 256-1024 tokens); 0: the CUDA-core
// form in this file, kept as the reference point of that comparison
#ifndef LAR_PF_TC
#define LAR_PF_TC 1
#endif

lar_status launch_prefill(const DecodeParams& p, void* stream) {
    if (p.K != PK || p.V != PV) return LAR_ERR_SHAPE;
    if (LAR_PF_TC) return launch_prefill_tc(p, stream);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = p.pool_dt == LAR_BF16;
    if (p.form == FORM_LA) return bf ? launch_prefill_form<FORM_LA, 2>(p, st) : launch_prefill_form<FORM_LA, 4>(p, st);
    if (p.form == FORM_GDN) return bf ? launch_prefill_form<FORM_GDN, 2>(p, st) : launch_prefill_form<FORM_GDN, 4>(p, st);
    if (p.form == FORM_KDA) return bf ? launch_prefill_form<FORM_KDA, 2>(p, st) : launch_prefill_form<FORM_KDA, 4>(p, st);
    return LAR_ERR_ARG;
}

}  // namespace lar
