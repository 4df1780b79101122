// prefill_tc.cu -- the chunked prefill (gated delta rule with scalar decay GDN
// or per-key-channel decay KDA, and Lightning Attention) with its matrix
// products on the tensor cores.
//
// Same operation and chunk algebra as prefill.cu (32-token chunks; with S0 the
// state entering a chunk, a_t the decay factors, P[t][s] = a_{s+1} ... a_t,
// E_t = a_0 ... a_t):
//     d_t + sum_{s<t} beta_t P[t][s] (k_t . k_s) d_s = beta_t (v_t - E_t S0^T k_t)
//     o_t = E_t S0^T q_t + sum_{s<=t} P[t][s] (q_t . k_s) d_s
//     S   = E_31 S0 + sum_s P[31][s] k_s d_s^T          (LA: d_t = v_t)
// written for the tensor cores in the transposed form, value channels as the
// 128 rows of every product:
//     [U | P] = S0^T [K ; Q]^T        (128 x 64, reduction over the 128 keys)
//     O       = D M^T                 (128 x 32, reduction over the chunk)
//     S^T    += (D o W) K             (128 x 128, reduction over the chunk)
// with D [v][s] = d_s[v], M[t][s] = P[t][s] (q_t . k_s) and W_s = P[31][s].
// KDA (a decay factor a_t[c] per key channel) takes the decays into the
// operand rows: E_t[c] k_t[c] and E_t[c] q_t[c] in the first product,
// P[31][s][c] k_s[c] in the update, diag(E_31) scaling the state's key
// columns, and A, M from per-channel decay products (running products over
// the chunk, no exponentials of differences), reduced across a warp.
//
// Precision.  The products run as tcgen05.mma kind::tf32 in three passes
// (A_hi B_hi + A_hi B_lo + A_lo B_hi, each operand split as x = hi + lo with hi
// the nearest tf32 value): about 2^-21 relative per product term, so the fp32
// state keeps the 1e-4 relative tolerance over thousands of tokens.  The
// dropped A_lo B_lo term is below 2^-22 relative.
//
// Two kernels.  prefill_ws_kernel (prefill_ws.cu: GDN and LA with staged bf16
// q / k / v rows, the usual case) splits each CTA into warps that run the state
// chain and warps that prepare the next chunk, on bf16 operands (fewer
// tensor-core instructions).  prefill_tc_kernel, here, runs KDA, fp32 q / k and
// other layouts:
//
// Work.  One CTA of 256 threads per (sequence, v-head) keeps that pair's state
// on chip for the whole span: S^T in fp32 registers (thread (warp w, lane l)
// owns value row v = 32 (w % 4) + l, the two warps of a row split its
// columns) and its tf32 halves in tensor memory (the A operand of the next
// chunk's first product).  The tensor cores produce each chunk's state
// increment on its own, which the threads add to the decayed state with
// round-to-nearest fp32 adds: accumulating into the state on the tensor cores,
// whose adds do not round to nearest, left a drift that grew with the span
// (4.7e-6 after 257 tokens at a decay of 0.996).  Per chunk: the chunk's k and q rows into
// shared memory (l2-normalised when asked, fp32 copies and tf32 halves in the
// K-major tile layout the tensor cores read), the per-token decays and betas;
// one thread issues [U | P] while the others compute K K^T and Q K^T on the
// CUDA cores (32 x 32, the decay table folded in); the triangular solve runs
// per value row in registers; D and D o W go to tensor memory; one thread
// issues O and the state increment (D o W) K; the outputs E_t P + O are
// stored, the state becomes E_31 S + increment and its tf32 halves are written
// back.  Tensor memory (512 columns): S_hi / S_lo (0..255; reused for D and
// D o W once [U | P] has read them), [U | P] (256..319; O takes U's half once the
// solve has read U), [K ; Q] K^T (320..351), the increment (384..511).
//
// Every wait is bounded: a wait that gives up makes the whole CTA skip the
// rest of its span and its writeback, and sets LAR_DEVERR_TIMEOUT.
#include "prefill_common.cuh"

namespace lar {
namespace {
using namespace pf;

constexpr int TTH = 256;      // threads per CTA
constexpr uint32_t KQ_SBO = (TK / 4) * LBO + 16;      // [K ; Q] tile: 64 rows x 128 keys
constexpr uint32_t KQ_BYTES = 8 * KQ_SBO;
constexpr uint32_t KT_SBO = (TC / 4) * LBO + 16;      // K^T tile: 128 keys x 32 tokens
constexpr uint32_t KT_BYTES = (TK / 8) * KT_SBO;
constexpr int FROW = TK + 4;                          // fp32 k / q rows (padded)

// shared memory, bytes
constexpr uint32_t OFF_KQH = 0;
constexpr uint32_t OFF_KQL = OFF_KQH + KQ_BYTES;
constexpr uint32_t OFF_KTH = OFF_KQL + KQ_BYTES;
constexpr uint32_t OFF_KTL = OFF_KTH + KT_BYTES;
constexpr uint32_t OFF_MTH = OFF_KTL + KT_BYTES;
constexpr uint32_t OFF_MTL = OFF_MTH + MT_BYTES;
constexpr uint32_t OFF_K32 = OFF_MTL + MT_BYTES;
constexpr uint32_t OFF_Q32 = OFF_K32 + TC * FROW * 4;
constexpr uint32_t OFF_A = OFF_Q32 + TC * FROW * 4;     // beta_t P[t][s] (k_t . k_s), s < t
constexpr uint32_t OFF_P = OFF_A + TC * TROW * 4;       // P[t][s]
constexpr uint32_t OFF_AF = OFF_P + TC * TROW * 4;      // a_t
constexpr uint32_t OFF_E = OFF_AF + TC * 4;             // E_t
constexpr uint32_t OFF_W = OFF_E + TC * 4;              // P[31][s]
constexpr uint32_t OFF_B = OFF_W + TC * 4;              // beta_t
constexpr uint32_t OFF_AD = OFF_B + TC * 4;             // KDA: a_t[c] [C][K]
constexpr uint32_t OFF_EC = OFF_AD + TC * TK * 4;       // KDA: E_31[c] [K]
// staging of one chunk's raw inputs (bf16 rows with unit inner stride and
// 16-byte aligned rows): q, k, v, the KDA gate rows, then the fp32 gate and beta
// scalars; filled with cp.async one chunk ahead
constexpr uint32_t STG_Q = 0, STG_K = TC * STG_ROW, STG_V = 2 * TC * STG_ROW, STG_G = 3 * TC * STG_ROW;
constexpr uint32_t STG_GS = 4 * TC * STG_ROW, STG_BS = STG_GS + TC * 4, STG_BYTES = STG_BS + TC * 4;
constexpr uint32_t OFF_STG = OFF_EC + TK * 4;
constexpr uint32_t OFF_BAR = OFF_STG + STG_BYTES;       // three mbarriers
constexpr uint32_t OFF_TM = OFF_BAR + 24;               // TMEM base address (then the picked sequence)
constexpr uint32_t TC_SMEM = OFF_TM + 16;
static_assert(OFF_KQL % 16 == 0 && OFF_KTH % 16 == 0 && OFF_KTL % 16 == 0 && OFF_MTH % 16 == 0 &&
                  OFF_MTL % 16 == 0 && OFF_K32 % 16 == 0 && OFF_Q32 % 16 == 0 && OFF_A % 16 == 0 &&
                  OFF_BAR % 8 == 0,
              "tile and barrier alignment");
static_assert(tc::kmaj(63, TK - 1, LBO, KQ_SBO) + 4 <= KQ_BYTES && tc::kmaj(TK - 1, TC - 1, LBO, KT_SBO) + 4 <= KT_BYTES &&
                  tc::kmaj(TC - 1, TC - 1, LBO, MT_SBO) + 4 <= MT_BYTES,
              "tiles hold their elements");
static_assert(TC_SMEM <= 227 * 1024, "fits one CTA's shared memory");
static_assert(OFF_STG % 16 == 0 && TVV == TK, "staging rows are 16-byte aligned");
static_assert(kLptMax * 4 <= STG_BYTES, "the span lengths fit the staging buffer");

// tensor-memory columns
constexpr uint32_t COL_SHI = 0, COL_SLO = 128;   // the state's tf32 halves; COL_UP, COL_KK, COL_DS as shared
// O takes U's columns (U is dead once the solve has read it), so the new state's
// halves (0..255) can be written while O is still being read
constexpr uint32_t COL_DHI = 0, COL_DLO = 32, COL_DWHI = 64, COL_DWLO = 96, COL_O = COL_UP;

// ---- the chunk's products, each issued by one thread in three tf32 passes
// [K ; Q] K^T into COL_KK (M = 64: rows 0..31 K K^T, rows 32..63 Q K^T; N = 32)
__device__ __forceinline__ void issue_kk(uint32_t tm, uint32_t kqh, uint32_t kql) {
    constexpr uint32_t idesc_kk = tc::idesc_tf32(64, TC);
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
        const uint32_t ab = ps == 2 ? kql : kqh, bb = ps == 1 ? kql : kqh;
#pragma unroll 1
        for (int kb = 0; kb < TK / 8; ++kb)
            tc::mma_ss(tm + COL_KK, tc::smem_desc(ab + kb * 2 * LBO, LBO, KQ_SBO),
                       tc::smem_desc(bb + kb * 2 * LBO, LBO, KQ_SBO), idesc_kk, ps > 0 || kb > 0);
    }
}

// [U | P] = S^T [K ; Q]^T into COL_UP from the state's tf32 halves (COL_SHI,
// COL_SLO); LA needs P only (the q rows, into COL_UP + TC)
template <bool LA>
__device__ __forceinline__ void issue_up(uint32_t tm, uint32_t kqh, uint32_t kql) {
    constexpr int NUP = LA ? TC : 2 * TC;
    constexpr uint32_t idesc = tc::idesc_tf32(TVV, NUP);
    const uint32_t boff = LA ? 4 * KQ_SBO : 0;
    const uint32_t dcol = tm + COL_UP + (LA ? TC : 0);
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
        const uint32_t acol = tm + (ps == 2 ? COL_SLO : COL_SHI);
        const uint32_t bb = (ps == 1 ? kql : kqh) + boff;
#pragma unroll 1
        for (int kb = 0; kb < TK / 8; ++kb)
            tc::mma_ts(dcol, acol + 8 * kb, tc::smem_desc(bb + kb * 2 * LBO, LBO, KQ_SBO), idesc, ps > 0 || kb > 0);
    }
}

// O = D M^T into COL_O and the increment (D o W) K into COL_DS, from D and
// D o W in tensor memory and the M and K^T tiles
__device__ __forceinline__ void issue_os(uint32_t tm, uint32_t mth, uint32_t mtl, uint32_t kth, uint32_t ktl) {
    constexpr uint32_t idesc_o = tc::idesc_tf32(TVV, TC);
    constexpr uint32_t idesc_s = tc::idesc_tf32(TVV, TK);
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
        const uint32_t ad = tm + (ps == 2 ? COL_DLO : COL_DHI);
        const uint32_t aw = tm + (ps == 2 ? COL_DWLO : COL_DWHI);
        const uint32_t bm = ps == 1 ? mtl : mth;
        const uint32_t bk = ps == 1 ? ktl : kth;
#pragma unroll 1
        for (int kb = 0; kb < TC / 8; ++kb) {
            tc::mma_ts(tm + COL_O, ad + 8 * kb, tc::smem_desc(bm + kb * 2 * LBO, LBO, MT_SBO), idesc_o, ps > 0 || kb > 0);
            tc::mma_ts(tm + COL_DS, aw + 8 * kb, tc::smem_desc(bk + kb * 2 * LBO, LBO, KT_SBO), idesc_s,
                       ps > 0 || kb > 0);
        }
    }
}

// token t's k and q values (this lane's 4 channels, c = 4 lane ..) into the
// [K ; Q] tile and the K^T tile as tf32 halves
__device__ __forceinline__ void put_kq(unsigned char* kqh, unsigned char* kql, unsigned char* kth,
                                       unsigned char* ktl, int t, int lane, const float* kx, const float* qx) {
    float kh[4], kl[4], qh[4], ql[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        kh[e] = tc::tf32_hi(kx[e]);
        kl[e] = kx[e] - kh[e];
        qh[e] = tc::tf32_hi(qx[e]);
        ql[e] = qx[e] - qh[e];
    }
    const uint32_t ok_ = tc::kmaj(t, 4 * lane, LBO, KQ_SBO), oq_ = tc::kmaj(TC + t, 4 * lane, LBO, KQ_SBO);
    *reinterpret_cast<float4*>(kqh + ok_) = make_float4(kh[0], kh[1], kh[2], kh[3]);
    *reinterpret_cast<float4*>(kql + ok_) = make_float4(kl[0], kl[1], kl[2], kl[3]);
    *reinterpret_cast<float4*>(kqh + oq_) = make_float4(qh[0], qh[1], qh[2], qh[3]);
    *reinterpret_cast<float4*>(kql + oq_) = make_float4(ql[0], ql[1], ql[2], ql[3]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t o = tc::kmaj(4 * lane + e, t, LBO, KT_SBO);
        *reinterpret_cast<float*>(kth + o) = kh[e];
        *reinterpret_cast<float*>(ktl + o) = kl[e];
    }
}

// l2-normalise a token's q and k rows held 4 channels per lane across a warp
__device__ __forceinline__ void l2_rows(float* qx, float* kx) {
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        sq = fmaf(qx[e], qx[e], sq);
        sk = fmaf(kx[e], kx[e], sk);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
    }
    const float iq = 1.f / sqrtf(sq + 1e-6f), ik = 1.f / sqrtf(sk + 1e-6f);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        qx[e] *= iq;
        kx[e] *= ik;
    }
}

// The A and M tables from the [K ; Q] K^T rows a warp of quarter `quarter`
// holds (x: its lane's 32 columns; lanes 0..15 hold rows): A[t][s] = beta_t
// P[t][s] (k_t . k_s) (s < t) from quarters 0, 1; M[t][s] = P[t][s] (q_t . k_s)
// as tf32 halves in the M tile from quarters 2, 3.
template <bool WITH_A>
__device__ __forceinline__ void kk_tables(int quarter, int lane, const float* x, const float* Pt, const float* Bt,
                                          float* At, unsigned char* mth, unsigned char* mtl) {
    if (lane >= 16) return;
    const int t = 16 * (quarter & 1) + lane;
    const float* pr = Pt + t * TROW;
    if (quarter < 2) {
        if constexpr (WITH_A) {
            const float bt = Bt[t];
#pragma unroll
            for (int s4 = 0; s4 < TC; s4 += 4)
                *reinterpret_cast<float4*>(At + t * TROW + s4) =
                    make_float4(s4 < t ? bt * pr[s4] * x[s4] : 0.f, s4 + 1 < t ? bt * pr[s4 + 1] * x[s4 + 1] : 0.f,
                                s4 + 2 < t ? bt * pr[s4 + 2] * x[s4 + 2] : 0.f,
                                s4 + 3 < t ? bt * pr[s4 + 3] * x[s4 + 3] : 0.f);
        }
    } else {
#pragma unroll
        for (int s4 = 0; s4 < TC; s4 += 4) {
            float m[4], mh[4], ml[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                m[e] = pr[s4 + e] * x[s4 + e];
                mh[e] = tc::tf32_hi(m[e]);
                ml[e] = m[e] - mh[e];
            }
            const uint32_t o = tc::kmaj(t, s4, LBO, MT_SBO);
            *reinterpret_cast<float4*>(mth + o) = make_float4(mh[0], mh[1], mh[2], mh[3]);
            *reinterpret_cast<float4*>(mtl + o) = make_float4(ml[0], ml[1], ml[2], ml[3]);
        }
    }
}

// The triangular solve of one value row: d_t = beta_t (v_t - E_t u_t) -
// sum_{s<t} A[t][s] d_s, with u (= (S0^T k_t)[v]) read from tensor memory and
// v_t from vin(t), 16 tokens at a time.  Four partial sums shorten the
// dependent chain.
template <typename VIn>
__device__ __forceinline__ void solve_row(uint32_t u_taddr, VIn vin, const float* At, const float* Bt,
                                          const float* E, float* d) {
#pragma unroll
    for (int t0 = 0; t0 < TC; t0 += 16) {
        float u[16], vv[16];
        tc::tmem_ld16(u_taddr + t0, u);
#pragma unroll
        for (int i = 0; i < 16; ++i) vv[i] = vin(t0 + i);
        tc::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int t = t0 + i;
            float acc0 = Bt[t] * fmaf(-E[t], u[i], vv[i]), acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
            for (int s = 0; s < (t & ~3); s += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(At + t * TROW + s);
                acc0 = fmaf(-a4.x, d[s], acc0);
                acc1 = fmaf(-a4.y, d[s + 1], acc1);
                acc2 = fmaf(-a4.z, d[s + 2], acc2);
                acc3 = fmaf(-a4.w, d[s + 3], acc3);
            }
#pragma unroll
            for (int s = t & ~3; s < t; ++s) acc0 = fmaf(-At[t * TROW + s], d[s], acc0);
            d[t] = (acc0 + acc1) + (acc2 + acc3);
        }
    }
}

template <int FORM, int SB>
__global__ void __launch_bounds__(TTH, 1) prefill_tc_kernel(const DecodeParams p) {
    constexpr bool LA = FORM == FORM_LA;
    constexpr bool KDA = FORM == FORM_KDA;
    extern __shared__ __align__(1024) unsigned char smem[];
    float* K32 = reinterpret_cast<float*>(smem + OFF_K32);
    float* Q32 = reinterpret_cast<float*>(smem + OFF_Q32);
    float* At = reinterpret_cast<float*>(smem + OFF_A);
    float* Pt = reinterpret_cast<float*>(smem + OFF_P);
    float* Af = reinterpret_cast<float*>(smem + OFF_AF);
    float* E = reinterpret_cast<float*>(smem + OFF_E);
    float* Wd = reinterpret_cast<float*>(smem + OFF_W);
    float* Bt = reinterpret_cast<float*>(smem + OFF_B);
    float* Ad = reinterpret_cast<float*>(smem + OFF_AD);       // KDA only
    float* EC = reinterpret_cast<float*>(smem + OFF_EC);       // KDA only
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tm_slot = reinterpret_cast<uint32_t*>(smem + OFF_TM);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quarter = warp & 3, half = warp >> 2;
    const int vrow = quarter * 32 + lane;                      // this thread's value row (TMEM lane)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int hv = blockIdx.x;
    const int h = hv / p.group;

#if LAR_PDL
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif
    // ---- which sequence: longest spans first; in a split variable-length call
    // only the long ones (pick_sequence); the staging buffer is not in use yet
    const int n = pick_sequence<TTH>(p, reinterpret_cast<int*>(smem + OFF_STG),
                                      reinterpret_cast<int*>(smem + OFF_TM) + 1);
    if (n < 0) return;
    // ---- span and slots (reversed or overlong spans run as empty and are flagged)
    const int64_t lo = ld_idx(p.cu, n * p.cu_s, p.cu_dt);
    const int64_t hi = ld_idx(p.cu, (n + 1) * p.cu_s, p.cu_dt);
    const bool span_ok = lo >= 0 && hi >= lo && hi <= p.ntok;
    const int64_t tb = span_ok ? lo : 0;
    const int64_t L = span_ok ? hi - lo : 0;
    // a variable-length call sends only its long spans here (the rest run token by token)
    if (p.split_len > 0 && L < p.split_len) return;
    const int64_t r = ld_idx(p.ridx, n * p.ri_s, p.ri_dt);
    const int64_t w = p.widx ? ld_idx(p.widx, n * p.wi_s, p.wi_dt) : r;
    const bool rd = r >= 0 && r < p.P;
    const bool wr = w >= 0 && w < p.P;
    if (tid == 0 && blockIdx.x == 0 && p.dev_err) {
        const int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0) |
                      (span_ok ? 0 : LAR_DEVERR_SEQLEN);
        if (e) atomicOr(p.dev_err, e);
    }

    if (tid == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        tc::mbar_init(&bar[2], 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tm_slot, TMEM_COLS);
    tc_sync();
    const uint32_t tm = *tm_slot;
    const uint32_t my = tm + lane_off;                         // this thread's lane, column 0
    const int col0 = 64 * half;                                // this thread's 64 state columns

    // ---- S0: this thread's 64 state values (row vrow, columns col0 ..) into
    // registers, its tf32 halves into tensor memory
    float S[64];
    {
        const unsigned char* src = static_cast<const unsigned char*>(p.pool) +
                                   ((rd ? r : 0) * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1] +
                                    static_cast<int64_t>(vrow) * p.ps[2] + col0) * SB;
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
            float* x = S + c;
            if (rd) {
                if constexpr (SB == 4) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f = __ldg(reinterpret_cast<const float4*>(src + c * 4) + i);
                        x[4 * i] = f.x; x[4 * i + 1] = f.y; x[4 * i + 2] = f.z; x[4 * i + 3] = f.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const uint4 u = __ldg(reinterpret_cast<const uint4*>(src + c * 2) + i);
                        const unsigned wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            x[8 * i + 2 * e] = __uint_as_float(wd[e] << 16);
                            x[8 * i + 2 * e + 1] = __uint_as_float(wd[e] & 0xffff0000u);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = 0.f;
            }
        }
        split_store<64>(my + COL_SHI + col0, my + COL_SLO + col0, S);
        tc::tmem_st_wait();
    }
    tc_sync();

    const bool l2 = !LA && (p.flags & LAR_QK_L2NORM) != 0;
    const bool gate_raw = (p.flags & LAR_GATE_RAW) != 0;
    const bool beta_raw = (p.flags & LAR_BETA_RAW) != 0;
    const uint32_t kqh = tc::smem_addr(smem + OFF_KQH), kql = tc::smem_addr(smem + OFF_KQL);
    const uint32_t kth = tc::smem_addr(smem + OFF_KTH), ktl = tc::smem_addr(smem + OFF_KTL);
    const uint32_t mth = tc::smem_addr(smem + OFF_MTH), mtl = tc::smem_addr(smem + OFF_MTL);
    // Inputs staged through shared memory when every row is bf16 with unit inner
    // stride and 16-byte aligned (each row a run of 16-byte chunks); other
    // layouts are read element by element (same results).
    auto rows16 = [](const void* base, int dt, const int64_t* st, int n) {
        bool okr = dt == LAR_BF16 && st[3] == 1 && (reinterpret_cast<uintptr_t>(base) & 15) == 0;
        for (int i = 1; i < n; ++i) okr = okr && (st[i] * 2) % 16 == 0;
        return okr;
    };
    const bool staged = rows16(p.q, p.q_dt, p.qs, 3) && rows16(p.k, p.k_dt, p.ks, 3) && rows16(p.v, p.v_dt, p.vs, 3) &&
                        (!KDA || rows16(p.g, p.g_dt, p.gs, 3));
    const bool stage_scal = !LA && !KDA && p.g_dt == LAR_F32 && p.beta_dt == LAR_F32;
    const bool stage_beta = KDA && p.beta_dt == LAR_F32;
    unsigned char* stg = smem + OFF_STG;
    // issue this thread's copies of the chunk that starts at token cs of the span
    auto stage = [&](int64_t cs) {
        const int Ln = static_cast<int>(L - cs < TC ? L - cs : TC);
        constexpr int NR = KDA ? 4 : 3;
#pragma unroll 1
        for (int i = tid; i < NR * TC * 16; i += TTH) {
            const int which = i / (TC * 16), rem = i - which * (TC * 16), t = rem >> 4, c = rem & 15;
            if (t >= Ln) continue;
            const int64_t gt = tb + cs + t;
            const unsigned char* src;
            if (which == 0) src = static_cast<const unsigned char*>(p.q) + (gt * p.qs[1] + h * p.qs[2]) * 2;
            else if (which == 1) src = static_cast<const unsigned char*>(p.k) + (gt * p.ks[1] + h * p.ks[2]) * 2;
            else if (which == 2)
                src = static_cast<const unsigned char*>(p.v) + (gt * p.vs[1] + static_cast<int64_t>(hv) * p.vs[2]) * 2;
            else
                src = static_cast<const unsigned char*>(p.g) + (gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2]) * 2;
            cp_async16(stg + which * (TC * STG_ROW) + t * STG_ROW + c * 16, src + c * 16);
        }
        if ((stage_scal || stage_beta) && tid < TC && tid < Ln) {
            const int64_t gt = tb + cs + tid;
            if (stage_scal)
                cp_async4(stg + STG_GS + tid * 4, static_cast<const float*>(p.g) + gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2]);
            cp_async4(stg + STG_BS + tid * 4,
                      static_cast<const float*>(p.beta) + gt * p.bs[1] + static_cast<int64_t>(hv) * p.bs[2]);
        }
        cp_async_commit();
    };
    if (staged && L > 0) stage(0);

    bool ok = true;
    int chunk = 0;
    // KDA gate chain constants of this head and of this lane's four key channels
    float negA = 0.f, bias4[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (KDA) {
        if (gate_raw) {
            negA = -expf(p.A_log[hv * p.A_s]);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                bias4[e] = p.dt_bias ? p.dt_bias[(static_cast<int64_t>(hv) * TK + lane * 4 + e) * p.dtb_s] : 0.f;
        }
    }

#pragma unroll 1
    for (int64_t c0 = 0; c0 < L; c0 += TC, ++chunk) {
        const int Lc = static_cast<int>(L - c0 < TC ? L - c0 : TC);
        const uint32_t par = static_cast<uint32_t>(chunk & 1);

        // ---- (1) the chunk's inputs: staged ones have landed (this thread's copies,
        // then everyone's through the barrier)
        if (staged) {
            cp_async_wait<0>();
            __syncthreads();
        }
        // value inputs of this thread's row (the solve's right-hand side; LA: d itself)
        float vv[TC];
        if (half == 0) {
            if (staged) {
                const unsigned short* sv = reinterpret_cast<const unsigned short*>(stg + STG_V) + vrow;
#pragma unroll
                for (int t = 0; t < TC; ++t) vv[t] = t < Lc ? bf16_bits_to_float(sv[t * TK]) : 0.f;
            } else {
#pragma unroll
                for (int t = 0; t < TC; ++t)
                    vv[t] = t < Lc ? ld_in(p.v, (tb + c0 + t) * p.vs[1] + static_cast<int64_t>(hv) * p.vs[2] +
                                                    static_cast<int64_t>(vrow) * p.vs[3], p.v_dt)
                                   : 0.f;
            }
        }
        // k and q rows: warp w takes tokens w, w + 8, ...; lane l channels 4l .. 4l + 3.
        // All of a thread's loads are issued before any is used.
        constexpr int RPW = TC / (TTH / 32);
        float qa[RPW][4], ka[RPW][4], ga[KDA ? RPW : 1][4];
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const int t = warp + j * (TTH / 32);
            const int64_t gt = tb + c0 + t;
            const int64_t c = lane * 4;
            if (t < Lc && staged) {
                auto widen = [&](uint32_t off, float* x) {
                    const uint2 u = *reinterpret_cast<const uint2*>(stg + off + t * STG_ROW + lane * 8);
                    x[0] = __uint_as_float(u.x << 16);
                    x[1] = __uint_as_float(u.x & 0xffff0000u);
                    x[2] = __uint_as_float(u.y << 16);
                    x[3] = __uint_as_float(u.y & 0xffff0000u);
                };
                widen(STG_Q, qa[j]);
                widen(STG_K, ka[j]);
                if constexpr (KDA) widen(STG_G, ga[j]);
            } else if (t < Lc) {
                ld_in4(p.q, gt * p.qs[1] + h * p.qs[2] + c * p.qs[3], p.qs[3], p.q_dt, qa[j]);
                ld_in4(p.k, gt * p.ks[1] + h * p.ks[2] + c * p.ks[3], p.ks[3], p.k_dt, ka[j]);
                if constexpr (KDA)
                    ld_in4(p.g, gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2] + c * p.gs[3], p.gs[3], p.g_dt,
                           ga[j]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qa[j][e] = ka[j][e] = 0.f;
                    if constexpr (KDA) ga[j][e] = 0.f;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < RPW; ++j) {
            const int t = warp + j * (TTH / 32);
            const bool tok = t < Lc;
            float* qx = qa[j];
            float* kx = ka[j];
            const float* gk = ga[KDA ? j : 0];
            if constexpr (KDA) {
                // per-channel decay factors a_t[c] (gate chain included); padding tokens: 1
                float a4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x = gk[e];
                    if (gate_raw) x = negA * softplus_f(x + bias4[e]);
                    a4[e] = tok ? expf(x) : 1.f;
                }
                *reinterpret_cast<float4*>(Ad + t * TK + 4 * lane) = make_float4(a4[0], a4[1], a4[2], a4[3]);
            }
            if (l2) l2_rows(qx, kx);
            *reinterpret_cast<float4*>(K32 + t * FROW + 4 * lane) = make_float4(kx[0], kx[1], kx[2], kx[3]);
            *reinterpret_cast<float4*>(Q32 + t * FROW + 4 * lane) = make_float4(qx[0], qx[1], qx[2], qx[3]);
            if constexpr (!KDA)       // KDA's operand rows carry the decays: written below
                put_kq(smem + OFF_KQH, smem + OFF_KQL, smem + OFF_KTH, smem + OFF_KTL, t, lane, kx, qx);
        }
        // decay factors and betas (warp 1, lane t); the decay table is built from them
        // while the tensor cores run
        if (warp == 1) {
            const int t = lane;
            float a = 1.f, bt = 0.f;   // padding tokens: no decay, no update
            if (t < Lc) {
                const int64_t gt = tb + c0 + t;
                if constexpr (LA) {
                    a = p.decay[h * p.dec_s];
                    bt = 1.f;
                } else {
                    if constexpr (!KDA) {   // KDA: the decay is per channel (Ad), the scalar factor 1
                        float x = staged && stage_scal ? reinterpret_cast<const float*>(stg + STG_GS)[t]
                                                       : ld_in(p.g, gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2], p.g_dt);
                        if (gate_raw) {
                            const float bias = p.dt_bias ? p.dt_bias[hv * p.dtb_s] : 0.f;
                            x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
                        }
                        a = expf(x);
                    }
                    const float bx = staged && (stage_scal || stage_beta)
                                         ? reinterpret_cast<const float*>(stg + STG_BS)[t]
                                         : ld_in(p.beta, gt * p.bs[1] + static_cast<int64_t>(hv) * p.bs[2], p.beta_dt);
                    bt = beta_raw ? 1.f / (1.f + expf(-bx)) : bx;
                }
            }
            Af[t] = a;
            Bt[t] = bt;
        }
        if constexpr (KDA) {
            __syncthreads();
            // ---- (1b) KDA: A[t][s] = beta_t sum_c k_t[c] k_s[c] P[t][s][c] (s < t) and
            // M[t][s] = sum_c q_t[c] k_s[c] P[t][s][c] (s <= t), P[t][s][c] = a_{s+1}[c] ... a_t[c]
            // kept as a running product over t (factors <= 1: nothing overflows).  Warp w
            // takes its four s = w, w + 8, w + 16, w + 24 together, so each token row is read
            // once per warp; lane l channels 4l .. 4l + 3.  Over a block of 8 tokens each lane
            // holds 64 partial sums, value j = 16 i + 2 tt + kind for s_i, t = 8 b + tt and
            // kind 0 (A) / 1 (M); recursive halving across the warp leaves lane l holding
            // j = 2l and 2l + 1: the pair (t = 8 b + l % 8, s = w + 8 (l / 8)).
            static_assert(TC == 32 && TTH == 256, "8 warps x 4 s-values; 4 blocks of 8 tokens");
            {
                float4 ks[4], pr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    ks[i] = *reinterpret_cast<const float4*>(K32 + (warp + 8 * i) * FROW + 4 * lane);
                    pr[i] = make_float4(1.f, 1.f, 1.f, 1.f);
                }
#pragma unroll 1
                for (int b8 = 0; b8 < TC / 8; ++b8) {
                    float v[64];
#pragma unroll
                    for (int tt = 0; tt < 8; ++tt) {
                        const int t = 8 * b8 + tt;
                        const float4 a4 = *reinterpret_cast<const float4*>(Ad + t * TK + 4 * lane);
                        const float4 kt = *reinterpret_cast<const float4*>(K32 + t * FROW + 4 * lane);
                        const float4 qt = *reinterpret_cast<const float4*>(Q32 + t * FROW + 4 * lane);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int si = warp + 8 * i;
                            if (t > si) pr[i] = make_float4(pr[i].x * a4.x, pr[i].y * a4.y, pr[i].z * a4.z, pr[i].w * a4.w);
                            const float wx = ks[i].x * pr[i].x, wy = ks[i].y * pr[i].y, wz = ks[i].z * pr[i].z,
                                        ww = ks[i].w * pr[i].w;
                            const bool on = t >= si;
                            v[16 * i + 2 * tt] = on ? fmaf(kt.w, ww, fmaf(kt.z, wz, fmaf(kt.y, wy, kt.x * wx))) : 0.f;
                            v[16 * i + 2 * tt + 1] = on ? fmaf(qt.w, ww, fmaf(qt.z, wz, fmaf(qt.y, wy, qt.x * wx))) : 0.f;
                        }
                    }
#pragma unroll
                    for (int half = 32, lb = 16; half >= 2; half >>= 1, lb >>= 1) {
                        const bool up = (lane & lb) != 0;
#pragma unroll
                        for (int i = 0; i < half; ++i) {
                            const float send = up ? v[i] : v[i + half];
                            const float keep = up ? v[i + half] : v[i];
                            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, lb);
                        }
                    }
                    const int t = 8 * b8 + (lane & 7), s = warp + 8 * (lane >> 3);
                    At[t * TROW + s] = t > s ? Bt[t] * v[0] : 0.f;
                    const float m = t >= s ? v[1] : 0.f;
                    const float mh = tc::tf32_hi(m);
                    const uint32_t o = tc::kmaj(t, s, LBO, MT_SBO);
                    *reinterpret_cast<float*>(smem + OFF_MTH + o) = mh;
                    *reinterpret_cast<float*>(smem + OFF_MTL + o) = m - mh;
                }
            }
            // per channel c: the update's rows P[31][s][c] k_s[c] (a running product from the
            // chunk's end; threads 0..127), the first product's rows E_t[c] k_t[c] and
            // E_t[c] q_t[c], and E_31[c] (threads 128..255)
            static_assert(TTH == 2 * TK, "one thread per channel for each half of the tiles");
            if (tid < TK) {
                const int c = tid;
                float wv = 1.f;
#pragma unroll 4
                for (int s2 = TC - 1; s2 >= 0; --s2) {
                    const float x = K32[s2 * FROW + c] * wv;
                    const float xh = tc::tf32_hi(x);
                    const uint32_t o = tc::kmaj(c, s2, LBO, KT_SBO);
                    *reinterpret_cast<float*>(smem + OFF_KTH + o) = xh;
                    *reinterpret_cast<float*>(smem + OFF_KTL + o) = x - xh;
                    wv *= Ad[s2 * TK + c];
                }
            } else {
                const int c = tid - TK;
                float ev = 1.f;
#pragma unroll 4
                for (int t = 0; t < TC; ++t) {
                    ev *= Ad[t * TK + c];
                    const float xk = K32[t * FROW + c] * ev, xq = Q32[t * FROW + c] * ev;
                    const float kh = tc::tf32_hi(xk), qh = tc::tf32_hi(xq);
                    const uint32_t ok_ = tc::kmaj(t, c, LBO, KQ_SBO), oq_ = tc::kmaj(TC + t, c, LBO, KQ_SBO);
                    *reinterpret_cast<float*>(smem + OFF_KQH + ok_) = kh;
                    *reinterpret_cast<float*>(smem + OFF_KQL + ok_) = xk - kh;
                    *reinterpret_cast<float*>(smem + OFF_KQH + oq_) = qh;
                    *reinterpret_cast<float*>(smem + OFF_KQL + oq_) = xq - qh;
                }
                EC[c] = ev;
            }
        }
        tc::fence_smem_to_async();
        tc_sync();
        // the staging buffer has been read: the next chunk's copies go out now
        if (staged && c0 + TC < L) stage(c0 + TC);

        // ---- (2) [K ; Q] K^T (GDN, LA; completes on bar[0]), then [U | P] = S0^T [K ; Q]^T
        // (LA: P only; completes on bar[2]), three tf32 passes each
        if (tid == 0) {
            if constexpr (!KDA) {
                issue_kk(tm, kqh, kql);
                tc::mma_commit(&bar[0]);
            }
            issue_up<LA>(tm, kqh, kql);
            tc::mma_commit(&bar[2]);
        }
        if (warp == 1) decay_table(lane, Af, Pt, E, Wd);

        // ---- (3) wait for [K ; Q] K^T (GDN, LA), the A and M tables from it while
        // [U | P] still runs, then wait for [U | P]
        if constexpr (!KDA) {
            ok = tc::mbar_wait(&bar[0], par);
            ok = !__syncthreads_or(!ok);
            if (!ok) break;
            tc::fence_after_sync();
        } else {
            __syncthreads();   // the decay table (all ones for KDA: its decays sit in the operand rows)
        }
        if (!KDA && half == 0) {
            // rows of K K^T (quarters 0, 1) and Q K^T (quarters 2, 3) with the decay table
            float x[TC];
            tc::tmem_ld16(my + COL_KK, x);
            tc::tmem_ld16(my + COL_KK + 16, x + 16);
            tc::tmem_ld_wait();
            kk_tables<!LA>(quarter, lane, x, Pt, Bt, At, smem + OFF_MTH, smem + OFF_MTL);
        }
        tc::fence_smem_to_async();
        ok = tc::mbar_wait(&bar[2], par);
        ok = !__syncthreads_or(!ok);
        if (!ok) break;
        tc::fence_after_sync();
        float pv[TC];
        if (half == 1) {
#pragma unroll
            for (int c = 0; c < TC; c += 16) tc::tmem_ld16(my + COL_UP + TC + c, pv + c);
            tc::tmem_ld_wait();
        }

        // ---- (4) the solve per value row, D and D o W into tensor memory
        if (half == 0) {
            float d[TC];
            if constexpr (LA) {
#pragma unroll
                for (int t = 0; t < TC; ++t) d[t] = vv[t];
            } else {
                solve_row(my + COL_UP, [&](int t) { return vv[t]; }, At, Bt, E, d);
            }
            split_store<TC>(my + COL_DHI, my + COL_DLO, d);
#pragma unroll
            for (int t = 0; t < TC; ++t) d[t] *= Wd[t];
            split_store<TC>(my + COL_DWHI, my + COL_DWLO, d);
            tc::tmem_st_wait();
        }
        tc_sync();

        // ---- (5) O = D M^T and the increment (D o W) K, three tf32 passes each
        if (tid == 0) {
            issue_os(tm, mth, mtl, kth, ktl);
            tc::mma_commit(&bar[1]);
        }
        ok = tc::mbar_wait(&bar[1], par);
        ok = !__syncthreads_or(!ok);
        if (!ok) break;
        tc::fence_after_sync();

        // ---- (6) outputs o_t = E_t P[v][t] + O[v][t] (half 1), then the new state's tf32 halves
        if (half == 1) {
            float o[TC];
#pragma unroll
            for (int c = 0; c < TC; c += 16) tc::tmem_ld16(my + COL_O + c, o + c);
            tc::tmem_ld_wait();
            const bool obf = p.out_dt == LAR_BF16;
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                if (t < Lc) {
                    const float y = fmaf(E[t], pv[t], o[t]) * p.scale;
                    const int64_t off = (tb + c0 + t) * p.os[1] + static_cast<int64_t>(hv) * p.os[2] +
                                        static_cast<int64_t>(vrow) * p.os[3];
                    if (obf) static_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(y);
                    else static_cast<float*>(p.out)[off] = y;
                }
            }
        }
        // the new state E_31 S + increment (KDA: E_31 per key column), rounded to
        // nearest, and its tf32 halves for the next chunk's first product
        {
            const float ec = E[TC - 1];
            const bool more = c0 + TC < L;
#pragma unroll
            for (int c = 0; c < 64; c += 16) {
                float x[16];
                tc::tmem_ld16(my + COL_DS + col0 + c, x);
                tc::tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) S[c + i] = fmaf(KDA ? EC[col0 + c + i] : ec, S[c + i], x[i]);
                if (more) split_store<16>(my + COL_SHI + col0 + c, my + COL_SLO + col0 + c, S + c);
            }
            if (more) tc::tmem_st_wait();
        }
        tc_sync();
    }

    cp_async_wait<0>();   // nothing may be left in flight into shared memory at exit
    if (!ok) {
        if (tid == 0 && p.dev_err) atomicOr(p.dev_err, LAR_DEVERR_TIMEOUT);
    } else if (wr) {
        // ---- pool[w][hv][v][k] = S^T[v][k]
        unsigned char* dst = static_cast<unsigned char*>(p.pool) +
                             (w * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1] + static_cast<int64_t>(vrow) * p.ps[2] +
                              col0) * SB;
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
            const float* x = S + c;
            if constexpr (SB == 4) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    __stcs(reinterpret_cast<float4*>(dst + c * 4) + i,
                           make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]));
            } else {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    unsigned wd[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(x[8 * i + 2 * e], x[8 * i + 2 * e + 1]);
                        wd[e] = *reinterpret_cast<const unsigned*>(&b2);
                    }
                    __stcs(reinterpret_cast<uint4*>(dst + c * 2) + i, make_uint4(wd[0], wd[1], wd[2], wd[3]));
                }
            }
        }
    }
    tc_sync();
    if (warp == 0) tc::tmem_dealloc(tm, TMEM_COLS);
}



// GDN and LA with bf16 q / k / v rows that can be staged run in the
// warp-specialised kernel (prefill_ws.cu); KDA (whose per-channel tables need
// the shared memory that kernel's second buffers take), fp32 q or k (not exact
// in tf32) and other layouts here.  The build flag LAR_PF_WS=0 runs everything
// here.
#ifndef LAR_PF_WS
#define LAR_PF_WS 1
#endif
template <int FORM, int SB>
lar_status launch_tc_form(const DecodeParams& p, cudaStream_t stream) {
#if LAR_PF_WS
    if constexpr (FORM != FORM_KDA) {
        // every q / k / v row bf16 with unit inner stride, starting on a 16-byte boundary
        auto rows16 = [](const void* base, int dt, const int64_t* st) {
            return dt == LAR_BF16 && st[3] == 1 && (reinterpret_cast<uintptr_t>(base) & 15) == 0 &&
                   (st[1] * 2) % 16 == 0 && (st[2] * 2) % 16 == 0;
        };
        if (rows16(p.q, p.q_dt, p.qs) && rows16(p.k, p.k_dt, p.ks) && rows16(p.v, p.v_dt, p.vs)) {
            bool launched = false;
            const lar_status st = launch_prefill_ws(p, stream, &launched);
            if (launched) return st;
        }
    }
#endif
    return launch_kernel(prefill_tc_kernel<FORM, SB>, TTH, TC_SMEM, p, p, stream);
}

}  // namespace

lar_status launch_prefill_tc(const DecodeParams& p, void* stream) {
    if (p.K != TK || p.V != TVV) return LAR_ERR_SHAPE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = p.pool_dt == LAR_BF16;
    if (p.form == FORM_LA) return bf ? launch_tc_form<FORM_LA, 2>(p, st) : launch_tc_form<FORM_LA, 4>(p, st);
    if (p.form == FORM_GDN) return bf ? launch_tc_form<FORM_GDN, 2>(p, st) : launch_tc_form<FORM_GDN, 4>(p, st);
    if (p.form == FORM_KDA) return bf ? launch_tc_form<FORM_KDA, 2>(p, st) : launch_tc_form<FORM_KDA, 4>(p, st);
    return LAR_ERR_ARG;
}

}  // namespace lar
