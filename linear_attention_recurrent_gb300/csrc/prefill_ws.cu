// prefill_ws.cu -- the chunked prefill for GDN and LA (bf16 q / k / v rows with
// unit inner stride, 16-byte aligned: the usual layouts) as a warp-specialised
// tensor-core kernel.  Same operation and chunk algebra as prefill_tc.cu, whose
// header states it; other forms and layouts run there.
#include <type_traits>

#include <cuda.h>   // CUtensorMap and its encoder's signature (called through the runtime's driver entry point)

#include "prefill_common.cuh"

namespace lar {
namespace {
using namespace pf;

// Warp-specialised form (GDN, LA; bf16 q / k / v rows, 16-byte aligned).  Per
// (sequence, head) the chunks form one dependent chain: [U | P] from the state,
// the solve, the increment, the new state.  Everything that does not depend on
// the state -- the chunk's k / q tiles, K K^T, the decay table, the A and M
// tables -- and the output product O are handled by four "side" warps beside
// the eight "chain" warps.
//
// bf16 operands.  q and k arrive as bf16, so the [K ; Q] and K^T tiles hold the
// raw bf16 values and the l2 norms (when asked) enter as per-token factors
// 1/|k_t|, 1/|q_t| on the products' rows and columns.  The tensor-core operands
// that are computed fp32 values -- the state and D o W -- are split into three
// bf16 terms x = b1 + b2 + b3 (b1 the nearest bf16, each further term the
// nearest bf16 to the exact remainder: 24 significant bits), so every product
// is exact and accumulates in fp32: K K^T and Q K^T in one kind::f16 pass (8
// instructions of K = 16), S^T [K ; Q]^T in three (24), (D o W / |k|) K in
// three (6).  O = D M^T keeps the tf32 three-pass form (12 instructions).  A
// tensor-core instruction takes about the same time whatever its N (up to 128)
// and type, so instruction counts set the products' cost.
//
// Hand-offs (mbarriers; [2]: one per chunk parity, completing every other chunk):
//   KQ_READY[2]   side -> chain   chunk c's [K ; Q] and K^T tiles are written
//   TAB_READY[2]  side -> chain   chunk c's A and M tables and factors are written
//   D_READY[2]    chain -> side   chunk c's D is in tensor memory (and every read
//                                 of chunk c's side buffers by the chain threads is
//                                 done): the side issues O(c)
//   DS_DONE[2]    tensor cores    [U | P](c) and the increment of chunk c have
//                                 completed
//   O_DONE[2]     tensor cores    O(c) has completed
//   UP_DONE, KK_DONE, STG_FULL    [U | P], the side's K K^T, a chunk's input boxes
// The side refills chunk c's buffers with chunk c + 2 once DS_DONE(c) and
// O_DONE(c) are in, so it can run up to two chunks ahead.  O(c) enters the
// tensor pipe right behind the increment and runs while the chain updates the
// state; its accumulator (columns 352..383) starts from E_t P[v][t] / |q_t|,
// written by the chain's first half once it has handed its half of the solve
// over (the second half finishes the solve meanwhile), and its outputs are
// stored by the second half early in the next chunk, while [U | P] runs.  A wait that
// gives up sets a shared abort flag; the waits of the other group see it and
// give up too, both groups leave their loops, and the CTA skips its writeback.
namespace ws {
constexpr int NCHAIN = 256;   // warps 0..7
constexpr int NSIDE = 128;    // warps 8..11 (one per tensor-memory lane quarter)
constexpr int NT = NCHAIN + NSIDE;
constexpr int NVB = 3;        // v staging ring
// bf16 tiles, K-major, no swizzle (16-byte core-matrix rows of 8 elements)
constexpr uint32_t BLBO = 144;                                // K-adjacent core matrices
constexpr uint32_t BKQ_SBO = (TK / 8) * BLBO + 16;            // [K ; Q]: 64 rows x 128 keys
constexpr uint32_t BKQ_BYTES = 8 * BKQ_SBO;
constexpr uint32_t BKT_SBO = (TC / 8) * BLBO + 16;            // K^T: 128 keys x 32 tokens
constexpr uint32_t BKT_BYTES = (TK / 8) * BKT_SBO;
constexpr uint32_t OFF_KQ = 0;                                // [parity] [K ; Q] tile
constexpr uint32_t OFF_KT = OFF_KQ + 2 * BKQ_BYTES;           // [parity] K^T tile
constexpr uint32_t OFF_MT = OFF_KT + 2 * BKT_BYTES;           // [parity][hi, lo] M tile (tf32)
constexpr uint32_t OFF_AT = OFF_MT + 4 * MT_BYTES;            // [parity] A transposed: [s][t]
constexpr uint32_t OFF_P = OFF_AT + 2 * TC * TROW * 4;        // decay table P[t][s] (side)
constexpr uint32_t OFF_AF = OFF_P + TC * TROW * 4;            // a_t (side)
constexpr uint32_t OFF_IQ = OFF_AF + TC * 4;                  // 1/|q_t| (side)
constexpr uint32_t OFF_IK = OFF_IQ + TC * 4;                  // 1/|k_t| (side)
constexpr uint32_t OFF_B = OFF_IK + TC * 4;                   // [parity] beta_t
constexpr uint32_t OFF_EK = OFF_B + 2 * TC * 4;               // [parity] E_t / |k_t|
constexpr uint32_t OFF_EQ = OFF_EK + 2 * TC * 4;              // [parity] E_t / |q_t|
constexpr uint32_t OFF_WK = OFF_EQ + 2 * TC * 4;              // [parity] W_s / |k_s|
constexpr uint32_t OFF_E31 = OFF_WK + 2 * TC * 4;             // [parity] E_31 (16 bytes each)
// staging (tensor-copy destinations, 128-byte aligned): q rows, k rows, fp32
// gates, fp32 betas (one chunk), then the v ring
constexpr uint32_t OFF_STG = (OFF_E31 + 2 * 16 + 127) / 128 * 128;
constexpr uint32_t SQ = 0, SK = TC * STG_ROW, SG = 2 * TC * STG_ROW, SBT = SG + TC * 4, S_BYTES = SBT + TC * 4;
constexpr uint32_t OFF_V = OFF_STG + S_BYTES;                 // [NVB][TC] bf16 rows
constexpr uint32_t OFF_BAR = OFF_V + NVB * TC * STG_ROW;
enum {
    KQ_READY = 0, TAB_READY = 2, D_READY = 4, DS_DONE = 6, O_DONE = 8, UP_DONE = 10, KK_DONE = 11, STG_FULL = 12,
    NBAR = 13
};
constexpr uint32_t OFF_TM = OFF_BAR + NBAR * 8;               // TMEM base, picked sequence, abort flag
// the solve's hand-over: d_0..15 of each value row (rows padded to 20 floats, so
// a quarter-warp's 16-byte accesses fall in distinct banks)
constexpr int XROW = 20;
constexpr uint32_t OFF_X = (OFF_TM + 16 + 15) / 16 * 16;
constexpr uint32_t SMEM = OFF_X + TVV * XROW * 4;
// tensor-memory columns: the state's three bf16 planes (64 columns each; D o W's
// three planes of 16 reuse them once [U | P] has read the state), D's tf32
// halves for O, [U | P], K K^T, O's accumulator, the increment
constexpr uint32_t COL_SP = 0, SP_STRIDE = 64, COL_DWP = 0, DWP_STRIDE = 16;
constexpr uint32_t COL_DH = 192, COL_DL = 224, COL_O2 = 352;
static_assert(COL_SP + 3 * SP_STRIDE <= COL_DH && COL_DL + TC <= COL_UP && COL_O2 >= COL_KK + TC &&
                  COL_O2 + TC <= COL_DS,
              "tensor-memory map");
static_assert(OFF_KT % 16 == 0 && OFF_MT % 16 == 0 && OFF_AT % 16 == 0 && OFF_STG % 128 == 0 && SK % 128 == 0 &&
                  OFF_V % 128 == 0 && (TC * STG_ROW) % 128 == 0 && OFF_BAR % 8 == 0 && BKQ_BYTES % 16 == 0 &&
                  BKT_BYTES % 16 == 0 && MT_BYTES % 16 == 0,
              "tile, staging and barrier alignment");
static_assert(tc::kmaj16(63, TK - 1, BLBO, BKQ_SBO) + 2 <= BKQ_BYTES &&
                  tc::kmaj16(TK - 1, TC - 1, BLBO, BKT_SBO) + 2 <= BKT_BYTES,
              "bf16 tiles hold their elements");
static_assert(SMEM <= 227 * 1024, "fits one CTA's shared memory");
static_assert(kLptMax * 4 <= NVB * TC * STG_ROW, "the span lengths fit the v ring");
static_assert(NSIDE == 128 && TC == 32, "one side warp per lane quarter; 8 tokens per side warp");

// K K^T and Q K^T from the [K ; Q] tile (M = 64, N = 32): one pass
__device__ __forceinline__ void issue_kk(uint32_t tm, uint32_t kq) {
    constexpr uint32_t idesc = tc::idesc_bf16(64, TC);
#pragma unroll 1
    for (int kb = 0; kb < TK / 16; ++kb)
        tc::mma_ss(tm + COL_KK, tc::smem_desc(kq + kb * 2 * BLBO, BLBO, BKQ_SBO),
                   tc::smem_desc(kq + kb * 2 * BLBO, BLBO, BKQ_SBO), idesc, kb > 0);
}

// [U | P] = S^T [K ; Q]^T (LA: P only) from the state's three bf16 planes
template <bool LA>
__device__ __forceinline__ void issue_up(uint32_t tm, uint32_t kq) {
    constexpr int NUP = LA ? TC : 2 * TC;
    constexpr uint32_t idesc = tc::idesc_bf16(TVV, NUP);
    const uint32_t bb = kq + (LA ? 4 * BKQ_SBO : 0);
    const uint32_t dcol = tm + COL_UP + (LA ? TC : 0);
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
#pragma unroll 1
        for (int kb = 0; kb < TK / 16; ++kb)
            tc::mma_ts(dcol, tm + COL_SP + ps * SP_STRIDE + 8 * kb, tc::smem_desc(bb + kb * 2 * BLBO, BLBO, BKQ_SBO),
                       idesc, ps > 0 || kb > 0);
    }
}

// the increment (D o W / |k|) K from D o W's three bf16 planes and the K^T tile
__device__ __forceinline__ void issue_ds(uint32_t tm, uint32_t kt) {
    constexpr uint32_t idesc = tc::idesc_bf16(TVV, TK);
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
#pragma unroll 1
        for (int kb = 0; kb < TC / 16; ++kb)
            tc::mma_ts(tm + COL_DS, tm + COL_DWP + ps * DWP_STRIDE + 8 * kb,
                       tc::smem_desc(kt + kb * 2 * BLBO, BLBO, BKT_SBO), idesc, ps > 0 || kb > 0);
    }
}

// O += D M^T (tf32, three passes, onto the accumulator's starting value)
__device__ __forceinline__ void issue_o(uint32_t tm, uint32_t mth, uint32_t mtl) {
    constexpr uint32_t idesc = tc::idesc_tf32(TVV, TC);
#pragma unroll 1
    for (int ps = 0; ps < 3; ++ps) {
        const uint32_t ad = tm + (ps == 2 ? COL_DL : COL_DH);
        const uint32_t bm = ps == 1 ? mtl : mth;
#pragma unroll 1
        for (int kb = 0; kb < TC / 8; ++kb)
            tc::mma_ts(tm + COL_O2, ad + 8 * kb, tc::smem_desc(bm + kb * 2 * LBO, LBO, MT_SBO), idesc, true);
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// x (N values, a multiple of 32) into tensor memory as three bf16 planes
// (plane i at taddr + i * stride, N / 2 columns of element pairs):
// x = b1 + b2 + b3 with b1 the nearest bf16 to x and b2, b3 the nearest bf16 to
// the remainders x - b1 and x - b1 - b2 (both exact in fp32)
template <int N>
__device__ __forceinline__ void split3_store(uint32_t taddr, uint32_t stride, const float* x) {
#pragma unroll
    for (int i0 = 0; i0 < N; i0 += 32) {
        float w1[16], w2[16], w3[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float a = x[i0 + 2 * j], b = x[i0 + 2 * j + 1];
            const uint32_t p1 = pack_bf16x2(a, b);
            const float ra = a - bf16_lo(p1), rb = b - bf16_hi(p1);
            const uint32_t p2 = pack_bf16x2(ra, rb);
            const uint32_t p3 = pack_bf16x2(ra - bf16_lo(p2), rb - bf16_hi(p2));
            w1[j] = __uint_as_float(p1);
            w2[j] = __uint_as_float(p2);
            w3[j] = __uint_as_float(p3);
        }
        tc::tmem_st16(taddr + i0 / 2, w1);
        tc::tmem_st16(taddr + stride + i0 / 2, w2);
        tc::tmem_st16(taddr + 2 * stride + i0 / 2, w3);
    }
}

// The right-looking elimination of d_t for t in [TLO, THI) by every d_s, s < t
// (s < THI - 1): once d_s is final it is taken out of each later row, one
// dependent multiply-add per step.  AT[s][t] is the coefficient of d_s in row t.
// First group of four t's that step s updates.
__host__ __device__ constexpr int elim_first(int s, int tlo) { return ((s + 1) & ~3) > tlo ? ((s + 1) & ~3) : tlo; }

template <int TLO, int THI>
__device__ __forceinline__ void eliminate(float* d, const float* AT) {
    // each step's row of A is loaded while the step before it runs: the steps
    // wait on one multiply-add of the previous step, not on shared memory
    constexpr int NG = (THI - TLO) / 4;
    float4 a[NG], an[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g)
        if (TLO + 4 * g >= elim_first(0, TLO)) a[g] = *reinterpret_cast<const float4*>(AT + TLO + 4 * g);
#pragma unroll
    for (int s = 0; s < THI - 1; ++s) {
        if (s + 1 < THI - 1) {
#pragma unroll
            for (int g = 0; g < NG; ++g)
                if (TLO + 4 * g >= elim_first(s + 1, TLO))
                    an[g] = *reinterpret_cast<const float4*>(AT + (s + 1) * TROW + TLO + 4 * g);
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int t4 = TLO + 4 * g;
            if (t4 < elim_first(s, TLO)) continue;
            if (t4 > s) d[t4] = fmaf(-a[g].x, d[s], d[t4]);
            if (t4 + 1 > s) d[t4 + 1] = fmaf(-a[g].y, d[s], d[t4 + 1]);
            if (t4 + 2 > s) d[t4 + 2] = fmaf(-a[g].z, d[s], d[t4 + 2]);
            d[t4 + 3] = fmaf(-a[g].w, d[s], d[t4 + 3]);
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) a[g] = an[g];
    }
}

// 16 values into tensor memory as three bf16 planes of 8 columns (as split3_store)
__device__ __forceinline__ void split3_store16(uint32_t taddr, uint32_t stride, const float* x) {
    float w1[8], w2[8], w3[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float a = x[2 * j], b = x[2 * j + 1];
        const uint32_t p1 = pack_bf16x2(a, b);
        const float ra = a - bf16_lo(p1), rb = b - bf16_hi(p1);
        const uint32_t p2 = pack_bf16x2(ra, rb);
        const uint32_t p3 = pack_bf16x2(ra - bf16_lo(p2), rb - bf16_hi(p2));
        w1[j] = __uint_as_float(p1);
        w2[j] = __uint_as_float(p2);
        w3[j] = __uint_as_float(p3);
    }
    tc::tmem_st8(taddr, w1);
    tc::tmem_st8(taddr + stride, w2);
    tc::tmem_st8(taddr + 2 * stride, w3);
}

// One value row's outputs of a chunk: the Lo finished accumulator columns at
// taddr, times the scale, to p.out at element offset off0 + t * os[1] (kept out
// of line: the output stores run once per chunk, and the kernel's code has to
// share the instruction caches among three concurrent code paths).
__device__ __noinline__ void store_outputs(uint32_t taddr, const DecodeParams& p, int64_t off0, int Lo) {
    float o[TC];
#pragma unroll
    for (int i = 0; i < TC; i += 16) tc::tmem_ld16(taddr + i, o + i);
    tc::tmem_ld_wait();
    const int64_t st = p.os[1];
    if (p.out_dt == LAR_BF16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + off0;
#pragma unroll
        for (int t = 0; t < TC; ++t)
            if (t < Lo) out[t * st] = __float2bfloat16_rn(o[t] * p.scale);
    } else {
        float* out = static_cast<float*>(p.out) + off0;
#pragma unroll
        for (int t = 0; t < TC; ++t)
            if (t < Lo) out[t * st] = o[t] * p.scale;
    }
}
}  // namespace ws

// The call's arguments and tiled tensor maps over the token-major q, k and v
// arrays ({channel, head, token}, 16-bit elements, box 128 x 1 x 32: one
// chunk's rows of one head), which the side warps load one box per chunk.
struct WsParams {
    DecodeParams p;
    CUtensorMap tq, tk, tv;
};

template <int FORM, int SB>
__global__ void __launch_bounds__(ws::NT, 1) prefill_ws_kernel(const __grid_constant__ WsParams wp) {
    static_assert(FORM != FORM_KDA, "KDA runs in prefill_tc_kernel");
    const DecodeParams& p = wp.p;
    constexpr bool LA = FORM == FORM_LA;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + ws::OFF_BAR);
    uint32_t* tm_slot = reinterpret_cast<uint32_t*>(smem + ws::OFF_TM);
    volatile int* abort_f = reinterpret_cast<volatile int*>(smem + ws::OFF_TM + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool chain = tid < ws::NCHAIN;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int vrow = quarter * 32 + lane;                      // chain: this thread's value row
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int hv = blockIdx.x;
    const int h = hv / p.group;

#if LAR_PDL
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif
    // ---- which sequence: longest spans first; in a split variable-length call
    // only the long ones (pick_sequence); the v ring is not in use yet
    const int n = pick_sequence<ws::NT>(p, reinterpret_cast<int*>(smem + ws::OFF_V),
                                      reinterpret_cast<int*>(smem + ws::OFF_TM) + 1);
    if (n < 0) return;
    // ---- span and slots (reversed or overlong spans run as empty and are flagged)
    const int64_t lo = ld_idx(p.cu, n * p.cu_s, p.cu_dt);
    const int64_t hi = ld_idx(p.cu, (n + 1) * p.cu_s, p.cu_dt);
    const bool span_ok = lo >= 0 && hi >= lo && hi <= p.ntok;
    const int64_t tb = span_ok ? lo : 0;
    const int64_t L = span_ok ? hi - lo : 0;
    // a variable-length call sends only its long spans here (the rest run token by token)
    if (p.split_len > 0 && L < p.split_len) return;
    const int nch = static_cast<int>((L + TC - 1) / TC);
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
        for (int i = 0; i < ws::NBAR; ++i) tc::mbar_init(&bar[i], 1);
        *abort_f = 0;
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc(tm_slot, TMEM_COLS);
    tc_sync();
    const uint32_t tm = *tm_slot;

    const bool l2 = !LA && (p.flags & LAR_QK_L2NORM) != 0;
    const bool gate_raw = (p.flags & LAR_GATE_RAW) != 0;
    const bool beta_raw = (p.flags & LAR_BETA_RAW) != 0;
    // q, k and v rows are staged through shared memory (the launcher sends
    // only bf16 rows with unit inner stride and 16-byte alignment here)
    const bool stage_scal = !LA && p.g_dt == LAR_F32 && p.beta_dt == LAR_F32;

    if (chain) {
        // ================= chain warps =================
        // registers: the chain's two warpgroups take 200 a thread, the side's
        // warpgroup 104 (256 x 200 + 128 x 104 = 384 x 168, the launch's total)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;\n" ::: "memory");
        const uint32_t my = tm + lane_off;
        const int col0 = 64 * half;                              // this thread's 64 state columns
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
            ws::split3_store<64>(my + ws::COL_SP + col0 / 2, ws::SP_STRIDE, S);
            tc::tmem_st_wait();
        }
        tc::fence_before_sync();
        tc::bar_sync(1, ws::NCHAIN);
        tc::fence_after_sync();

        // outputs of chunk cc (half 1): the finished accumulator E P / |q| + D M^T
        auto store_outputs = [&](int cc) {
            const int64_t o0 = static_cast<int64_t>(cc) * TC;
            ws::store_outputs(my + ws::COL_O2, p, (tb + o0) * p.os[1] + static_cast<int64_t>(hv) * p.os[2] +
                                                       static_cast<int64_t>(vrow) * p.os[3],
                              static_cast<int>(L - o0 < TC ? L - o0 : TC));
        };

        bool done = true;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const int64_t c0 = static_cast<int64_t>(c) * TC;
            const int Lc = static_cast<int>(L - c0 < TC ? L - c0 : TC);
            const uint32_t par = static_cast<uint32_t>(c & 1), par2 = static_cast<uint32_t>((c >> 1) & 1);
            const float* AT = reinterpret_cast<const float*>(smem + ws::OFF_AT) + b * TC * TROW;
            const float* Bt = reinterpret_cast<const float*>(smem + ws::OFF_B) + b * TC;
            const float* EK = reinterpret_cast<const float*>(smem + ws::OFF_EK) + b * TC;
            const float* EQ = reinterpret_cast<const float*>(smem + ws::OFF_EQ) + b * TC;
            const float* WK = reinterpret_cast<const float*>(smem + ws::OFF_WK) + b * TC;

            // ---- [U | P] once the side warps have written the chunk's tiles
            bool ok = true;
            if (tid == 0) {
                ok = tc::mbar_wait_or(&bar[ws::KQ_READY + b], par2, abort_f);
                if (ok) {
                    tc::fence_after_sync();
                    ws::issue_up<LA>(tm, tc::smem_addr(smem + ws::OFF_KQ + b * ws::BKQ_BYTES));
                    tc::mma_commit(&bar[ws::UP_DONE]);
                }
            }
            // the previous chunk's outputs (half 1) while [U | P] runs, once its O has
            // completed ([U | P] does not touch O's columns)
            const int cp = c - 1;
            if (half == 1 && c > 0) {
                if (tc::mbar_wait_or(&bar[ws::O_DONE + (cp & 1)], static_cast<uint32_t>((cp >> 1) & 1), abort_f)) {
                    tc::fence_after_sync();
                    store_outputs(cp);
                } else {
                    ok = false;
                }
            }
            ok = ok && tc::mbar_wait_or(&bar[ws::UP_DONE], par, abort_f) &&
                 tc::mbar_wait_or(&bar[ws::TAB_READY + b], par2, abort_f);
            if (!ok) *abort_f = 1;
            if (tc::bar_or(1, ws::NCHAIN, !ok)) {
                done = false;
                break;
            }
            tc::fence_after_sync();
            // every read of the side warps' chunk-c buffers happens before D_READY
            // (E_31 is taken now)
            const float ec = reinterpret_cast<const float*>(smem + ws::OFF_E31)[4 * b];

            {
                // ---- the solve per value row, right-looking (once d_s is final it is
                // taken out of every later row, one dependent FMA per step), split by
                // tokens between the chain's halves: half 0 finishes d_0..15 and hands
                // them over through shared memory, half 1 takes them out of d_16..31 and
                // finishes those (the operations and their order those of one thread
                // doing all 32).  Each half then stores its own tokens' D, and half 0
                // starts O's accumulator.  v_t: the staged row (the side warps reported
                // the chunk ready).
                const unsigned short* sv =
                    reinterpret_cast<const unsigned short*>(smem + ws::OFF_V + (c % ws::NVB) * TC * STG_ROW) + vrow;
                auto vin = [&](int t) -> float { return t < Lc ? bf16_bits_to_float(sv[t * TVV]) : 0.f; };
                float* xr = reinterpret_cast<float*>(smem + ws::OFF_X) + vrow * ws::XROW;
                auto solve = [&](auto half_c) {
                    constexpr int T0 = decltype(half_c)::value * 16;
                    float d[TC];
                    {
                        // d_t starts as beta_t (v_t - E_t u_t / |k_t|) (LA: v_t), u from [U | P]
                        float u[16], vv[16];
                        if constexpr (!LA) tc::tmem_ld16(my + COL_UP + T0, u);
#pragma unroll
                        for (int i = 0; i < 16; ++i) vv[i] = vin(T0 + i);
                        if constexpr (LA) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) d[T0 + i] = vv[i];
                        } else {
                            tc::tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < 16; ++i) d[T0 + i] = Bt[T0 + i] * fmaf(-EK[T0 + i], u[i], vv[i]);
                        }
                    }
                    if constexpr (!LA && T0 == 0) {
                        ws::eliminate<0, 16>(d, AT);
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4*>(xr + i) = make_float4(d[i], d[i + 1], d[i + 2], d[i + 3]);
                    }
                    // the hand-over; also orders half 1's reads of O's accumulator (the
                    // previous chunk's outputs) before half 0 restarts it
                    tc::fence_before_sync();
                    tc::bar_sync(1, ws::NCHAIN);
                    tc::fence_after_sync();
                    if constexpr (!LA && T0 == 16) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4) {
                            const float4 x = *reinterpret_cast<const float4*>(xr + i);
                            d[i] = x.x;
                            d[i + 1] = x.y;
                            d[i + 2] = x.z;
                            d[i + 3] = x.w;
                        }
                        ws::eliminate<16, 32>(d, AT);
                    }
                    // D's tf32 halves for O (once the previous chunk's O has read its D) and
                    // D o W / |k| as three bf16 planes for the increment
                    if (c > 0 &&
                        !tc::mbar_wait_or(&bar[ws::O_DONE + (cp & 1)], static_cast<uint32_t>((cp >> 1) & 1), abort_f))
                        *abort_f = 1;
                    tc::fence_after_sync();
                    split_store<16>(my + ws::COL_DH + T0, my + ws::COL_DL + T0, d + T0);
#pragma unroll
                    for (int i = 0; i < 16; ++i) d[T0 + i] *= WK[T0 + i];
                    ws::split3_store16(my + ws::COL_DWP + T0 / 2, ws::DWP_STRIDE, d + T0);
                    if constexpr (T0 == 0) {
                        // ---- O's accumulator starts as E_t P[v][t] / |q_t|
                        float pv[TC];
#pragma unroll
                        for (int i = 0; i < TC; i += 16) tc::tmem_ld16(my + COL_UP + TC + i, pv + i);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int t = 0; t < TC; ++t) pv[t] *= EQ[t];
#pragma unroll
                        for (int i = 0; i < TC; i += 16) tc::tmem_st16(my + ws::COL_O2 + i, pv + i);
                    }
                    tc::tmem_st_wait();
                };
                if (half == 0)
                    solve(std::integral_constant<int, 0>{});
                else
                    solve(std::integral_constant<int, 1>{});
            }
            tc::fence_before_sync();
            tc::bar_sync(1, ws::NCHAIN);
            tc::fence_after_sync();

            // ---- the increment; D is ready for the side warps' O
            if (tid == 0) {
                ws::issue_ds(tm, tc::smem_addr(smem + ws::OFF_KT + b * ws::BKT_BYTES));
                tc::mma_commit(&bar[ws::DS_DONE + b]);
                tc::mbar_arrive(&bar[ws::D_READY + b]);
            }
            ok = tc::mbar_wait_or(&bar[ws::DS_DONE + b], par2, abort_f);
            if (!ok) *abort_f = 1;
            if (tc::bar_or(1, ws::NCHAIN, !ok)) {
                done = false;
                break;
            }
            tc::fence_after_sync();

            // ---- the new state E_31 S + increment, rounded to nearest, and its bf16
            // planes for the next chunk's first product
            {
                const bool more = c + 1 < nch;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    float x[32];
                    tc::tmem_ld16(my + COL_DS + col0 + cc, x);
                    tc::tmem_ld16(my + COL_DS + col0 + cc + 16, x + 16);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) S[cc + i] = fmaf(ec, S[cc + i], x[i]);
                    if (more) ws::split3_store<32>(my + ws::COL_SP + (col0 + cc) / 2, ws::SP_STRIDE, S + cc);
                }
                if (more) tc::tmem_st_wait();
            }
            tc::fence_before_sync();
            tc::bar_sync(1, ws::NCHAIN);
            tc::fence_after_sync();
        }
        // the last chunk's outputs, once its O has completed
        if (done && nch > 0 && half == 1) {
            const int cl = nch - 1;
            if (tc::mbar_wait_or(&bar[ws::O_DONE + (cl & 1)], static_cast<uint32_t>((cl >> 1) & 1), abort_f)) {
                tc::fence_after_sync();
                store_outputs(cl);
            } else {
                *abort_f = 1;
            }
        }

        __syncthreads();
        if (*abort_f == 0 && wr) {
            // ---- pool[w][hv][v][k] = S^T[v][k]
            unsigned char* dst = static_cast<unsigned char*>(p.pool) +
                                 (w * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1] +
                                  static_cast<int64_t>(vrow) * p.ps[2] + col0) * SB;
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
    } else {
        // ================= side warps =================
        asm volatile("setmaxnreg.dec.sync.aligned.u32 104;\n" ::: "memory");
        const int sw = warp - ws::NCHAIN / 32;                   // 0..3: also the tensor-memory lane quarter
        const int stid = tid - ws::NCHAIN;
        unsigned char* stg = smem + ws::OFF_STG;
        float* Pt = reinterpret_cast<float*>(smem + ws::OFF_P);
        float* Af = reinterpret_cast<float*>(smem + ws::OFF_AF);
        float* Iq = reinterpret_cast<float*>(smem + ws::OFF_IQ);
        float* Ik = reinterpret_cast<float*>(smem + ws::OFF_IK);
        // chunk `ci`'s inputs (tokens from cs on; side warp 0): one box each of q, k
        // (this head's rows) into the staging and of v into the ring, completing on
        // STG_FULL; the fp32 gates and betas with cp.async
        auto stage = [&](int64_t cs, int ci) {
            const int Ln = static_cast<int>(L - cs < TC ? L - cs : TC);
            if (lane == 0) {
                tc::fence_smem_to_async();   // earlier reads of these buffers come first
                tc::mbar_arrive_expect_tx(&bar[ws::STG_FULL], 3 * TC * STG_ROW);
                const int z = static_cast<int>(tb + cs);
                tc::tma_load_3d(stg + ws::SQ, &wp.tq, 0, h, z, &bar[ws::STG_FULL]);
                tc::tma_load_3d(stg + ws::SK, &wp.tk, 0, h, z, &bar[ws::STG_FULL]);
                tc::tma_load_3d(smem + ws::OFF_V + (ci % ws::NVB) * TC * STG_ROW, &wp.tv, 0, hv, z, &bar[ws::STG_FULL]);
            }
            if (stage_scal && lane < Ln) {
                const int64_t gt = tb + cs + lane;
                cp_async4(stg + ws::SG + lane * 4,
                          static_cast<const float*>(p.g) + gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2]);
                cp_async4(stg + ws::SBT + lane * 4,
                          static_cast<const float*>(p.beta) + gt * p.bs[1] + static_cast<int64_t>(hv) * p.bs[2]);
            }
            cp_async_commit();
        };
        if (sw == 0 && L > 0) stage(0, 0);

#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
            const int b = c & 1;
            const int64_t c0 = static_cast<int64_t>(c) * TC;
            const int Lc = static_cast<int>(L - c0 < TC ? L - c0 : TC);
            float* AT = reinterpret_cast<float*>(smem + ws::OFF_AT) + b * TC * TROW;
            float* Bt = reinterpret_cast<float*>(smem + ws::OFF_B) + b * TC;
            unsigned char* kq = smem + ws::OFF_KQ + b * ws::BKQ_BYTES;
            unsigned char* kt = smem + ws::OFF_KT + b * ws::BKT_BYTES;
            unsigned char* mt = smem + ws::OFF_MT + b * 2 * MT_BYTES;
            const uint32_t pm2 = static_cast<uint32_t>(((c - 2) >> 1) & 1);   // chunk c - 2's phase

            // ---- O of chunk c - 2 (side warp 3) once its D is ready: it enters the
            // tensor pipe right behind that chunk's increment
            bool ok = true;
            if (c >= 2 && stid == 96) {
                ok = tc::mbar_wait_or(&bar[ws::D_READY + b], pm2, abort_f);
                if (ok) {
                    tc::fence_after_sync();
                    ws::issue_o(tm, tc::smem_addr(mt), tc::smem_addr(mt + MT_BYTES));
                    tc::mma_commit(&bar[ws::O_DONE + b]);
                }
            }
            // ---- chunk c - 2's [U | P] and increment have completed (this parity's
            // [K ; Q] and K^T tiles, tables and factors are free), and the chunk's
            // inputs have landed
            ok = ok && (c < 2 || tc::mbar_wait_or(&bar[ws::DS_DONE + b], pm2, abort_f)) &&
                 tc::mbar_wait_or(&bar[ws::STG_FULL], static_cast<uint32_t>(c & 1), abort_f);
            cp_async_wait<0>();
            if (!ok) *abort_f = 1;
            if (tc::bar_or(2, ws::NSIDE, !ok)) break;
            tc::fence_after_sync();

            // ---- raw k and q rows: side warp sw takes tokens 8 sw .. 8 sw + 7 in two
            // runs of 4 (a run's loads issued before any is used), lane l channels
            // 4l .. 4l + 3
            constexpr int RPW = TC / 4;
#pragma unroll 1
            for (int j0 = 0; j0 < RPW; j0 += 4) {
                uint2 qr[4], kr[4];                    // raw bf16 bits (padding tokens: zero)
                float qa[4][4], ka[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = RPW * sw + j0 + j;
                    qr[j] = t < Lc ? *reinterpret_cast<const uint2*>(stg + ws::SQ + t * STG_ROW + lane * 8) : make_uint2(0, 0);
                    kr[j] = t < Lc ? *reinterpret_cast<const uint2*>(stg + ws::SK + t * STG_ROW + lane * 8) : make_uint2(0, 0);
                    auto widen = [](uint2 u, float* x) {
                        x[0] = ws::bf16_lo(u.x);
                        x[1] = ws::bf16_hi(u.x);
                        x[2] = ws::bf16_lo(u.y);
                        x[3] = ws::bf16_hi(u.y);
                    };
                    widen(qr[j], qa[j]);
                    widen(kr[j], ka[j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int t = RPW * sw + j0 + j;
                    float iq = 1.f, ik = 1.f;
                    if (l2) {
                        float sq = 0.f, sk = 0.f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            sq = fmaf(qa[j][e], qa[j][e], sq);
                            sk = fmaf(ka[j][e], ka[j][e], sk);
                        }
#pragma unroll
                        for (int off = 16; off > 0; off >>= 1) {
                            sq += __shfl_xor_sync(0xffffffffu, sq, off);
                            sk += __shfl_xor_sync(0xffffffffu, sk, off);
                        }
                        iq = 1.f / sqrtf(sq + 1e-6f);
                        ik = 1.f / sqrtf(sk + 1e-6f);
                    }
                    if (lane == 0) {
                        Iq[t] = iq;
                        Ik[t] = ik;
                    }
                    *reinterpret_cast<uint2*>(kq + tc::kmaj16(t, 4 * lane, ws::BLBO, ws::BKQ_SBO)) = kr[j];
                    *reinterpret_cast<uint2*>(kq + tc::kmaj16(TC + t, 4 * lane, ws::BLBO, ws::BKQ_SBO)) = qr[j];
                }
                // K^T: channel c = 4 lane + e, the run's 4 tokens as one 8-byte run
                auto bits = [](float x) { return __float_as_uint(x) >> 16; };   // x holds a bf16 value
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    *reinterpret_cast<uint2*>(kt + tc::kmaj16(4 * lane + e, RPW * sw + j0, ws::BLBO, ws::BKT_SBO)) =
                        make_uint2(bits(ka[0][e]) | (bits(ka[1][e]) << 16), bits(ka[2][e]) | (bits(ka[3][e]) << 16));
            }
            // decay factors and betas (side warp 1, lane t; padding tokens: no decay, no update)
            if (sw == 1) {
                const int t = lane;
                float a = 1.f, bt = 0.f;
                if (t < Lc) {
                    const int64_t gt = tb + c0 + t;
                    if constexpr (LA) {
                        a = p.decay[h * p.dec_s];
                        bt = 1.f;
                    } else {
                        float x = stage_scal ? reinterpret_cast<const float*>(stg + ws::SG)[t]
                                             : ld_in(p.g, gt * p.gs[1] + static_cast<int64_t>(hv) * p.gs[2], p.g_dt);
                        if (gate_raw) {
                            const float bias = p.dt_bias ? p.dt_bias[hv * p.dtb_s] : 0.f;
                            x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
                        }
                        a = expf(x);
                        const float bx = stage_scal
                                             ? reinterpret_cast<const float*>(stg + ws::SBT)[t]
                                             : ld_in(p.beta, gt * p.bs[1] + static_cast<int64_t>(hv) * p.bs[2], p.beta_dt);
                        bt = beta_raw ? 1.f / (1.f + expf(-bx)) : bx;
                    }
                }
                Af[t] = a;
                Bt[t] = bt;
            }
            tc::fence_smem_to_async();
            tc::bar_sync(2, ws::NSIDE);
            // the tiles are complete: the chain may issue [U | P]; K K^T goes out
            // (side warp 3), and the staging takes the next chunk's copies (side warp 0)
            if (stid == 96) {
                tc::fence_after_sync();
                tc::mbar_arrive(&bar[ws::KQ_READY + b]);
                ws::issue_kk(tm, tc::smem_addr(kq));
                tc::mma_commit(&bar[ws::KK_DONE]);
            }
            if (sw == 0 && c + 1 < nch) stage(c0 + TC, c + 1);
            if (sw == 1) {
                // the decay table, then the factors the chain applies: E_t / |k_t|,
                // E_t / |q_t|, W_s / |k_s|, E_31
                float* E = reinterpret_cast<float*>(smem + ws::OFF_EK) + b * TC;   // E_t first, scaled below
                float* Wd = reinterpret_cast<float*>(smem + ws::OFF_WK) + b * TC;
                decay_table(lane, Af, Pt, E, Wd);
                const int t = lane;
                const float et = E[t];
                if (t == TC - 1) reinterpret_cast<float*>(smem + ws::OFF_E31)[4 * b] = et;
                reinterpret_cast<float*>(smem + ws::OFF_EQ)[b * TC + t] = et * Iq[t];
                E[t] = et * Ik[t];
                Wd[t] *= Ik[t];
            }
            tc::bar_sync(2, ws::NSIDE);

            // ---- the A (transposed) and M tables from K K^T and Q K^T:
            // A[t][s] = beta_t P[t][s] (k_t . k_s) / (|k_t| |k_s|) for s < t, and
            // M[t][s] = P[t][s] (q_t . k_s) / (|q_t| |k_s|)
            // (the M tile's buffer also waits for chunk c - 2's O)
            ok = tc::mbar_wait_or(&bar[ws::KK_DONE], static_cast<uint32_t>(c & 1), abort_f) &&
                 (c < 2 || tc::mbar_wait_or(&bar[ws::O_DONE + b], pm2, abort_f));
            if (!ok) *abort_f = 1;
            if (tc::bar_or(2, ws::NSIDE, !ok)) break;
            tc::fence_after_sync();
            {
                float x[TC];
                const uint32_t q0 = tm + (static_cast<uint32_t>(sw * 32) << 16) + COL_KK;
                tc::tmem_ld16(q0, x);
                tc::tmem_ld16(q0 + 16, x + 16);
                tc::tmem_ld_wait();
                if (lane < 16) {
                    const int t = 16 * (sw & 1) + lane;
                    const float* pr = Pt + t * TROW;
                    if (sw < 2) {
                        if constexpr (!LA) {
                            const float bk = Bt[t] * Ik[t];
#pragma unroll
                            for (int s = 0; s < TC; ++s) AT[s * TROW + t] = s < t ? bk * pr[s] * Ik[s] * x[s] : 0.f;
                        }
                    } else {
                        const float iqt = Iq[t];
#pragma unroll
                        for (int s4 = 0; s4 < TC; s4 += 4) {
                            float m[4], mh[4], ml[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                m[e] = iqt * pr[s4 + e] * Ik[s4 + e] * x[s4 + e];
                                mh[e] = tc::tf32_hi(m[e]);
                                ml[e] = m[e] - mh[e];
                            }
                            const uint32_t o = tc::kmaj(t, s4, LBO, MT_SBO);
                            *reinterpret_cast<float4*>(mt + o) = make_float4(mh[0], mh[1], mh[2], mh[3]);
                            *reinterpret_cast<float4*>(mt + MT_BYTES + o) = make_float4(ml[0], ml[1], ml[2], ml[3]);
                        }
                    }
                }
            }
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            tc::bar_sync(2, ws::NSIDE);
            if (stid == 0) tc::mbar_arrive(&bar[ws::TAB_READY + b]);
        }
        // the last two chunks' O
        if (stid == 96 && *abort_f == 0) {
#pragma unroll 1
            for (int cc = nch >= 2 ? nch - 2 : 0; cc < nch; ++cc) {
                const int bb = cc & 1;
                if (!tc::mbar_wait_or(&bar[ws::D_READY + bb], static_cast<uint32_t>((cc >> 1) & 1), abort_f)) {
                    *abort_f = 1;
                    break;
                }
                tc::fence_after_sync();
                unsigned char* mt = smem + ws::OFF_MT + bb * 2 * MT_BYTES;
                ws::issue_o(tm, tc::smem_addr(mt), tc::smem_addr(mt + MT_BYTES));
                tc::mma_commit(&bar[ws::O_DONE + bb]);
            }
        }
        cp_async_wait<0>();   // nothing may be left in flight into shared memory at exit
        __syncthreads();
    }

    tc_sync();
    if (tid == 0 && *abort_f != 0 && p.dev_err) atomicOr(p.dev_err, LAR_DEVERR_TIMEOUT);
    if (warp == 0) tc::tmem_dealloc(tm, TMEM_COLS);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (null when unavailable).
EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Tensor map over a token-major bf16 array (element strides st: -, token,
// head, channel with st[3] == 1): {channel 128, head `heads`, token ntok}, box
// 128 x 1 x TC.  False when the encoder refuses it.
bool token_map(CUtensorMap* m, const void* base, int64_t heads, int64_t ntok, const int64_t* st) {
    const EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr || heads < 1 || ntok < 1) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(TK), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(ntok)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(st[2]) * 2, static_cast<cuuint64_t>(st[1]) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(TK), 1, static_cast<cuuint32_t>(TC)};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FORM, int SB>
lar_status launch_ws_form(const DecodeParams& p, cudaStream_t stream, bool* launched) {
    // positive strides and token indices that fit the tensor copies' coordinates;
    // maps the encoder accepts
    *launched = false;
    if (p.qs[1] <= 0 || p.qs[2] <= 0 || p.ks[1] <= 0 || p.ks[2] <= 0 || p.vs[1] <= 0 || p.vs[2] <= 0 ||
        p.ntok < 1 || p.ntok >= (int64_t(1) << 31))
        return LAR_OK;
    WsParams wp;
    wp.p = p;
    if (!token_map(&wp.tq, p.q, p.H, p.ntok, p.qs) || !token_map(&wp.tk, p.k, p.H, p.ntok, p.ks) ||
        !token_map(&wp.tv, p.v, p.HV, p.ntok, p.vs))
        return LAR_OK;
    *launched = true;
    return launch_kernel(prefill_ws_kernel<FORM, SB>, ws::NT, ws::SMEM, wp, p, stream);
}

}  // namespace

lar_status launch_prefill_ws(const DecodeParams& p, void* stream, bool* launched) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = p.pool_dt == LAR_BF16;
    *launched = false;
    if (p.K != TK || p.V != TVV) return LAR_OK;
    if (p.form == FORM_LA) return bf ? launch_ws_form<FORM_LA, 2>(p, st, launched) : launch_ws_form<FORM_LA, 4>(p, st, launched);
    if (p.form == FORM_GDN) return bf ? launch_ws_form<FORM_GDN, 2>(p, st, launched) : launch_ws_form<FORM_GDN, 4>(p, st, launched);
    return LAR_OK;
}

}  // namespace lar
