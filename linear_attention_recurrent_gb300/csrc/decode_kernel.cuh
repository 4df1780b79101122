// decode_kernel.cuh -- the sm_103a decode kernel shared by GDN, KDA and LA.
//
// Work decomposition.  A tile is TV consecutive state rows of one
// (batch entry b, v-head hv) pair; a state row is one value channel v with its
// K key channels (K fp32 or bf16 values, contiguous in the pool).  Tiles are numbered with
// the V-tile fastest, then hv, then b, and a persistent grid of
// (SM count x resident CTAs per SM) CTAs takes contiguous, equal ranges of
// them.  The grid is sized from the active batch B*HV, never from the pool.
//
// State streaming.  Every thread owns the same 16-byte chunks of every tile
// (lane group of LPR lanes per row, lane j holding chunks j, j+LPR, ...), and
// moves them HBM -> shared memory with cp.async through an S-stage ring: the
// copies for tile i+S-1 are in flight while tile i is computed.  Because each
// thread only ever reads back the chunks it copied itself, the ring needs no
// barrier between threads (cp.async.wait_group orders a thread's own copies).
// Updated rows go from registers straight back to HBM with streaming stores.
//
// Per token (aiter KDA review recurrence, S^T stored row-wise):
//     s      <- s * exp(g)              (per element for KDA, scalar for GDN)
//     u      =  s . k_hat,  p = s . q_hat     (both reduced over the LPR group)
//     delta  =  beta (v_row - u)
//     s      <- s + delta * k_hat
//     o_row  =  scale * (p + delta * (k_hat . q_hat))      [= scale * s_new . q_hat]
// LA:  s <- lambda s;  p = s . q;  s <- s + v_row k;  o_row = scale (p + v_row (k . q)).
//
// The per-token vectors (q, k, the KDA decay row) and scalars of the current
// (b, hv) pair are built by the whole CTA in shared memory (gate chain and l2
// norms included) when the pair changes, into one of two buffers so that
// building the next pair's vectors never races with readers of the last.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode_params.h"

// K = 128 tile shape: rows per thread, warps per CTA, ring stages.
#ifndef LAR_K128_NR
#define LAR_K128_NR 2
#endif
#ifndef LAR_K128_NW
#define LAR_K128_NW 4
#endif
// Resident CTAs per SM that register-heavy K = 128 kernels are compiled for
// (caps registers at 65536 / (3 x 128) -> 168 per thread, so three 4-warp
// CTAs fit).
#ifndef LAR_K128_MIN_BLOCKS
#define LAR_K128_MIN_BLOCKS 3
#endif
// Resident CTAs per SM the fp32 GDN and the bf16 K = 128 kernels are
// compiled for (1: no register cap; the bf16 CTAs have 64 threads, so any
// value up to 3 leaves the compiler all 255 registers).  fp32 GDN: 3, which
// keeps every instance within 168 registers (the single-token one takes 128
// and runs 4 CTAs per SM).
#ifndef LAR_K128_GDN_MB
#define LAR_K128_GDN_MB 3
#endif
#ifndef LAR_K128_BF16_MB
#define LAR_K128_BF16_MB 1
#endif
// Resident CTAs per SM the fp32 single-token GDN / KDA instances are compiled
// for.
#ifndef LAR_K128_MB1
#define LAR_K128_MB1 3
#endif
#ifndef LAR_K128_LPR
#define LAR_K128_LPR 8
#endif
#ifndef LAR_PDL
#define LAR_PDL 1
#endif
// upper bound on the resident CTAs per SM the persistent grid is sized for
#ifndef LAR_OCC_CAP
#define LAR_OCC_CAP 64
#endif
#ifndef LAR_K128_BF16_S
#define LAR_K128_BF16_S 3
#endif
#ifndef LAR_K128_S
#define LAR_K128_S 2
#endif
// ring stages of the fp32 K = 128 multi-token instances
#ifndef LAR_K128_S_MTP
#define LAR_K128_S_MTP LAR_K128_S
#endif
// bf16 K = 128 tile: lanes per row, rows per thread, warps per CTA
#ifndef LAR_K128_BF16_LPR
#define LAR_K128_BF16_LPR 4
#endif
#ifndef LAR_K128_BF16_NR
#define LAR_K128_BF16_NR 1
#endif
#ifndef LAR_K128_BF16_NW
#define LAR_K128_BF16_NW 2
#endif

namespace lar {

__device__ __forceinline__ float bf16_bits_to_float(unsigned short x) {
    return __uint_as_float(static_cast<unsigned int>(x) << 16);  // bf16 is the top half of fp32
}

__device__ __forceinline__ float ld_in(const void* base, int64_t off, int dt) {
    if (dt == LAR_F32) return __ldg(static_cast<const float*>(base) + off);
    return bf16_bits_to_float(__ldg(static_cast<const unsigned short*>(base) + off));
}

// x[e] = element off + e * st (e = 0..3), fp32 or bf16, with one vector load
// when the four are contiguous and aligned for it
__device__ __forceinline__ void ld_in4(const void* base, int64_t off, int64_t st, int dt, float* x) {
    if (st == 1) {
        if (dt == LAR_BF16) {
            const unsigned short* q = static_cast<const unsigned short*>(base) + off;
            if ((reinterpret_cast<uintptr_t>(q) & 7) == 0) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(q));
                x[0] = __uint_as_float(u.x << 16);
                x[1] = __uint_as_float(u.x & 0xffff0000u);
                x[2] = __uint_as_float(u.y << 16);
                x[3] = __uint_as_float(u.y & 0xffff0000u);
                return;
            }
        } else {
            const float* q = static_cast<const float*>(base) + off;
            if ((reinterpret_cast<uintptr_t>(q) & 15) == 0) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(q));
                x[0] = f.x;
                x[1] = f.y;
                x[2] = f.z;
                x[3] = f.w;
                return;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = ld_in(base, off + e * st, dt);
}

__device__ __forceinline__ int64_t ld_idx(const void* base, int64_t off, int dt) {
    if (dt == LAR_I32) return static_cast<int64_t>(__ldg(static_cast<const int*>(base) + off));
    return static_cast<int64_t>(__ldg(static_cast<const long long*>(base) + off));
}

__device__ __forceinline__ void st_out(void* base, int64_t off, int dt, float x) {
    if (dt == LAR_F32) static_cast<float*>(base)[off] = x;
    else static_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float softplus_f(float x) { return x > 20.f ? x : log1pf(expf(x)); }

// 16-byte global -> shared copy that bypasses L1 (the state is touched once).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
    const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(gmem_src) : "memory");
}

// 4-byte global -> shared copy (through L1; the 16-byte form above bypasses it)
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Tile geometry shared by the kernel and its launcher.  SB is the byte size
// of a pool element (4: fp32, 2: bf16); rows move in 16-byte chunks.
template <int K, int LPR, int NR, int NW, int SB>
struct Tile {
    static constexpr int EPC = 16 / SB;       // state elements per 16-byte chunk
    static constexpr int KPL = K / LPR;       // state elements of a row held by one lane
    static constexpr int NCH = KPL / EPC;     // 16-byte chunks of a row held by one lane
    static constexpr int RPW = 32 / LPR;      // rows covered by one warp instruction
    static constexpr int TV = NW * NR * RPW;  // rows per tile
    static_assert(KPL % EPC == 0 && NCH >= 1, "a lane holds whole 16-byte chunks");
    static_assert(32 % LPR == 0, "row groups tile the warp");
};

// 16-byte shared-memory chunk of EPC pool elements -> EPC/2 float pairs
// (element 2i in .x, 2i+1 in .y; bf16 widens exactly).
template <int SB>
__device__ __forceinline__ void chunk_to_f2(const unsigned char* p, float2* d) {
    if constexpr (SB == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        d[0] = make_float2(v.x, v.y);
        d[1] = make_float2(v.z, v.w);
    } else {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)   // low half: element 2q, high half: element 2q+1
            d[q] = make_float2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
    }
}

__device__ __forceinline__ void st_shared_zero16(void* smem_dst) {
    *reinterpret_cast<float4*>(smem_dst) = make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low 16 bits)
    return *reinterpret_cast<const unsigned*>(&h);
}

// State stores are streaming (evict-first): a written state is not read again
// by this launch (default write-back stores measured 3-8 % slower).
template <typename V>
__device__ __forceinline__ void st_state(V* p, const V& v) {
    __stcs(p, v);
}

// Store of N floats held as N/2 pairs (N = 4 or 8, contiguous), as fp32 or as
// bf16 (RNE).
template <int N>
__device__ __forceinline__ void store_pairs(void* g, const float2* d, bool bf16) {
    if (bf16) {
        if constexpr (N == 8) {
            st_state(reinterpret_cast<uint4*>(g), make_uint4(pack_bf16x2(d[0].x, d[0].y), pack_bf16x2(d[1].x, d[1].y),
                                                            pack_bf16x2(d[2].x, d[2].y), pack_bf16x2(d[3].x, d[3].y)));
        } else {
            st_state(reinterpret_cast<uint2*>(g), make_uint2(pack_bf16x2(d[0].x, d[0].y), pack_bf16x2(d[1].x, d[1].y)));
        }
    } else {
#pragma unroll
        for (int q = 0; q < N / 4; ++q)
            st_state(reinterpret_cast<float4*>(g) + q,
                     make_float4(d[2 * q].x, d[2 * q].y, d[2 * q + 1].x, d[2 * q + 1].y));
    }
}

// v values of a (b, hv) pair are staged in shared memory with the other
// per-pair vectors when T * V is at most this many floats; otherwise the
// token loop reads them from global memory.
constexpr int kStageVMax = 4096;

__host__ __device__ constexpr bool stage_v(int T, int V) { return T * V <= kStageVMax; }

// Per-token scalars of a pair, kScal floats per token (16-byte aligned):
// beta, decay, 1/|q|, 1/|k|, q.k / (|q| |k|), 3 unused.
constexpr int kScal = 8;

// Offset of the scalars in a vector buffer: after q, k (and the KDA decay
// rows) and the staged v values, rounded up to 16 bytes.
__host__ __device__ constexpr int scal_offset(int form, int K, int T, int V) {
    return ((form == FORM_KDA ? 3 : 2) * T * K + (stage_v(T, V) ? T * V : 0) + 3) & ~3;
}

// Floats of one per-pair vector buffer; a multiple of 4 so the second buffer
// stays 16-byte aligned.
template <int FORM, int K>
__host__ __device__ constexpr int vec_floats(int T, int V) {
    return scal_offset(FORM, K, T, V) + kScal * T;
}

template <int FORM, int K, int LPR, int NR, int NW, int S, int SB>
__host__ __device__ constexpr size_t decode_smem_bytes(int T, int V) {
    using G = Tile<K, LPR, NR, NW, SB>;
    return static_cast<size_t>(S) * G::TV * K * SB + 2 * static_cast<size_t>(vec_floats<FORM, K>(T, V)) * sizeof(float) +
           2 * kMaxTokens * sizeof(long long);   // per-pair tables of per-token write slots
}

// Per-(b, hv) vectors into the buffer vb: the raw q and k rows of all T tokens,
// the KDA decay rows exp(g) (gate chain included), the pair's v values when
// staged, and per token (kScal floats each) beta, the scalar decay, 1/|q|,
// 1/|k| and q.k / (|q| |k|).  All threads of the CTA take part; ends with a barrier.
template <int FORM, int K, int NW, int TT>
__device__ __forceinline__ void build_pair_vectors(const DecodeParams& p, float* vb, int b, int hv, int h,
                                                   int64_t v_off, bool sv_on, int o_k, int o_d, int o_v,
                                                   int o_s, int64_t t0 = 0, int nt = -1) {
    // T: the tokens built, t0 onward (all of the call's tokens by default); the
    // buffer layout offsets come from the caller
    const int T = nt >= 0 ? nt : (TT > 0 ? TT : p.T);
    const int V = p.V;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool gate_raw = (p.flags & LAR_GATE_RAW) != 0;
    const bool l2 = FORM != FORM_LA && (p.flags & LAR_QK_L2NORM) != 0;
    const int64_t q_off = b * p.qs[0] + h * p.qs[2];
    const int64_t k_off = b * p.ks[0] + h * p.ks[2];
#pragma unroll 4
    for (int i = threadIdx.x; i < T * K; i += NW * 32) {
        const int t = i / K;
        const int c = i - t * K;
        vb[i] = ld_in(p.q, q_off + (t0 + t) * p.qs[1] + c * p.qs[3], p.q_dt);
        vb[o_k + i] = ld_in(p.k, k_off + (t0 + t) * p.ks[1] + c * p.ks[3], p.k_dt);
        if constexpr (FORM == FORM_KDA) {
            float x = ld_in(p.g, b * p.gs[0] + (t0 + t) * p.gs[1] + hv * p.gs[2] + c * p.gs[3], p.g_dt);
            if (gate_raw) {
                const float bias =
                    p.dt_bias ? p.dt_bias[(static_cast<int64_t>(hv) * K + c) * p.dtb_s] : 0.f;
                x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
            }
            vb[o_d + i] = expf(x);
        }
    }
    if (sv_on) {
        // tokens innermost and unrolled, so one thread's loads are in flight together
        for (int row = threadIdx.x; row < V; row += NW * 32) {
#pragma unroll 4
            for (int t = 0; t < T; ++t)
                vb[o_v + t * V + row] = ld_in(p.v, v_off + (t0 + t) * p.vs[1] + row * p.vs[3], p.v_dt);
        }
    }
    float* sc = vb + o_s;
    for (int t = threadIdx.x; t < T; t += NW * 32) {
        float bt = 0.f, dec = 1.f;
        if constexpr (FORM != FORM_LA) {
            bt = ld_in(p.beta, b * p.bs[0] + (t0 + t) * p.bs[1] + hv * p.bs[2], p.beta_dt);
            if (p.flags & LAR_BETA_RAW) bt = 1.f / (1.f + expf(-bt));
        }
        if constexpr (FORM == FORM_GDN) {
            float x = ld_in(p.g, b * p.gs[0] + (t0 + t) * p.gs[1] + hv * p.gs[2], p.g_dt);
            if (gate_raw) {
                const float bias = p.dt_bias ? p.dt_bias[hv * p.dtb_s] : 0.f;
                x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
            }
            dec = expf(x);
        } else if constexpr (FORM == FORM_LA) {
            dec = p.decay[h * p.dec_s];
        }
        sc[kScal * t] = bt;
        sc[kScal * t + 1] = dec;
    }
    __syncthreads();
    for (int t = warp; t < T; t += NW) {
        float qq = 0.f, kk = 0.f, kq = 0.f;
        for (int c = lane; c < K; c += 32) {
            const float a = vb[t * K + c], bb = vb[o_k + t * K + c];
            qq = fmaf(a, a, qq);
            kk = fmaf(bb, bb, kk);
            kq = fmaf(a, bb, kq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        if (lane == 0) {
            const float iq = l2 ? 1.f / sqrtf(qq + 1e-6f) : 1.f;
            const float ik = l2 ? 1.f / sqrtf(kk + 1e-6f) : 1.f;
            sc[kScal * t + 2] = iq;
            sc[kScal * t + 3] = ik;
            sc[kScal * t + 4] = kq * iq * ik;
        }
    }
    __syncthreads();}

// Variable-length spans: the tile range [t_begin, t_end) of this CTA, ranges of
// nearly equal weight.  A tile of sequence n weighs L_n + kVlTileCost: its
// tokens, plus a fixed cost in token units for loading and storing its state
// (one token: of 1, 2, 4, 8 and 16, the smallest balanced a mix of 1-4 token
// spans and 16-128 token spans best); a reversed or overlong span counts as
// empty.  The
// weighted start of the j-th tile of sequence n is U (sum over n' < n of the
// weights) + j (L_n + kVlTileCost), U = HV * (tiles per head); CTA i takes the
// tiles whose weighted start lies in [i W / G, (i+1) W / G), W the total and G
// the grid size.  Every CTA scans all of cu_seqlens (each thread a contiguous
// run of sequences, then a block-wide scan) and derives the same boundaries,
// so the ranges tile [0, total) exactly.  `red`: shared scratch of NTH / 32 + 2
// entries.  Weighted positions reach about 2^82 at the largest accepted sizes,
// hence 128-bit arithmetic.
#ifndef LAR_VL_TILE_COST
#define LAR_VL_TILE_COST 1
#endif
constexpr int kVlTileCost = LAR_VL_TILE_COST;
// variable-length instance tile shape: rows per thread (a multiple of the
// form's own; for a bf16 pool twice as many, which amortises the per-token
// vector loads over two rows: 7-25 % faster on long spans, while for fp32 the
// second row costs registers and CTAs per SM) and warps per CTA (0: the
// form's own)
#ifndef LAR_VL_NR_MUL
#define LAR_VL_NR_MUL 1
#endif
#ifndef LAR_VL_BF16_NR_MUL
#define LAR_VL_BF16_NR_MUL 2
#endif
#ifndef LAR_VL_NW
#define LAR_VL_NW 0
#endif

template <int NTH>
__device__ __forceinline__ void vl_partition(const DecodeParams& p, int64_t U, int64_t total, long long* red,
                                             int64_t& t_begin, int64_t& t_end, long long* split_out) {
    constexpr int NWARP = NTH / 32;
    static_assert(NWARP + 2 < 2 * kMaxTokens, "the scratch leaves the slot tables' last entry (split_out) alone");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t N = p.B;
    const int64_t seg = (N + NTH - 1) / NTH;
    const int64_t lo = min(N, tid * seg), hi = min(N, lo + seg);
    auto span = [&](int64_t b, bool& rev) -> int64_t {
        const int64_t a = ld_idx(p.cu, b * p.cu_s, p.cu_dt);
        const int64_t e = ld_idx(p.cu, (b + 1) * p.cu_s, p.cu_dt);
        rev = e < a;
        return a >= 0 && e >= a && e <= p.ntok ? e - a : 0;
    };
    // spans the chunked kernel takes cost this kernel only their (empty) tiles;
    // a split call leaves it its long spans only when no span is reversed (then
    // the valid spans are disjoint, which the chunked kernel's grid relies on)
    long long own_split = 0, own_all = 0;
    bool rev_any = false, rev;
    for (int64_t b = lo; b < hi; ++b) {
        const int64_t len = span(b, rev);
        rev_any |= rev;
        own_all += len + kVlTileCost;
        own_split += (p.split_len > 0 && len >= p.split_len ? 0 : len) + kVlTileCost;
    }
    const int split = p.split_len > 0 && !__syncthreads_or(rev_any) ? p.split_len : 0;
    if (tid == 0) *split_out = split;   // visible after the barrier below
    auto weight = [&](int64_t b) -> long long {
        bool r;
        const int64_t len = span(b, r);
        return (split > 0 && len >= split ? 0 : len) + kVlTileCost;
    };
    const long long own = split > 0 ? own_split : own_all;
    long long incl = own;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) red[warp] = incl;
    if (tid == 0) red[NWARP] = red[NWARP + 1] = 0;   // boundaries at weight 0 match no tile start below
    __syncthreads();
    long long w = incl - own, sum = 0;
#pragma unroll
    for (int i = 0; i < NWARP; ++i) {
        if (i < warp) w += red[i];
        sum += red[i];
    }
    using u128 = unsigned __int128;
    const u128 tot = static_cast<u128>(U) * static_cast<u128>(sum);
    const u128 x0 = tot * blockIdx.x / gridDim.x;
    const u128 x1 = tot * (blockIdx.x + 1) / gridDim.x;
    // the tiles that start below x: all of the sequences before the one whose
    // weight interval (W_n, W_n+1] holds x, and ceil((x - W_n) / weight) of its own
    for (int64_t b = lo; b < hi; ++b) {
        const long long c = weight(b);
        const u128 wb = static_cast<u128>(U) * static_cast<u128>(w);
        const u128 wn = static_cast<u128>(U) * static_cast<u128>(w + c);
        if (wb < x0 && x0 <= wn) red[NWARP] = b * U + static_cast<long long>((x0 - wb + c - 1) / c);
        if (wb < x1 && x1 <= wn) red[NWARP + 1] = b * U + static_cast<long long>((x1 - wb + c - 1) / c);
        w += c;
    }
    __syncthreads();
    t_begin = min(max(static_cast<int64_t>(red[NWARP]), int64_t{0}), total);
    t_end = min(max(static_cast<int64_t>(red[NWARP + 1]), t_begin), total);
}

// TOK: per-token pool slots (seed from the accepted count or read_idx, the state
// after every token stored to its slot, no final writeback); compiled
// separately so the plain decode carries none of it.  TT: the token count when
// fixed at compile time (single-token decode without a state cache), 0 when
// taken from the call.  VL: variable-length sequences (token spans from
// cu_seqlens, any length; the per-token vectors are staged in chunks of a
// few tokens, T being the chunk size).
template <int FORM, int K, int LPR, int NR, int NW, int S, int SB, int MB, bool TOK, int TT, bool VL>
__global__ void __launch_bounds__(NW * 32, MB)
decode_kernel(const DecodeParams p) {
    using G = Tile<K, LPR, NR, NW, SB>;
    constexpr int NCH = G::NCH, RPW = G::RPW, TV = G::TV, EPC = G::EPC, KPL = G::KPL;

    extern __shared__ __align__(16) unsigned char smem[];
    const int T = TT > 0 ? TT : p.T;
    const int V = p.V;
    const bool sv_on = stage_v(T, V);
    unsigned char* ring = smem;                                               // [S][TV][K] pool elements
    float* vecs = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * TV * K * SB);  // 2 x vec_floats
    long long* slot_tab = reinterpret_cast<long long*>(vecs + 2 * vec_floats<FORM, K>(T, V));  // 2 x kMaxTokens
    const unsigned char* pool_b = static_cast<const unsigned char*>(p.pool);
    const bool inter_bf16 = p.inter_dt == LAR_BF16;
    const int inter_es = inter_bf16 ? 2 : 4;
    // the single-token instance is only launched without a state cache
    const bool has_inter = TT != 1 && p.inter != nullptr;
    const bool out_bf16 = p.out_dt == LAR_BF16;
    const int out_es = out_bf16 ? 2 : 4;
    const int vstride = vec_floats<FORM, K>(T, V);
    // offsets inside a vector buffer
    const int o_k = T * K;
    const int o_d = 2 * T * K;
    const int o_v = (FORM == FORM_KDA ? 3 : 2) * T * K;
    const int o_s = scal_offset(FORM, K, T, V);        // per-token scalars

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int j = lane % LPR;
    const int gi = lane / LPR;

    const int nvt = (V + TV - 1) / TV;
    const int64_t total = static_cast<int64_t>(p.B) * p.HV * nvt;
    int64_t t_begin, t_end;
    // varlen: spans of this many tokens or more are the chunked kernel's (0: none);
    // kept in the last entry of the per-token slot tables (which only the
    // per-token-slot instances use, and the partition's scratch does not reach)
    // and read once per pair, so that it holds no register
    volatile long long* vl_split_slot = slot_tab + 2 * kMaxTokens - 1;
    auto vl_split = [&]() -> int { return VL ? static_cast<int>(*vl_split_slot) : 0; };
    if constexpr (VL) {
#if LAR_PDL
        // the span offsets may come from the previous kernel on the stream
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif
        vl_partition<NW * 32>(p, static_cast<int64_t>(p.HV) * nvt, total, slot_tab, t_begin, t_end, const_cast<long long*>(vl_split_slot));
    } else {
        t_begin = blockIdx.x * total / gridDim.x;
        t_end = (blockIdx.x + 1) * total / gridDim.x;
    }

    if (t_begin >= t_end) return;

    // A thread's rows in a tile are row0, row0 + RPW, ... and its chunks in a
    // row are CSTEP bytes apart, so every address below is a per-pair base,
    // advanced by a fixed step per tile, plus compile-time offsets.
    const int row0 = (warp * NR) * RPW + gi;
    constexpr int CSTEP = LPR * 16;                 // between a lane's chunks of one row
    constexpr int STAGE = TV * K * SB;              // one ring stage
    constexpr int S_RSTEP = RPW * K * SB;           // between a thread's rows in a stage
    const int s_row0 = row0 * K * SB + j * 16;
    const int64_t g_row0 = static_cast<int64_t>(row0) * p.ps[2] * SB + j * 16;
    const int64_t g_rstep = static_cast<int64_t>(RPW) * p.ps[2] * SB;
    const int64_t g_tile = static_cast<int64_t>(TV) * p.ps[2] * SB;
    const int64_t o_rstep = static_cast<int64_t>(RPW) * p.os[3] * out_es;
    const int64_t o_tstep = p.os[1] * out_es;
    const int64_t o_tile = static_cast<int64_t>(TV) * p.os[3] * out_es;
    const int64_t i_rstep = static_cast<int64_t>(RPW) * p.is[3] * inter_es;
    const int64_t i_tstep = p.is[1] * inter_es;
    const int64_t i_tile = static_cast<int64_t>(TV) * p.is[3] * inter_es;

    // Read slot of entry b: read_idx[b], or, with accepted-token counts, the
    // slot that holds the state after the last accepted token,
    // state_idx[b][num_accepted[b] - 1]; a count outside [1, T] has no such
    // slot and yields kBadCount (zero seed, flagged).
    constexpr int64_t kBadCount = INT64_MIN;
    auto seed_of = [&](int b) -> int64_t {
        if constexpr (VL) {
            // a span the chunked kernel takes: no state to load here
            if (p.split_len > 0) {
                const int sl = vl_split();
                const int64_t lo = ld_idx(p.cu, b * p.cu_s, p.cu_dt), hi = ld_idx(p.cu, (b + 1) * p.cu_s, p.cu_dt);
                if (sl > 0 && lo >= 0 && hi >= lo && hi <= p.ntok && hi - lo >= sl) return -1;
            }
        }
        if (!TOK || p.nacc == nullptr) return ld_idx(p.ridx, b * p.ri_s, p.ri_dt);
        const int64_t a = ld_idx(p.nacc, b * p.na_s, p.na_dt);
        if (a < 1 || a > T) return kBadCount;
        return ld_idx(p.tslot, b * p.tsl_s[0] + (a - 1) * p.tsl_s[1], p.tsl_dt);
    };

    // ---- issue cursor: the next tile whose copies go out.  Its read slot is
    // loaded one tile before the copies need it (a_r), and its source address
    // is a running pointer rebuilt only when the cursor enters a new pair.
    int64_t a_left = t_end - t_begin;
    int a_vt, a_hv, a_b;
    {
        const int64_t u = t_begin / nvt;
        a_vt = static_cast<int>(t_begin - u * nvt);
        a_b = static_cast<int>(u / p.HV);
        a_hv = static_cast<int>(u - static_cast<int64_t>(a_b) * p.HV);
    }
    const int c_vt0 = a_vt, c_hv0 = a_hv, c_b0 = a_b;   // the consumer starts where the issuer does

#if LAR_PDL
    // Programmatic dependent launch.  Everything above is arithmetic on the
    // launch parameters and overlaps the previous kernel's tail; everything
    // below may read what the previous kernel on the stream wrote, so wait for
    // it here (variable-length calls waited before reading the span offsets).
    // Then let the next kernel's CTAs be scheduled as soon as ours retire.
    if constexpr (!VL) {
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    }
#endif
    int a_rb = a_b;                  // batch entry whose read slot a_r holds
    int64_t a_r = seed_of(a_b);
    bool a_new = true;               // a_src must be rebuilt from a_r before the next issue
    bool a_ok = false;
    const unsigned char* a_src = pool_b;

    // issue this thread's copies of the next tile into ring stage `st`; chunks
    // with no state behind them (no valid read slot, rows past V) are zeroed in
    // place, so the consumer reads every chunk unconditionally
    auto issue = [&](int st) {
        if (a_left > 0) {
            if (a_new) {
                a_ok = a_r >= 0 && a_r < p.P;
                a_src = pool_b + ((a_ok ? a_r : 0) * p.ps[0] + static_cast<int64_t>(a_hv) * p.ps[1]) * SB +
                        a_vt * g_tile + g_row0;
                a_new = false;
            }
            unsigned char* dst = ring + st * STAGE + s_row0;
            const int rl = V - a_vt * TV - row0;     // rows of the tile from this thread's first row on
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const bool ok = a_ok && i * RPW < rl;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (ok) cp_async16(dst + i * S_RSTEP + c * CSTEP, a_src + i * g_rstep + c * CSTEP);
                    else st_shared_zero16(dst + i * S_RSTEP + c * CSTEP);
                }
            }
            if (--a_left > 0) {
                if (++a_vt == nvt) {
                    a_vt = 0;
                    if (++a_hv == p.HV) {
                        a_hv = 0;
                        ++a_b;
                    }
                    if (a_b != a_rb) {       // the slot load's latency hides behind one tile of work
                        a_rb = a_b;
                        a_r = seed_of(a_b);
                    }
                    a_new = true;
                } else {
                    a_src += g_tile;
                }
            }
        }
        cp_async_commit();   // always commit, so group counting stays uniform
    };

    // ---- prologue: S-1 tiles in flight before the first is consumed
#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    // ---- consumer cursor and the current pair's running pointers
    int c_vt = c_vt0, c_hv = c_hv0, c_b = c_b0;
    int buf = 1;
    bool wr = false;
    unsigned char* wb = nullptr;         // this thread's first row of the tile in the write slot
    unsigned char* op = nullptr;         // its output element for token 0
    unsigned char* ip = nullptr;         // its first cached chunk for token 0
    unsigned char* tk = nullptr;         // per-token slots: head + tile + row offset inside a slot
    int64_t v_off = 0;
    int64_t tb = 0;                      // varlen: the pair's first token
    int L = 0;                           // varlen: the pair's token count
    bool fresh = false;                  // varlen: this tile built the pair's first chunk
    const float scale = p.scale;
    bool pair_start = true;

    int stage = 0;                 // ring stage of the tile being consumed
    int stage_next = S - 1;        // ring stage the next issue goes to
#pragma unroll 1
    for (int64_t n = t_end - t_begin; n > 0; --n) {
        const int b = c_b, hv = c_hv, vt = c_vt;
        if (pair_start) {
            // ---- new (b, hv) pair: slots, bases and per-token vectors
            pair_start = false;
            const int h = hv / p.group;
            buf ^= 1;
            const int64_t r = seed_of(b);
            // with per-token slots every token's state is stored; there is no final writeback
            const int64_t w = TOK ? -1 : (p.widx ? ld_idx(p.widx, b * p.wi_s, p.wi_dt) : r);
            wr = w >= 0 && w < p.P;
            if constexpr (TOK) {
                long long* tab = slot_tab + buf * kMaxTokens;
                for (int t = threadIdx.x; t < T; t += NW * 32)
                    tab[t] = ld_idx(p.tslot, b * p.tsl_s[0] + t * p.tsl_s[1], p.tsl_dt);
            }
            bool span_ok = true;
            if constexpr (VL) {
                // token span [cu[b], cu[b+1]); a span that is reversed or runs
                // past the token arrays is treated as empty and flagged
                const int64_t lo = ld_idx(p.cu, b * p.cu_s, p.cu_dt);
                const int64_t hi = ld_idx(p.cu, (b + 1) * p.cu_s, p.cu_dt);
                span_ok = lo >= 0 && hi >= lo && hi <= p.ntok;
                tb = span_ok ? lo : 0;
                L = span_ok ? static_cast<int>(hi - lo) : 0;
                fresh = true;
                // a span the chunked kernel takes: nothing to compute or write here
                if (p.split_len > 0 && vl_split() > 0 && L >= vl_split()) {
                    L = 0;
                    wr = false;
                }
            }
            if (threadIdx.x == 0 && hv == 0 && p.dev_err) {
                int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0) |
                        (r == kBadCount ? LAR_DEVERR_ACCEPTED : 0) | (span_ok ? 0 : LAR_DEVERR_SEQLEN);
                if (TOK)
                    for (int t = 0; t < T; ++t)
                        if (ld_idx(p.tslot, b * p.tsl_s[0] + t * p.tsl_s[1], p.tsl_dt) >= p.P) e |= LAR_DEVERR_WRITE_SLOT;
                if (e) atomicOr(p.dev_err, e);
            }
            const int64_t head_tile = static_cast<int64_t>(hv) * p.ps[1] * SB + vt * g_tile + g_row0;
            wb = static_cast<unsigned char*>(p.pool) + (wr ? w : 0) * p.ps[0] * SB + head_tile;
            tk = static_cast<unsigned char*>(p.pool) + head_tile;
            const int64_t first_row = static_cast<int64_t>(vt) * TV + row0;
            v_off = b * p.vs[0] + hv * p.vs[2];
            op = static_cast<unsigned char*>(p.out) +
                 (b * p.os[0] + tb * p.os[1] + hv * p.os[2] + first_row * p.os[3]) * out_es;
            if (has_inter)
                ip = static_cast<unsigned char*>(p.inter) +
                     (b * p.is[0] + tb * p.is[1] + hv * p.is[2] + first_row * p.is[3] + j * EPC) * inter_es;

            if constexpr (VL)
                build_pair_vectors<FORM, K, NW, TT>(p, vecs + buf * vstride, b, hv, h, v_off, sv_on, o_k, o_d, o_v,
                                                    o_s, tb, L < T ? L : T);
            else
                build_pair_vectors<FORM, K, NW, TT>(p, vecs + buf * vstride, b, hv, h, v_off, sv_on, o_k, o_d, o_v,
                                                    o_s);
        }

        // ---- this thread's copies of the tile have landed: pull its rows into registers
        cp_async_wait<S - 2>();
        float2 s[NR][KPL / 2];   // element 2e in .x, 2e+1 in .y
        {
            const unsigned char* src = ring + stage * STAGE + s_row0;
#pragma unroll
            for (int i = 0; i < NR; ++i)
#pragma unroll
                for (int c = 0; c < NCH; ++c) chunk_to_f2<SB>(src + i * S_RSTEP + c * CSTEP, &s[i][c * EPC / 2]);
        }
        // refill the stage consumed in the previous iteration (its rows were used long ago)
        issue(stage_next);
        stage = stage + 1 == S ? 0 : stage + 1;
        stage_next = stage_next + 1 == S ? 0 : stage_next + 1;

        const int rl = V - vt * TV - row0;   // rows of the tile from this thread's first row on

        // ---- token loop: the state never leaves registers between tokens.  The
        // arithmetic runs on element pairs (packed fp32x2 multiply / fma); each
        // reduction keeps one pair accumulator (even and odd elements), summed
        // before the shuffles.
        constexpr int KP = KPL / 2;   // element pairs per lane and row
        unsigned char* opt = op;
        unsigned char* ipt = ip;
        // varlen spans run in chunks of up to T tokens; each chunk's vectors are
        // built when it is not the one already in the buffer (the pair's first
        // chunk, built at the pair start, serves every tile of a short span)
        int c0 = 0;
        do {
        int nt = T;
        int64_t tg0 = 0;              // first token of the chunk in the token arrays
        if constexpr (VL) {
            nt = L - c0 < T ? L - c0 : T;
            tg0 = tb + c0;
            if (c0 > 0 || (!fresh && L > T)) {
                buf ^= 1;
                build_pair_vectors<FORM, K, NW, TT>(p, vecs + buf * vstride, b, hv, hv / p.group, v_off, sv_on,
                                                    o_k, o_d, o_v, o_s, tg0, nt);
            }
        }
        const float* vb = vecs + buf * vstride;
        const float* sc = vb + o_s;
#pragma unroll 1
        for (int t = 0; t < nt; ++t, opt += o_tstep, ipt += i_tstep) {
            const float4 s4 = *reinterpret_cast<const float4*>(sc + kScal * t);
            const float bt = s4.x, dec = s4.y, iq = s4.z, ik = s4.w, kq = sc[kScal * t + 4];
            float2 kv[KP], qv[KP], dv[KP];
            const float* qrow = vb + t * K + j * EPC;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
#pragma unroll
                for (int e4 = 0; e4 < EPC / 4; ++e4) {
                    const int kidx = c * LPR * EPC + 4 * e4;
                    const int e = (c * EPC + 4 * e4) / 2;
                    const float4 a4 = *reinterpret_cast<const float4*>(qrow + kidx);
                    const float4 b4 = *reinterpret_cast<const float4*>(qrow + o_k + kidx);
                    qv[e] = make_float2(a4.x, a4.y);
                    qv[e + 1] = make_float2(a4.z, a4.w);
                    kv[e] = make_float2(b4.x, b4.y);
                    kv[e + 1] = make_float2(b4.z, b4.w);
                    if constexpr (FORM == FORM_KDA) {
                        const float4 d4 = *reinterpret_cast<const float4*>(qrow + o_d + kidx);
                        dv[e] = make_float2(d4.x, d4.y);
                        dv[e + 1] = make_float2(d4.z, d4.w);
                    }
                }
            }
            const float2 dec2 = make_float2(dec, dec);
            long long ts = -1;
            if constexpr (TOK) ts = slot_tab[buf * kMaxTokens + t];
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const bool rv = i * RPW < rl;
                const int row = vt * TV + row0 + i * RPW;
                // rows past V compute on zeros and store nothing; their staged-v read is
                // clamped into the row range instead of branched around
                float vval = 0.f;
                if (sv_on) vval = vb[o_v + t * V + min(row, V - 1)];
                else if (rv) vval = ld_in(p.v, v_off + (tg0 + t) * p.vs[1] + row * p.vs[3], p.v_dt);
#pragma unroll
                for (int e = 0; e < KP; ++e) s[i][e] = __fmul2_rn(s[i][e], FORM == FORM_KDA ? dv[e] : dec2);
                // q_hat = iq q and k_hat = ik k: the norms scale the reduced sums
                float o;
                if constexpr (FORM == FORM_LA) {
                    float2 p2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < KP; ++e) p2 = __ffma2_rn(s[i][e], qv[e], p2);
                    float pp = p2.x + p2.y;
#pragma unroll
                    for (int off = LPR / 2; off > 0; off >>= 1) pp += __shfl_xor_sync(0xffffffffu, pp, off);
                    const float a = vval * ik;
                    const float2 a2 = make_float2(a, a);
#pragma unroll
                    for (int e = 0; e < KP; ++e) s[i][e] = __ffma2_rn(a2, kv[e], s[i][e]);
                    o = fmaf(vval, kq, pp * iq);
                } else {
                    float2 u2 = make_float2(0.f, 0.f), p2 = u2;
#pragma unroll
                    for (int e = 0; e < KP; ++e) {
                        u2 = __ffma2_rn(s[i][e], kv[e], u2);
                        p2 = __ffma2_rn(s[i][e], qv[e], p2);
                    }
                    float uu = u2.x + u2.y;
                    float pp = p2.x + p2.y;
#pragma unroll
                    for (int off = LPR / 2; off > 0; off >>= 1) {
                        uu += __shfl_xor_sync(0xffffffffu, uu, off);
                        pp += __shfl_xor_sync(0xffffffffu, pp, off);
                    }
                    const float delta = bt * (vval - uu * ik);
                    const float a = delta * ik;
                    const float2 a2 = make_float2(a, a);
#pragma unroll
                    for (int e = 0; e < KP; ++e) s[i][e] = __ffma2_rn(a2, kv[e], s[i][e]);
                    o = fmaf(delta, kq, pp * iq);
                }
                if (j == 0 && rv) {
                    unsigned char* dst = opt + i * o_rstep;
                    if (out_bf16) *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(o * scale);
                    else *reinterpret_cast<float*>(dst) = o * scale;
                }
                if (has_inter && rv) {
                    unsigned char* dst = ipt + i * i_rstep;
                    const int cstep = LPR * EPC * inter_es;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) store_pairs<EPC>(dst + c * cstep, &s[i][c * EPC / 2], inter_bf16);
                }
                if (TOK && rv && ts >= 0 && ts < p.P) {
                    unsigned char* dst = tk + ts * p.ps[0] * SB + i * g_rstep;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) store_pairs<EPC>(dst + c * CSTEP, &s[i][c * EPC / 2], SB == 2);
                }
            }
        }
        c0 += T;
        } while (VL && c0 < L);
        if constexpr (VL) fresh = false;

        // ---- writeback to the write slot (skipped for negative / out-of-range slots)
        if (wr) {
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                if (i * RPW < rl) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        store_pairs<EPC>(wb + i * g_rstep + c * CSTEP, &s[i][c * EPC / 2], SB == 2);
                }
            }
        }

        // ---- advance the consumer: next tile of this pair, or the next pair
        if (++c_vt == nvt) {
            c_vt = 0;
            if (++c_hv == p.HV) {
                c_hv = 0;
                ++c_b;
            }
            pair_start = true;
        } else {
            wb += g_tile;
            tk += g_tile;
            op += o_tile;
            ip += i_tile;
        }
    }
    cp_async_wait<0>();   // nothing may be left in flight into shared memory at exit
}

// Resident CTAs per SM for a kernel instance and shared-memory size, looked up
// once per (device, size) and cached.
int cached_occupancy(const void* kern, int threads, size_t smem, size_t smem_max, int* sms_out);

template <int FORM, int K, int LPR, int NR, int NW, int S, int SB, int MB, bool TOK, int TT, bool VL = false>
lar_status launch_tile_mode(const DecodeParams& p, cudaStream_t stream) {
    using G = Tile<K, LPR, NR, NW, SB>;
    auto kern = decode_kernel<FORM, K, LPR, NR, NW, S, SB, MB, TOK, TT, VL>;
    const size_t smem = decode_smem_bytes<FORM, K, LPR, NR, NW, S, SB>(p.T, p.V);
    // the largest footprint any call can ask for (T = 16 with staged v)
    constexpr size_t smem_max = decode_smem_bytes<FORM, K, LPR, NR, NW, S, SB>(16, kStageVMax / 16);
    int sms = 0;
    int occ = cached_occupancy(reinterpret_cast<const void*>(kern), NW * 32, smem, smem_max, &sms);
    if (occ < 1) return LAR_ERR_LAUNCH;
    if (occ > LAR_OCC_CAP) occ = LAR_OCC_CAP;
    const int nvt = (p.V + G::TV - 1) / G::TV;
    const int64_t tiles = static_cast<int64_t>(p.B) * p.HV * nvt;
    const int64_t cap = static_cast<int64_t>(sms) * occ;
    const int64_t grid = tiles < cap ? tiles : cap;
#if LAR_PDL
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? LAR_OK : LAR_ERR_LAUNCH;
#else
    kern<<<static_cast<unsigned>(grid), NW * 32, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? LAR_OK : LAR_ERR_LAUNCH;
#endif
}


// S1: ring stages of the single-token instance (K = 128 only; 0: no such
// instance, single tokens take the general one).  The per-token-slot instance
// stores every token's state, so it streams like a single-token call and
// takes S1 stages too.
template <int FORM, int K, int LPR, int NR, int NW, int S, int SB, int MB = 1, int S1 = 0, int MB1 = MB>
lar_status launch_tile(const DecodeParams& p, cudaStream_t stream) {
    if (p.cu != nullptr)
        return launch_tile_mode<FORM, K, LPR, NR * (SB == 2 ? LAR_VL_BF16_NR_MUL : LAR_VL_NR_MUL),
                                (LAR_VL_NW > 0 ? LAR_VL_NW : NW), S, SB, MB, false, 0, true>(p, stream);
    if constexpr (FORM != FORM_LA) {
        if (p.tslot != nullptr)
            return launch_tile_mode<FORM, K, LPR, NR, NW, (S1 > 0 ? S1 : S), SB, MB, true, 0>(p, stream);
    }
    if constexpr (S1 > 0) {
        if (p.T == 1 && p.inter == nullptr)
            return launch_tile_mode<FORM, K, LPR, NR, NW, S1, SB, MB1, false, 1>(p, stream);
    }
    return launch_tile_mode<FORM, K, LPR, NR, NW, S, SB, MB, false, 0>(p, stream);
}

// Tile shapes per key size and pool type: a row is split over LPR lanes so each
// lane holds whole 16-byte chunks (fp32 K = 128: 8 lanes x 4 chunks of 4
// elements); 32-row tiles at K = 128, a 2-stage ring (one tile in flight while
// one is computed) for fp32 and 3 stages for bf16, whose tiles are half the
// bytes.  Instances whose unconstrained
// register count would exceed 168 (fp32 KDA and LA) are compiled for 3
// resident CTAs per SM.  At K = 128 single-token GDN / KDA calls (and bf16 LA)
// take an instance with T fixed at 1; fp32 LA keeps one 2-stage instance for
// every T (both the T = 1 instance and 3 stages measured slower for it).
template <int FORM>
lar_status launch_form(const DecodeParams& p, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p.pool_dt == LAR_F32) {
        switch (p.K) {
            case 16: return launch_tile<FORM, 16, 4, 2, 2, 3, 4>(p, st);
            case 32: return launch_tile<FORM, 32, 8, 2, 4, 3, 4>(p, st);
            case 64: return launch_tile<FORM, 64, 8, 2, 4, 3, 4>(p, st);
            case 128:
                if constexpr (FORM == FORM_LA)
                    return launch_tile<FORM, 128, LAR_K128_LPR, LAR_K128_NR, LAR_K128_NW, LAR_K128_S, 4,
                                       LAR_K128_MIN_BLOCKS>(p, st);
                else
                    return launch_tile<FORM, 128, LAR_K128_LPR, LAR_K128_NR, LAR_K128_NW, LAR_K128_S_MTP, 4,
                                       FORM == FORM_GDN ? LAR_K128_GDN_MB : LAR_K128_MIN_BLOCKS, LAR_K128_S,
                                       LAR_K128_MB1>(p, st);
            default: return LAR_ERR_SHAPE;
        }
    }
    switch (p.K) {
        case 16: return launch_tile<FORM, 16, 2, 2, 2, 3, 2>(p, st);
        case 32: return launch_tile<FORM, 32, 4, 2, 4, 3, 2>(p, st);
        case 64: return launch_tile<FORM, 64, 8, 2, 4, 3, 2>(p, st);
        case 128:
            // bf16 rows are half the bytes: each lane holds 32 elements (4 lanes per
            // row, one row per thread), which halves the per-row bookkeeping, in
            // 2-warp CTAs (16-row tiles; up to 8 CTAs per SM progress independently).
            // Against 4-warp CTAs: GDN 6 % faster, KDA 19 % (its former 8-lane,
            // 2-row shape in 1-warp CTAs: 5 % slower).
            return launch_tile<FORM, 128, LAR_K128_BF16_LPR, LAR_K128_BF16_NR, LAR_K128_BF16_NW, LAR_K128_BF16_S, 2,
                               LAR_K128_BF16_MB, LAR_K128_BF16_S>(p, st);
        default: return LAR_ERR_SHAPE;
    }
}

}  // namespace lar
