// decode_kernel.cuh -- the sm_103a decode kernel shared by GDN, KDA and LA.
//
// Work decomposition.  A tile is TV consecutive state rows of one
// (batch entry b, v-head hv) pair; a state row is one value channel v with its
// K key channels (K fp32, contiguous in the pool).  Tiles are numbered with
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
#ifndef LAR_K128_LPR
#define LAR_K128_LPR 8
#endif
#ifndef LAR_PDL
#define LAR_PDL 1
#endif
#ifndef LAR_K128_BF16_S
#define LAR_K128_BF16_S 3
#endif
#ifndef LAR_K128_S
#define LAR_K128_S 2
#endif

namespace lar {

__device__ __forceinline__ float bf16_bits_to_float(unsigned short x) {
    return __uint_as_float(static_cast<unsigned int>(x) << 16);  // bf16 is the top half of fp32
}

__device__ __forceinline__ float ld_in(const void* base, int64_t off, int dt) {
    if (dt == LAR_F32) return __ldg(static_cast<const float*>(base) + off);
    return bf16_bits_to_float(__ldg(static_cast<const unsigned short*>(base) + off));
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

// 16-byte shared-memory chunk of EPC pool elements -> EPC floats (bf16 widens exactly).
template <int SB>
__device__ __forceinline__ void chunk_to_f32(const unsigned char* p, float* d) {
    if constexpr (SB == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
    } else {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            d[2 * q] = __uint_as_float(w[q] << 16);            // element 2q: low half
            d[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u); // element 2q+1: high half
        }
    }
}

__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low 16 bits)
    return *reinterpret_cast<const unsigned*>(&h);
}

// Streaming store of N floats (N = 4 or 8, contiguous) as fp32 or as bf16 (RNE).
template <int N>
__device__ __forceinline__ void store_run(void* g, const float* d, bool bf16) {
    if (bf16) {
        if constexpr (N == 8) {
            __stcs(reinterpret_cast<uint4*>(g), make_uint4(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3]),
                                                          pack_bf16x2(d[4], d[5]), pack_bf16x2(d[6], d[7])));
        } else {
            __stcs(reinterpret_cast<uint2*>(g), make_uint2(pack_bf16x2(d[0], d[1]), pack_bf16x2(d[2], d[3])));
        }
    } else {
#pragma unroll
        for (int q = 0; q < N / 4; ++q)
            __stcs(reinterpret_cast<float4*>(g) + q, make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]));
    }
}

// v values of a (b, hv) pair are staged in shared memory with the other
// per-pair vectors when T * V is at most this many floats; otherwise the
// token loop reads them from global memory.
constexpr int kStageVMax = 4096;

__host__ __device__ constexpr bool stage_v(int T, int V) { return T * V <= kStageVMax; }

// Floats of one per-pair vector buffer: q, k (and the KDA decay rows) for T
// tokens, the staged v values, and 5 scalars per token; a multiple of 4 so
// the second buffer stays 16-byte aligned.
template <int FORM, int K>
__host__ __device__ constexpr int vec_floats(int T, int V) {
    return ((FORM == FORM_KDA ? 3 : 2) * T * K + (stage_v(T, V) ? T * V : 0) + 5 * T + 3) & ~3;
}

template <int FORM, int K, int LPR, int NR, int NW, int S, int SB>
__host__ __device__ constexpr size_t decode_smem_bytes(int T, int V) {
    using G = Tile<K, LPR, NR, NW, SB>;
    return static_cast<size_t>(S) * G::TV * K * SB + 2 * static_cast<size_t>(vec_floats<FORM, K>(T, V)) * sizeof(float) +
           2 * kMaxTokens * sizeof(long long);   // per-pair tables of per-token write slots
}

// Per-(b, hv) vectors into the buffer vb: the raw q and k rows of all T tokens,
// the KDA decay rows exp(g) (gate chain included), the pair's v values when
// staged, and per token beta, the scalar decay, 1/|q|, 1/|k| and
// q.k / (|q| |k|).  All threads of the CTA take part; ends with a barrier.
template <int FORM, int K, int NW>
__device__ __forceinline__ void build_pair_vectors(const DecodeParams& p, float* vb, int b, int hv, int h,
                                                   int64_t v_off, bool sv_on, int o_k, int o_d, int o_v,
                                                   int o_s) {
    const int T = p.T;
    const int V = p.V;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool gate_raw = (p.flags & LAR_GATE_RAW) != 0;
    const bool l2 = FORM != FORM_LA && (p.flags & LAR_QK_L2NORM) != 0;
    const int64_t q_off = b * p.qs[0] + h * p.qs[2];
    const int64_t k_off = b * p.ks[0] + h * p.ks[2];
    for (int i = threadIdx.x; i < T * K; i += NW * 32) {
        const int t = i / K;
        const int c = i - t * K;
        vb[i] = ld_in(p.q, q_off + t * p.qs[1] + c * p.qs[3], p.q_dt);
        vb[o_k + i] = ld_in(p.k, k_off + t * p.ks[1] + c * p.ks[3], p.k_dt);
        if constexpr (FORM == FORM_KDA) {
            float x = ld_in(p.g, b * p.gs[0] + t * p.gs[1] + hv * p.gs[2] + c * p.gs[3], p.g_dt);
            if (gate_raw) {
                const float bias =
                    p.dt_bias ? p.dt_bias[(static_cast<int64_t>(hv) * K + c) * p.dtb_s] : 0.f;
                x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
            }
            vb[o_d + i] = expf(x);
        }
    }
    if (sv_on) {
        for (int i = threadIdx.x; i < T * V; i += NW * 32) {
            const int t = i / V;
            const int row = i - t * V;
            vb[o_v + i] = ld_in(p.v, v_off + t * p.vs[1] + row * p.vs[3], p.v_dt);
        }
    }
    float* sc = vb + o_s;
    for (int t = threadIdx.x; t < T; t += NW * 32) {
        float bt = 0.f, dec = 1.f;
        if constexpr (FORM != FORM_LA) {
            bt = ld_in(p.beta, b * p.bs[0] + t * p.bs[1] + hv * p.bs[2], p.beta_dt);
            if (p.flags & LAR_BETA_RAW) bt = 1.f / (1.f + expf(-bt));
        }
        if constexpr (FORM == FORM_GDN) {
            float x = ld_in(p.g, b * p.gs[0] + t * p.gs[1] + hv * p.gs[2], p.g_dt);
            if (gate_raw) {
                const float bias = p.dt_bias ? p.dt_bias[hv * p.dtb_s] : 0.f;
                x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
            }
            dec = expf(x);
        } else if constexpr (FORM == FORM_LA) {
            dec = p.decay[h * p.dec_s];
        }
        sc[t] = bt;
        sc[T + t] = dec;
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
            sc[2 * T + t] = iq;
            sc[3 * T + t] = ik;
            sc[4 * T + t] = kq * iq * ik;
        }
    }
    __syncthreads();}

// TOK: per-token pool slots (seed from the accepted count or read_idx, the state
// after every token stored to its slot, no final writeback); compiled
// separately so the plain decode carries none of it.
template <int FORM, int K, int LPR, int NR, int NW, int S, int SB, int MB, bool TOK>
__global__ void __launch_bounds__(NW * 32, MB)
decode_kernel(const DecodeParams p) {
    using G = Tile<K, LPR, NR, NW, SB>;
    constexpr int NCH = G::NCH, RPW = G::RPW, TV = G::TV, EPC = G::EPC, KPL = G::KPL;

    extern __shared__ __align__(16) unsigned char smem[];
    const int T = p.T;
    const int V = p.V;
    const bool sv_on = stage_v(T, V);
    unsigned char* ring = smem;                                               // [S][TV][K] pool elements
    float* vecs = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * TV * K * SB);  // 2 x vec_floats
    long long* slot_tab = reinterpret_cast<long long*>(vecs + 2 * vec_floats<FORM, K>(T, V));  // 2 x kMaxTokens
    const unsigned char* pool_b = static_cast<const unsigned char*>(p.pool);
    const bool inter_bf16 = p.inter_dt == LAR_BF16;
    const int inter_es = inter_bf16 ? 2 : 4;
    const int vstride = vec_floats<FORM, K>(T, V);
    // offsets inside a vector buffer
    const int o_k = T * K;
    const int o_d = 2 * T * K;
    const int o_v = (FORM == FORM_KDA ? 3 : 2) * T * K;
    const int o_s = o_v + (sv_on ? T * V : 0);                  // beta, decay, 1/|q|, 1/|k|, q.k/(|q||k|)

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int j = lane % LPR;
    const int gi = lane / LPR;

    const int nvt = (V + TV - 1) / TV;
    const int64_t total = static_cast<int64_t>(p.B) * p.HV * nvt;
    const int64_t t_begin = blockIdx.x * total / gridDim.x;
    const int64_t t_end = (blockIdx.x + 1) * total / gridDim.x;

#if LAR_PDL
    // programmatic dependent launch: everything below may read what the
    // previous kernel on the stream wrote, so wait for it first; then let the
    // next kernel's CTAs be scheduled as soon as ours retire.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif

    // local row (within a tile) of this thread's i-th row
    auto lrow = [&](int i) { return (warp * NR + i) * RPW + gi; };

    // Byte offsets fixed for the whole kernel.  A thread's rows in a tile are
    // row0, row0 + RPW, ... and its chunks in a row are CSTEP bytes apart, so
    // every chunk address is a per-tile base plus compile-time steps.
    const int row0 = lrow(0);
    constexpr int CSTEP = LPR * 16;                 // between a lane's chunks of one row
    constexpr int STAGE = TV * K * SB;              // one ring stage
    constexpr int S_RSTEP = RPW * K * SB;           // between a thread's rows in a stage
    const int s_row0 = row0 * K * SB + j * 16;
    const int64_t g_row0 = static_cast<int64_t>(row0) * p.ps[2] * SB + j * 16;
    const int64_t g_rstep = static_cast<int64_t>(RPW) * p.ps[2] * SB;
    const int64_t g_tile = static_cast<int64_t>(TV) * p.ps[2] * SB;

    // tile coordinates, advanced incrementally (no per-tile 64-bit division)
    struct Pos {
        int64_t tile;
        int vt, hv, b;
    };
    auto advance = [&](Pos& q) {
        ++q.tile;
        if (++q.vt == nvt) {
            q.vt = 0;
            if (++q.hv == p.HV) {
                q.hv = 0;
                ++q.b;
            }
        }
    };
    Pos cur;
    {
        const int64_t u = t_begin / nvt;
        cur.tile = t_begin;
        cur.vt = static_cast<int>(t_begin - u * nvt);
        cur.b = static_cast<int>(u / p.HV);
        cur.hv = static_cast<int>(u - static_cast<int64_t>(cur.b) * p.HV);
    }

    // read slot of a prefetch position, reloaded only when its batch entry changes
    int ahead_b = -1;
    int64_t ahead_r = -1;
    // Read slot of entry b: read_idx[b], or, with accepted-token counts, the
    // slot that holds the state after the last accepted token,
    // state_idx[b][num_accepted[b] - 1]; a count outside [1, T] has no such
    // slot and yields kBadCount (zero seed, flagged).
    constexpr int64_t kBadCount = INT64_MIN;
    auto seed_of = [&](int b) -> int64_t {
        if (!TOK || p.nacc == nullptr) return ld_idx(p.ridx, b * p.ri_s, p.ri_dt);
        const int64_t a = ld_idx(p.nacc, b * p.na_s, p.na_dt);
        if (a < 1 || a > T) return kBadCount;
        return ld_idx(p.tslot, b * p.tsl_s[0] + (a - 1) * p.tsl_s[1], p.tsl_dt);
    };
    auto slot_of = [&](const Pos& q) -> int64_t {
        if (q.tile >= t_end) return -1;
        if (q.b != ahead_b) {
            ahead_b = q.b;
            ahead_r = seed_of(q.b);
        }
        return ahead_r;
    };

    // issue this thread's copies of the tile at `q` (read slot r) into ring stage `st`
    auto issue = [&](const Pos& q, int64_t r, int st) {
        if (q.tile < t_end && r >= 0 && r < p.P) {
            const unsigned char* src = pool_b + (r * p.ps[0] + static_cast<int64_t>(q.hv) * p.ps[1]) * SB +
                                       q.vt * g_tile + g_row0;
            unsigned char* dst = ring + st * STAGE + s_row0;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                if (q.vt * TV + row0 + i * RPW < V) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        cp_async16(dst + i * S_RSTEP + c * CSTEP, src + i * g_rstep + c * CSTEP);
                }
            }
        }
        cp_async_commit();   // always commit, so group counting stays uniform
    };

    // ---- prologue: S-1 tiles in flight before the first is consumed
    Pos ahead = cur;
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        issue(ahead, slot_of(ahead), s);
        advance(ahead);
    }

    int buf = 1;
    bool rd = false, wr = false;
    unsigned char* dst_state = nullptr;     // state rows of the current pair (write slot)
    int64_t v_off = 0, o_off = 0;           // per-pair offsets into v and out
    unsigned char* inter_base = nullptr;
    const float scale = p.scale;

    int stage = 0;                 // ring stage of the tile being consumed
    int stage_next = S - 1;        // ring stage the next issue goes to
#pragma unroll 1
    for (; cur.tile < t_end; advance(cur)) {
        // read slot of the tile issued at the end of this iteration
        const int64_t r_ahead = slot_of(ahead);
        const int b = cur.b, hv = cur.hv, vt = cur.vt;
        if (vt == 0 || cur.tile == t_begin) {
            // ---- new (b, hv) pair: slots, bases and per-token vectors
            const int h = hv / p.group;
            buf ^= 1;
            const int64_t r = seed_of(b);
            // with per-token slots every token's state is stored; there is no final writeback
            const int64_t w = TOK ? -1 : (p.widx ? ld_idx(p.widx, b * p.wi_s, p.wi_dt) : r);
            rd = r >= 0 && r < p.P;
            wr = w >= 0 && w < p.P;
            if constexpr (TOK) {
                long long* tab = slot_tab + buf * kMaxTokens;
                for (int t = threadIdx.x; t < T; t += NW * 32)
                    tab[t] = ld_idx(p.tslot, b * p.tsl_s[0] + t * p.tsl_s[1], p.tsl_dt);
            }
            if (threadIdx.x == 0 && hv == 0 && p.dev_err) {
                int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0) |
                        (r == kBadCount ? LAR_DEVERR_ACCEPTED : 0);
                if (TOK)
                    for (int t = 0; t < T; ++t)
                        if (ld_idx(p.tslot, b * p.tsl_s[0] + t * p.tsl_s[1], p.tsl_dt) >= p.P) e |= LAR_DEVERR_WRITE_SLOT;
                if (e) atomicOr(p.dev_err, e);
            }
            dst_state = static_cast<unsigned char*>(p.pool) +
                        ((wr ? w : 0) * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1]) * SB;
            v_off = b * p.vs[0] + hv * p.vs[2];
            o_off = b * p.os[0] + hv * p.os[2];
            if (p.inter) inter_base = static_cast<unsigned char*>(p.inter) + (b * p.is[0] + hv * p.is[2]) * inter_es;

            build_pair_vectors<FORM, K, NW>(p, vecs + buf * vstride, b, hv, h, v_off, sv_on, o_k, o_d, o_v, o_s);
        }

        // ---- this thread's copies of the tile have landed: pull its rows into registers
        cp_async_wait<S - 2>();
        float s[NR][KPL];
        {
            const unsigned char* src = ring + stage * STAGE + s_row0;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const bool ok = rd && vt * TV + row0 + i * RPW < V;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (ok) {
                        chunk_to_f32<SB>(src + i * S_RSTEP + c * CSTEP, &s[i][c * EPC]);
                    } else {
#pragma unroll
                        for (int e = 0; e < EPC; ++e) s[i][c * EPC + e] = 0.f;
                    }
                }
            }
        }
        // refill the stage consumed in the previous iteration (its rows were used long ago)
        issue(ahead, r_ahead, stage_next);
        advance(ahead);
        stage = stage + 1 == S ? 0 : stage + 1;
        stage_next = stage_next + 1 == S ? 0 : stage_next + 1;

        // ---- token loop: the state never leaves registers between tokens
        const float* vb = vecs + buf * vstride;
        const float* sc = vb + o_s;
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            const float bt = sc[t], dec = sc[T + t];
            const float iq = sc[2 * T + t], ik = sc[3 * T + t], kq = sc[4 * T + t];
            float kv[KPL], qv[KPL], dv[KPL];
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
#pragma unroll
                for (int e4 = 0; e4 < EPC / 4; ++e4) {
                    const int kidx = t * K + (c * LPR + j) * EPC + 4 * e4;
                    const float4 a4 = *reinterpret_cast<const float4*>(vb + kidx);
                    const float4 b4 = *reinterpret_cast<const float4*>(vb + o_k + kidx);
                    float* qd = &qv[c * EPC + 4 * e4];
                    float* kd = &kv[c * EPC + 4 * e4];
                    qd[0] = a4.x; qd[1] = a4.y; qd[2] = a4.z; qd[3] = a4.w;
                    kd[0] = b4.x; kd[1] = b4.y; kd[2] = b4.z; kd[3] = b4.w;
                    if constexpr (FORM == FORM_KDA) {
                        const float4 d4 = *reinterpret_cast<const float4*>(vb + o_d + kidx);
                        float* dd = &dv[c * EPC + 4 * e4];
                        dd[0] = d4.x; dd[1] = d4.y; dd[2] = d4.z; dd[3] = d4.w;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const int row = vt * TV + lrow(i);
                const bool rv = row < V;
                float vval = 0.f;
                if (rv) vval = sv_on ? vb[o_v + t * V + row] : ld_in(p.v, v_off + t * p.vs[1] + row * p.vs[3], p.v_dt);
#pragma unroll
                for (int e = 0; e < KPL; ++e) s[i][e] *= (FORM == FORM_KDA ? dv[e] : dec);
                // q_hat = iq q and k_hat = ik k: the norms scale the reduced sums
                float o;
                if constexpr (FORM == FORM_LA) {
                    float pp = 0.f;
#pragma unroll
                    for (int e = 0; e < KPL; ++e) pp = fmaf(s[i][e], qv[e], pp);
#pragma unroll
                    for (int off = LPR / 2; off > 0; off >>= 1) pp += __shfl_xor_sync(0xffffffffu, pp, off);
                    const float a = vval * ik;
#pragma unroll
                    for (int e = 0; e < KPL; ++e) s[i][e] = fmaf(a, kv[e], s[i][e]);
                    o = fmaf(vval, kq, pp * iq);
                } else {
                    float uu = 0.f, pp = 0.f;
#pragma unroll
                    for (int e = 0; e < KPL; ++e) {
                        uu = fmaf(s[i][e], kv[e], uu);
                        pp = fmaf(s[i][e], qv[e], pp);
                    }
#pragma unroll
                    for (int off = LPR / 2; off > 0; off >>= 1) {
                        uu += __shfl_xor_sync(0xffffffffu, uu, off);
                        pp += __shfl_xor_sync(0xffffffffu, pp, off);
                    }
                    const float delta = bt * (vval - uu * ik);
                    const float a = delta * ik;
#pragma unroll
                    for (int e = 0; e < KPL; ++e) s[i][e] = fmaf(a, kv[e], s[i][e]);
                    o = fmaf(delta, kq, pp * iq);
                }
                if (j == 0 && rv)
                    st_out(p.out, o_off + t * p.os[1] + row * p.os[3], p.out_dt, o * scale);
                if (p.inter != nullptr && rv) {
                    unsigned char* ip = inter_base + (t * p.is[1] + row * p.is[3]) * inter_es + j * EPC * inter_es;
                    const int cstep = LPR * EPC * inter_es;
#pragma unroll
                    for (int c = 0; c < NCH; ++c) store_run<EPC>(ip + c * cstep, &s[i][c * EPC], inter_bf16);
                }
                if (TOK && rv) {
                    const long long ts = slot_tab[buf * kMaxTokens + t];
                    if (ts >= 0 && ts < p.P) {
                        unsigned char* tp = static_cast<unsigned char*>(p.pool) +
                                            (ts * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1]) * SB +
                                            vt * g_tile + g_row0 + i * g_rstep;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) store_run<EPC>(tp + c * CSTEP, &s[i][c * EPC], SB == 2);
                    }
                }
            }
        }

        // ---- writeback to the write slot (skipped for negative / out-of-range slots)
        if (wr) {
            unsigned char* wb = dst_state + vt * g_tile + g_row0;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                if (vt * TV + row0 + i * RPW < V) {
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        store_run<EPC>(wb + i * g_rstep + c * CSTEP, &s[i][c * EPC], SB == 2);
                }
            }
        }
    }
    cp_async_wait<0>();   // nothing may be left in flight into shared memory at exit
}

// Resident CTAs per SM for a kernel instance and shared-memory size, looked up
// once per (device, size) and cached.
int cached_occupancy(const void* kern, int threads, size_t smem, size_t smem_max, int* sms_out);

template <int FORM, int K, int LPR, int NR, int NW, int S, int SB, int MB, bool TOK>
lar_status launch_tile_mode(const DecodeParams& p, cudaStream_t stream) {
    using G = Tile<K, LPR, NR, NW, SB>;
    auto kern = decode_kernel<FORM, K, LPR, NR, NW, S, SB, MB, TOK>;
    const size_t smem = decode_smem_bytes<FORM, K, LPR, NR, NW, S, SB>(p.T, p.V);
    // the largest footprint any call can ask for (T = 16 with staged v)
    constexpr size_t smem_max = decode_smem_bytes<FORM, K, LPR, NR, NW, S, SB>(16, kStageVMax / 16);
    int sms = 0;
    const int occ = cached_occupancy(reinterpret_cast<const void*>(kern), NW * 32, smem, smem_max, &sms);
    if (occ < 1) return LAR_ERR_LAUNCH;
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


template <int FORM, int K, int LPR, int NR, int NW, int S, int SB, int MB = 1>
lar_status launch_tile(const DecodeParams& p, cudaStream_t stream) {
    if constexpr (FORM != FORM_LA) {
        if (p.tslot != nullptr) return launch_tile_mode<FORM, K, LPR, NR, NW, S, SB, MB, true>(p, stream);
    }
    return launch_tile_mode<FORM, K, LPR, NR, NW, S, SB, MB, false>(p, stream);
}

// Tile shapes per key size and pool type: a row is split over LPR lanes so each
// lane holds whole 16-byte chunks (fp32 K = 128: 8 lanes x 4 chunks of 4
// elements); 32-row tiles at K = 128, a 2-stage ring (one tile in flight while
// one is computed) for fp32 and a 3-stage ring for bf16, whose tiles are half
// the bytes.  Instances whose unconstrained register count would exceed 168
// (fp32 KDA and LA) are compiled for 3 resident CTAs per SM.
template <int FORM>
lar_status launch_form(const DecodeParams& p, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p.pool_dt == LAR_F32) {
        switch (p.K) {
            case 16: return launch_tile<FORM, 16, 4, 2, 2, 3, 4>(p, st);
            case 32: return launch_tile<FORM, 32, 8, 2, 4, 3, 4>(p, st);
            case 64: return launch_tile<FORM, 64, 8, 2, 4, 3, 4>(p, st);
            case 128:
                return launch_tile<FORM, 128, LAR_K128_LPR, LAR_K128_NR, LAR_K128_NW, LAR_K128_S, 4,
                                   FORM == FORM_GDN ? 1 : LAR_K128_MIN_BLOCKS>(p, st);
            default: return LAR_ERR_SHAPE;
        }
    }
    switch (p.K) {
        case 16: return launch_tile<FORM, 16, 2, 2, 2, 3, 2>(p, st);
        case 32: return launch_tile<FORM, 32, 4, 2, 4, 3, 2>(p, st);
        case 64: return launch_tile<FORM, 64, 8, 2, 4, 3, 2>(p, st);
        case 128:
            // bf16 rows are half the bytes: GDN/LA give each lane 32 elements (4 lanes
            // per row, one row per thread), which halves the per-row bookkeeping;
            // KDA keeps 8 lanes per row to stay within its register budget.
            if constexpr (FORM == FORM_KDA)
                return launch_tile<FORM, 128, 8, 2, LAR_K128_NW, LAR_K128_BF16_S, 2, LAR_K128_MIN_BLOCKS>(p, st);
            else
                return launch_tile<FORM, 128, 4, 1, LAR_K128_NW, LAR_K128_BF16_S, 2, 1>(p, st);
        default: return LAR_ERR_SHAPE;
    }
}

}  // namespace lar
