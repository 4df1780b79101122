// decode_kv_kernel.cuh -- decode kernel for the K x V state layout
// (pool[slot][hv][k][v] = S[k][v], v fastest; the "nontranspose" layout of the
// flashinfer GDN decode kernels).
//
// Tile: all K rows x 32 value columns of one (b, hv) pair.  A lane owns one
// 16-byte chunk of columns (EPC elements) in K / RG rows; CL lanes span the 32
// columns and the remaining lanes of the warp, and the CTA's warps, split the
// rows.  The reductions over k therefore run down the rows: each thread sums
// its rows, the warp combines its row lanes with shuffles, and the warps
// combine through shared memory (one barrier per token).  Tiles stream
// through the same persistent cp.async ring as the V x K kernel.
#pragma once

#include "decode_kernel.cuh"

namespace lar {

template <int K, int NW, int SB>
struct KvTile {
    static constexpr int EPC = 16 / SB;   // columns per 16-byte chunk
    static constexpr int TVC = 32;        // columns per tile
    static constexpr int CL = TVC / EPC;  // lanes across the columns (8 fp32, 4 bf16)
    static constexpr int RL = 32 / CL;    // lanes of a warp across rows
    static constexpr int RG = NW * RL;    // row groups in the CTA
    static constexpr int NRK = K / RG;    // rows per thread
    static_assert(K % RG == 0 && NRK >= 1, "the rows split evenly over the CTA");
};

template <int FORM, int K, int NW, int S>
__host__ __device__ constexpr size_t kv_red_floats() {
    return 2 * static_cast<size_t>(NW) * 2 * 32;   // [2 buffers][NW warps][u, p][32 columns]
}

template <int FORM, int K, int NW, int S, int SB>
__host__ __device__ constexpr size_t decode_kv_smem_bytes(int T, int V) {
    using G = KvTile<K, NW, SB>;
    return static_cast<size_t>(S) * K * G::TVC * SB +
           (2 * static_cast<size_t>(vec_floats<FORM, K>(T, V)) + kv_red_floats<FORM, K, NW, S>()) * sizeof(float);
}

template <int FORM, int K, int NW, int S, int SB, int MB>
__global__ void __launch_bounds__(NW * 32, MB)
decode_kv_kernel(const DecodeParams p) {
    using G = KvTile<K, NW, SB>;
    constexpr int EPC = G::EPC, TVC = G::TVC, CL = G::CL, RL = G::RL, RG = G::RG, NRK = G::NRK;

    extern __shared__ __align__(16) unsigned char smem[];
    const int T = p.T;
    const int V = p.V;
    const bool sv_on = stage_v(T, V);
    constexpr int STAGE = K * TVC * SB;                                   // one ring stage: [K][TVC]
    unsigned char* ring = smem;
    float* vecs = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * STAGE);
    const int vstride = vec_floats<FORM, K>(T, V);
    float* red = vecs + 2 * vstride;                                      // cross-warp partial sums
    const int o_k = T * K;
    const int o_d = 2 * T * K;
    const int o_v = (FORM == FORM_KDA ? 3 : 2) * T * K;
    const int o_s = o_v + (sv_on ? T * V : 0);
    const unsigned char* pool_b = static_cast<const unsigned char*>(p.pool);
    const bool inter_bf16 = p.inter_dt == LAR_BF16;
    const int inter_es = inter_bf16 ? 2 : 4;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int cl = lane % CL;
    const int rl = lane / CL;
    const int rg = warp * RL + rl;         // this thread's rows: rg, rg + RG, ...
    const int col0 = cl * EPC;             // its first column within a tile

    const int nvt = (V + TVC - 1) / TVC;
    const int64_t total = static_cast<int64_t>(p.B) * p.HV * nvt;
    const int64_t t_begin = blockIdx.x * total / gridDim.x;
    const int64_t t_end = (blockIdx.x + 1) * total / gridDim.x;

#if LAR_PDL
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif

    // byte offsets fixed for the kernel: rows are RG apart, chunks never move
    const int s_row0 = (rg * TVC + col0) * SB;
    constexpr int S_RSTEP = RG * TVC * SB;
    const int64_t g_row0 = (static_cast<int64_t>(rg) * p.ps[2] + col0) * SB;
    const int64_t g_rstep = static_cast<int64_t>(RG) * p.ps[2] * SB;
    constexpr int G_TILE = TVC * SB;

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
    int ahead_b = -1;
    int64_t ahead_r = -1;
    auto slot_of = [&](const Pos& q) -> int64_t {
        if (q.tile >= t_end) return -1;
        if (q.b != ahead_b) {
            ahead_b = q.b;
            ahead_r = ld_idx(p.ridx, q.b * p.ri_s, p.ri_dt);
        }
        return ahead_r;
    };
    auto issue = [&](const Pos& q, int64_t r, int st) {
        if (q.tile < t_end && r >= 0 && r < p.P && q.vt * TVC + col0 < V) {
            const unsigned char* src = pool_b + (r * p.ps[0] + static_cast<int64_t>(q.hv) * p.ps[1]) * SB +
                                       q.vt * G_TILE + g_row0;
            unsigned char* dst = ring + st * STAGE + s_row0;
#pragma unroll
            for (int i = 0; i < NRK; ++i) cp_async16(dst + i * S_RSTEP, src + i * g_rstep);
        }
        cp_async_commit();
    };

    Pos ahead = cur;
#pragma unroll
    for (int s = 0; s < S - 1; ++s) {
        issue(ahead, slot_of(ahead), s);
        advance(ahead);
    }

    int buf = 1;
    int rp = 0;                       // reduction buffer parity, alternates every token
    bool rd = false, wr = false;
    unsigned char* dst_state = nullptr;
    int64_t v_off = 0, o_off = 0;
    unsigned char* inter_base = nullptr;
    const float scale = p.scale;
    int stage = 0;
    int stage_next = S - 1;
#pragma unroll 1
    for (; cur.tile < t_end; advance(cur)) {
        const int64_t r_ahead = slot_of(ahead);
        const int b = cur.b, hv = cur.hv, vt = cur.vt;
        const bool cv = vt * TVC + col0 < V;   // this thread's column chunk exists
        if (vt == 0 || cur.tile == t_begin) {
            const int h = hv / p.group;
            buf ^= 1;
            const int64_t r = ld_idx(p.ridx, b * p.ri_s, p.ri_dt);
            const int64_t w = p.widx ? ld_idx(p.widx, b * p.wi_s, p.wi_dt) : r;
            rd = r >= 0 && r < p.P;
            wr = w >= 0 && w < p.P;
            if (threadIdx.x == 0 && hv == 0 && p.dev_err) {
                const int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0);
                if (e) atomicOr(p.dev_err, e);
            }
            dst_state = static_cast<unsigned char*>(p.pool) +
                        ((wr ? w : 0) * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1]) * SB;
            v_off = b * p.vs[0] + hv * p.vs[2];
            o_off = b * p.os[0] + hv * p.os[2];
            if (p.inter) inter_base = static_cast<unsigned char*>(p.inter) + (b * p.is[0] + hv * p.is[2]) * inter_es;
            build_pair_vectors<FORM, K, NW>(p, vecs + buf * vstride, b, hv, h, v_off, sv_on, o_k, o_d, o_v, o_s);
        }

        cp_async_wait<S - 2>();
        float s[NRK][EPC];
        {
            const unsigned char* src = ring + stage * STAGE + s_row0;
#pragma unroll
            for (int i = 0; i < NRK; ++i) {
                if (rd && cv) {
                    chunk_to_f32<SB>(src + i * S_RSTEP, s[i]);
                } else {
#pragma unroll
                    for (int e = 0; e < EPC; ++e) s[i][e] = 0.f;
                }
            }
        }
        issue(ahead, r_ahead, stage_next);
        advance(ahead);
        stage = stage + 1 == S ? 0 : stage + 1;
        stage_next = stage_next + 1 == S ? 0 : stage_next + 1;

        const float* vb = vecs + buf * vstride;
        const float* sc = vb + o_s;
#pragma unroll 1
        for (int t = 0; t < T; ++t) {
            const float bt = sc[t], dec = sc[T + t];
            const float iq = sc[2 * T + t], ik = sc[3 * T + t], kq = sc[4 * T + t];
            float kr[NRK], qr[NRK];
#pragma unroll
            for (int i = 0; i < NRK; ++i) {
                const int kk = rg + i * RG;
                kr[i] = vb[o_k + t * K + kk];
                qr[i] = vb[t * K + kk];
                const float d = FORM == FORM_KDA ? vb[o_d + t * K + kk] : dec;
#pragma unroll
                for (int e = 0; e < EPC; ++e) s[i][e] *= d;
            }
            // sums over this thread's rows, then over the warp's row lanes
            float u[EPC], pq[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                float a = 0.f, c = 0.f;
#pragma unroll
                for (int i = 0; i < NRK; ++i) {
                    a = fmaf(s[i][e], kr[i], a);
                    c = fmaf(s[i][e], qr[i], c);
                }
#pragma unroll
                for (int off = CL; off < 32; off <<= 1) {
                    a += __shfl_xor_sync(0xffffffffu, a, off);
                    c += __shfl_xor_sync(0xffffffffu, c, off);
                }
                u[e] = a;
                pq[e] = c;
            }
            // then over the warps, through shared memory
            float* rb = red + rp * (NW * 2 * TVC);
            if (rl == 0) {
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    rb[(warp * 2 + 0) * TVC + col0 + e] = u[e];
                    rb[(warp * 2 + 1) * TVC + col0 + e] = pq[e];
                }
            }
            __syncthreads();
            rp ^= 1;
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                float a = 0.f, c = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) {
                    a += rb[(w2 * 2 + 0) * TVC + col0 + e];
                    c += rb[(w2 * 2 + 1) * TVC + col0 + e];
                }
                const int col = vt * TVC + col0 + e;
                float vval = 0.f;
                if (cv) vval = sv_on ? vb[o_v + t * V + col] : ld_in(p.v, v_off + t * p.vs[1] + col * p.vs[3], p.v_dt);
                float o, coef;
                if constexpr (FORM == FORM_LA) {
                    coef = vval * ik;
                    o = fmaf(vval, kq, c * iq);
                } else {
                    const float delta = bt * (vval - a * ik);
                    coef = delta * ik;
                    o = fmaf(delta, kq, c * iq);
                }
                if (warp == 0 && rl == 0 && cv)
                    st_out(p.out, o_off + t * p.os[1] + col * p.os[3], p.out_dt, o * scale);
#pragma unroll
                for (int i = 0; i < NRK; ++i) s[i][e] = fmaf(coef, kr[i], s[i][e]);
            }
            if (p.inter != nullptr && cv) {
                unsigned char* ip = inter_base + (t * p.is[1] + static_cast<int64_t>(rg) * p.is[3] +
                                                  vt * TVC + col0) * inter_es;
#pragma unroll
                for (int i = 0; i < NRK; ++i)
                    store_run<EPC>(ip + static_cast<int64_t>(i) * RG * p.is[3] * inter_es, s[i], inter_bf16);
            }
        }

        if (wr && cv) {
            unsigned char* wb = dst_state + vt * G_TILE + g_row0;
#pragma unroll
            for (int i = 0; i < NRK; ++i) store_run<EPC>(wb + i * g_rstep, s[i], SB == 2);
        }
    }
    cp_async_wait<0>();
}

template <int FORM, int K, int NW, int S, int SB, int MB = 1>
lar_status launch_kv_tile(const DecodeParams& p, cudaStream_t stream) {
    auto kern = decode_kv_kernel<FORM, K, NW, S, SB, MB>;
    const size_t smem = decode_kv_smem_bytes<FORM, K, NW, S, SB>(p.T, p.V);
    constexpr size_t smem_max = decode_kv_smem_bytes<FORM, K, NW, S, SB>(16, kStageVMax / 16);
    int sms = 0;
    const int occ = cached_occupancy(reinterpret_cast<const void*>(kern), NW * 32, smem, smem_max, &sms);
    if (occ < 1) return LAR_ERR_LAUNCH;
    const int nvt = (p.V + KvTile<K, NW, SB>::TVC - 1) / KvTile<K, NW, SB>::TVC;
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

// K x V layout: 4 warps (2 for bf16 at K = 16, whose 32 row lanes would
// otherwise exceed the 16 rows), 2-stage ring.
template <int FORM>
lar_status launch_form_kv(const DecodeParams& p, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    constexpr int MB = LAR_K128_MIN_BLOCKS;
    if (p.pool_dt == LAR_F32) {
        switch (p.K) {
            case 16: return launch_kv_tile<FORM, 16, 4, 2, 4>(p, st);
            case 32: return launch_kv_tile<FORM, 32, 4, 2, 4>(p, st);
            case 64: return launch_kv_tile<FORM, 64, 4, 2, 4>(p, st);
            case 128: return launch_kv_tile<FORM, 128, 4, 2, 4, MB>(p, st);
            default: return LAR_ERR_SHAPE;
        }
    }
    switch (p.K) {
        case 16: return launch_kv_tile<FORM, 16, 2, 2, 2>(p, st);
        case 32: return launch_kv_tile<FORM, 32, 4, 2, 2>(p, st);
        case 64: return launch_kv_tile<FORM, 64, 4, 2, 2>(p, st);
        case 128: return launch_kv_tile<FORM, 128, 4, 2, 2, MB>(p, st);
        default: return LAR_ERR_SHAPE;
    }
}

}  // namespace lar
