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

// K = 128 tile: warps per CTA (row groups of the reduction), ring stages
#ifndef LAR_KV_NW
#define LAR_KV_NW 4
#endif
#ifndef LAR_KV_S
#define LAR_KV_S 2
#endif
#ifndef LAR_KV_MB
#define LAR_KV_MB LAR_K128_MIN_BLOCKS
#endif
// value columns per tile for bf16 pools (fp32: 32, one 128-byte line per row)
#ifndef LAR_KV_BF16_TVC
#define LAR_KV_BF16_TVC 32
#endif
#ifndef LAR_KV_BF16_NW
#define LAR_KV_BF16_NW 2
#endif
#ifndef LAR_KV_BF16_S
#define LAR_KV_BF16_S LAR_KV_S
#endif
#ifndef LAR_KV_BF16_MB
#define LAR_KV_BF16_MB LAR_KV_MB
#endif

namespace lar {

template <int K, int NW, int SB>
struct KvTile {
    static constexpr int EPC = 16 / SB;   // columns per 16-byte chunk
    static constexpr int TVC = SB == 2 ? LAR_KV_BF16_TVC : 32;   // columns per tile
    static constexpr int CL = TVC / EPC;  // lanes across the columns
    static constexpr int RL = 32 / CL;    // lanes of a warp across rows
    static constexpr int RG = NW * RL;    // row groups in the CTA
    static constexpr int NRK = K / RG;    // rows per thread
    static_assert(K % RG == 0 && NRK >= 1, "the rows split evenly over the CTA");
};

template <int K, int NW, int SB>
__host__ __device__ constexpr size_t kv_red_floats() {
    return 2 * static_cast<size_t>(NW) * 2 * KvTile<K, NW, SB>::TVC;   // [2 buffers][NW warps][u, p][TVC columns]
}

template <int FORM, int K, int NW, int S, int SB>
__host__ __device__ constexpr size_t decode_kv_smem_bytes(int T, int V) {
    using G = KvTile<K, NW, SB>;
    return static_cast<size_t>(S) * K * G::TVC * SB +
           (2 * static_cast<size_t>(vec_floats<FORM, K>(T, V)) + kv_red_floats<K, NW, SB>()) * sizeof(float);
}

template <int FORM, int K, int NW, int S, int SB, int MB, int TT>
__global__ void __launch_bounds__(NW * 32, MB)
decode_kv_kernel(const DecodeParams p) {
    using G = KvTile<K, NW, SB>;
    constexpr int EPC = G::EPC, TVC = G::TVC, CL = G::CL, RL = G::RL, RG = G::RG, NRK = G::NRK;
    constexpr int EP = EPC / 2;            // column pairs per chunk

    extern __shared__ __align__(16) unsigned char smem[];
    const int T = TT > 0 ? TT : p.T;
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
    const int o_s = scal_offset(FORM, K, T, V);
    const unsigned char* pool_b = static_cast<const unsigned char*>(p.pool);
    const bool inter_bf16 = p.inter_dt == LAR_BF16;
    const int inter_es = inter_bf16 ? 2 : 4;
    const bool has_inter = TT != 1 && p.inter != nullptr;   // single-token instances run without a cache
    const bool out_bf16 = p.out_dt == LAR_BF16;
    const int out_es = out_bf16 ? 2 : 4;

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

    if (t_begin >= t_end) return;

    // byte offsets fixed for the kernel: rows are RG apart, chunks never move;
    // every address below is a per-pair base advanced by a fixed step per tile
    const int s_row0 = (rg * TVC + col0) * SB;
    constexpr int S_RSTEP = RG * TVC * SB;
    const int64_t g_row0 = (static_cast<int64_t>(rg) * p.ps[2] + col0) * SB;
    const int64_t g_rstep = static_cast<int64_t>(RG) * p.ps[2] * SB;
    constexpr int G_TILE = TVC * SB;
    const int64_t o_cstep = p.os[3] * out_es;                 // between output columns
    const int64_t o_tstep = p.os[1] * out_es;
    const int64_t o_tile = static_cast<int64_t>(TVC) * p.os[3] * out_es;
    const int64_t i_rstep = static_cast<int64_t>(RG) * p.is[3] * inter_es;
    const int64_t i_tstep = p.is[1] * inter_es;
    const int i_tile = TVC * inter_es;

    // ---- issue cursor (see decode_kernel): running source pointer, read slot
    // loaded one tile before the copies need it
    const int64_t n_tiles = t_end - t_begin;
    int64_t a_left = n_tiles;
    int a_vt, a_hv, a_b;
    {
        const int64_t u = t_begin / nvt;
        a_vt = static_cast<int>(t_begin - u * nvt);
        a_b = static_cast<int>(u / p.HV);
        a_hv = static_cast<int>(u - static_cast<int64_t>(a_b) * p.HV);
    }
    const int c_vt0 = a_vt, c_hv0 = a_hv, c_b0 = a_b;
#if LAR_PDL
    // as in decode_kernel: arithmetic above, the first global read below
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
#endif
    int a_rb = a_b;
    int64_t a_r = ld_idx(p.ridx, a_b * p.ri_s, p.ri_dt);
    bool a_new = true, a_ok = false;
    const unsigned char* a_src = pool_b;
    // copies of the next tile into ring stage `st`; chunks with no state behind
    // them (no valid read slot, columns past V) are zeroed in place
    auto issue = [&](int st) {
        if (a_left > 0) {
            if (a_new) {
                a_ok = a_r >= 0 && a_r < p.P;
                a_src = pool_b + ((a_ok ? a_r : 0) * p.ps[0] + static_cast<int64_t>(a_hv) * p.ps[1]) * SB +
                        a_vt * G_TILE + g_row0;
                a_new = false;
            }
            unsigned char* dst = ring + st * STAGE + s_row0;
            const bool ok = a_ok && a_vt * TVC + col0 < V;
#pragma unroll
            for (int i = 0; i < NRK; ++i) {
                if (ok) cp_async16(dst + i * S_RSTEP, a_src + i * g_rstep);
                else st_shared_zero16(dst + i * S_RSTEP);
            }
            if (--a_left > 0) {
                if (++a_vt == nvt) {
                    a_vt = 0;
                    if (++a_hv == p.HV) {
                        a_hv = 0;
                        ++a_b;
                    }
                    if (a_b != a_rb) {
                        a_rb = a_b;
                        a_r = ld_idx(p.ridx, a_b * p.ri_s, p.ri_dt);
                    }
                    a_new = true;
                } else {
                    a_src += G_TILE;
                }
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int s = 0; s < S - 1; ++s) issue(s);

    int c_vt = c_vt0, c_hv = c_hv0, c_b = c_b0;
    int buf = 1;
    int rp = 0;                       // reduction buffer parity, alternates every token
    bool wr = false;
    unsigned char* wb = nullptr;      // this thread's first row chunk of the tile in the write slot
    unsigned char* op = nullptr;      // output of the tile's first column of this thread, token 0
    unsigned char* ip = nullptr;      // its first cached chunk, token 0
    int64_t v_off = 0;
    const float scale = p.scale;
    bool pair_start = true;
    int stage = 0;
    int stage_next = S - 1;
#pragma unroll 1
    for (int64_t n = n_tiles; n > 0; --n) {
        const int b = c_b, hv = c_hv, vt = c_vt;
        const bool cv = vt * TVC + col0 < V;   // this thread's column chunk exists
        if (pair_start) {
            pair_start = false;
            const int h = hv / p.group;
            buf ^= 1;
            const int64_t r = ld_idx(p.ridx, b * p.ri_s, p.ri_dt);
            const int64_t w = p.widx ? ld_idx(p.widx, b * p.wi_s, p.wi_dt) : r;
            wr = w >= 0 && w < p.P;
            if (threadIdx.x == 0 && hv == 0 && p.dev_err) {
                const int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0);
                if (e) atomicOr(p.dev_err, e);
            }
            wb = static_cast<unsigned char*>(p.pool) +
                 ((wr ? w : 0) * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1]) * SB + vt * G_TILE + g_row0;
            const int64_t first_col = static_cast<int64_t>(vt) * TVC + col0;
            v_off = b * p.vs[0] + hv * p.vs[2];
            op = static_cast<unsigned char*>(p.out) + (b * p.os[0] + hv * p.os[2] + first_col * p.os[3]) * out_es;
            if (has_inter)
                ip = static_cast<unsigned char*>(p.inter) +
                     (b * p.is[0] + hv * p.is[2] + static_cast<int64_t>(rg) * p.is[3] + first_col) * inter_es;
            build_pair_vectors<FORM, K, NW, TT>(p, vecs + buf * vstride, b, hv, h, v_off, sv_on, o_k, o_d, o_v, o_s);
        }

        cp_async_wait<S - 2>();
        float2 s[NRK][EP];          // columns 2e (.x) and 2e+1 (.y) of each own row
        {
            const unsigned char* src = ring + stage * STAGE + s_row0;
#pragma unroll
            for (int i = 0; i < NRK; ++i) chunk_to_f2<SB>(src + i * S_RSTEP, s[i]);
        }
        issue(stage_next);
        stage = stage + 1 == S ? 0 : stage + 1;
        stage_next = stage_next + 1 == S ? 0 : stage_next + 1;

        const float* vb = vecs + buf * vstride;
        const float* sc = vb + o_s;
        unsigned char* opt = op;
        unsigned char* ipt = ip;
#pragma unroll 1
        for (int t = 0; t < T; ++t, opt += o_tstep, ipt += i_tstep) {
            const float4 s4 = *reinterpret_cast<const float4*>(sc + kScal * t);
            const float bt = s4.x, dec = s4.y, iq = s4.z, ik = s4.w, kq = sc[kScal * t + 4];
            float2 kr[NRK];   // k of each own row, in both halves
            float2 u[EP], pq[EP];
#pragma unroll
            for (int e = 0; e < EP; ++e) u[e] = pq[e] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NRK; ++i) {
                const int kk = t * K + rg + i * RG;
                const float ki = vb[o_k + kk], qi = vb[kk];
                const float d = FORM == FORM_KDA ? vb[o_d + kk] : dec;
                kr[i] = make_float2(ki, ki);
                const float2 q2 = make_float2(qi, qi), d2 = make_float2(d, d);
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    s[i][e] = __fmul2_rn(s[i][e], d2);
                    u[e] = __ffma2_rn(s[i][e], kr[i], u[e]);
                    pq[e] = __ffma2_rn(s[i][e], q2, pq[e]);
                }
            }
            // sums over this thread's rows are done; now over the warp's row lanes
#pragma unroll
            for (int off = CL; off < 32; off <<= 1) {
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    u[e].x += __shfl_xor_sync(0xffffffffu, u[e].x, off);
                    u[e].y += __shfl_xor_sync(0xffffffffu, u[e].y, off);
                    pq[e].x += __shfl_xor_sync(0xffffffffu, pq[e].x, off);
                    pq[e].y += __shfl_xor_sync(0xffffffffu, pq[e].y, off);
                }
            }
            // then over the warps, through shared memory
            float* rb = red + rp * (NW * 2 * TVC);
            if (rl == 0) {
#pragma unroll
                for (int e = 0; e < EP; ++e) {
                    *reinterpret_cast<float2*>(rb + (warp * 2 + 0) * TVC + col0 + 2 * e) = u[e];
                    *reinterpret_cast<float2*>(rb + (warp * 2 + 1) * TVC + col0 + 2 * e) = pq[e];
                }
            }
            __syncthreads();
            rp ^= 1;
            float2 coef[EP];
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                float2 a = make_float2(0.f, 0.f), c = a;
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) {
                    a = __fadd2_rn(a, *reinterpret_cast<const float2*>(rb + (w2 * 2 + 0) * TVC + col0 + 2 * e));
                    c = __fadd2_rn(c, *reinterpret_cast<const float2*>(rb + (w2 * 2 + 1) * TVC + col0 + 2 * e));
                }
                float o[2], cf[2];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const float ah = h2 ? a.y : a.x, ch = h2 ? c.y : c.x;
                    const int col = vt * TVC + col0 + 2 * e + h2;
                    float vval = 0.f;
                    if (cv) vval = sv_on ? vb[o_v + t * V + col] : ld_in(p.v, v_off + t * p.vs[1] + col * p.vs[3], p.v_dt);
                    if constexpr (FORM == FORM_LA) {
                        cf[h2] = vval * ik;
                        o[h2] = fmaf(vval, kq, ch * iq);
                    } else {
                        const float delta = bt * (vval - ah * ik);
                        cf[h2] = delta * ik;
                        o[h2] = fmaf(delta, kq, ch * iq);
                    }
                }
                coef[e] = make_float2(cf[0], cf[1]);
                if (warp == 0 && rl == 0 && cv) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        unsigned char* dst = opt + (2 * e + h2) * o_cstep;
                        if (out_bf16) *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(o[h2] * scale);
                        else *reinterpret_cast<float*>(dst) = o[h2] * scale;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NRK; ++i)
#pragma unroll
                for (int e = 0; e < EP; ++e) s[i][e] = __ffma2_rn(kr[i], coef[e], s[i][e]);
            if (has_inter && cv) {
#pragma unroll
                for (int i = 0; i < NRK; ++i) store_pairs<EPC>(ipt + i * i_rstep, s[i], inter_bf16);
            }
        }

        if (wr && cv) {
#pragma unroll
            for (int i = 0; i < NRK; ++i) store_pairs<EPC>(wb + i * g_rstep, s[i], SB == 2);
        }

        if (++c_vt == nvt) {
            c_vt = 0;
            if (++c_hv == p.HV) {
                c_hv = 0;
                ++c_b;
            }
            pair_start = true;
        } else {
            wb += G_TILE;
            op += o_tile;
            ip += i_tile;
        }
    }
    cp_async_wait<0>();
}

template <int FORM, int K, int NW, int S, int SB, int MB, int TT>
lar_status launch_kv_tile_mode(const DecodeParams& p, cudaStream_t stream) {
    auto kern = decode_kv_kernel<FORM, K, NW, S, SB, MB, TT>;
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

// T1: compile a separate single-token instance (K = 128).
template <int FORM, int K, int NW, int S, int SB, int MB = 1, bool T1 = false>
lar_status launch_kv_tile(const DecodeParams& p, cudaStream_t stream) {
    if constexpr (T1) {
        if (p.T == 1 && p.inter == nullptr) return launch_kv_tile_mode<FORM, K, NW, S, SB, MB, 1>(p, stream);
    }
    return launch_kv_tile_mode<FORM, K, NW, S, SB, MB, 0>(p, stream);
}

// K x V layout: 4 warps (2 for bf16 at K = 16, whose 32 row lanes would
// otherwise exceed the 16 rows), 2-stage ring.  At K = 128, fp32 with 2 or 8
// warps and a 3-stage ring measured slower (gdn_b64_kv: 5745 / 4657 / 5516
// against 5753 GB/s); bf16 runs 2-warp CTAs (8 rows x 8 columns per thread),
// 27 % faster than 4 warps and far ahead of 8 warps or 64-column tiles.
template <int FORM>
lar_status launch_form_kv(const DecodeParams& p, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (p.pool_dt == LAR_F32) {
        switch (p.K) {
            case 16: return launch_kv_tile<FORM, 16, 4, 2, 4>(p, st);
            case 32: return launch_kv_tile<FORM, 32, 4, 2, 4>(p, st);
            case 64: return launch_kv_tile<FORM, 64, 4, 2, 4>(p, st);
            case 128: return launch_kv_tile<FORM, 128, LAR_KV_NW, LAR_KV_S, 4, LAR_KV_MB, true>(p, st);
            default: return LAR_ERR_SHAPE;
        }
    }
    switch (p.K) {
        case 16: return launch_kv_tile<FORM, 16, 2, 2, 2>(p, st);
        case 32: return launch_kv_tile<FORM, 32, 4, 2, 2>(p, st);
        case 64: return launch_kv_tile<FORM, 64, 4, 2, 2>(p, st);
        case 128: return launch_kv_tile<FORM, 128, LAR_KV_BF16_NW, LAR_KV_BF16_S, 2, LAR_KV_BF16_MB, true>(p, st);
        default: return LAR_ERR_SHAPE;
    }
}

}  // namespace lar
