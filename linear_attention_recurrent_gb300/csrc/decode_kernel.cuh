// decode_kernel.cuh -- the sm_103a decode kernel shared by GDN, KDA and LA.
//
// Work decomposition: one CTA per (V-tile, v-head hv, batch entry b); grid
// (ceil(V / TV), HV, B), sized from the active batch, never from the pool.
// Inside a CTA a state row (one value channel v, all K key channels = K fp32,
// contiguous in the pool) is owned by a group of LPR consecutive lanes; lane j
// of the group holds the 16-byte chunks j, j + LPR, j + 2 LPR, ... of the row,
// so one warp instruction moves RPW = 32 / LPR whole rows in full 128-byte
// lines.  Each thread keeps NR rows in registers for the whole step.
//
// Per token (aiter KDA review recurrence, S^T stored row-wise):
//     s      <- s * exp(g)              (per element for KDA, scalar for GDN)
//     u      =  s . k_hat,  p = s . q_hat     (both reduced over the LPR group)
//     delta  =  beta (v_row - u)
//     s      <- s + delta * k_hat
//     o_row  =  scale * (p + delta * (k_hat . q_hat))      [= scale * s_new . q_hat]
// LA:  s <- lambda s;  p = s . q;  s <- s + v_row k;  o_row = scale (p + v_row (k . q)).
//
// The per-token vectors (q, k, the KDA decay row) and scalars are built once
// per CTA in shared memory (gate chain and l2 norms included) while the state
// loads issued at kernel entry are in flight.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "decode_params.h"

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

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    return fmaf(a.w, b.w, acc);
}

__device__ __forceinline__ void axpy4(float4& s, const float a, const float4 x) {
    s.x = fmaf(a, x.x, s.x);
    s.y = fmaf(a, x.y, s.y);
    s.z = fmaf(a, x.z, s.z);
    s.w = fmaf(a, x.w, s.w);
}

template <int LPR>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Shared-memory bytes the kernel needs for T tokens.
template <int FORM, int K>
__host__ __device__ constexpr size_t decode_smem_bytes(int T) {
    return (static_cast<size_t>(FORM == FORM_KDA ? 3 : 2) * T * K + 5 * static_cast<size_t>(T)) *
           sizeof(float);
}

template <int FORM, int K, int LPR, int NR, int NW>
__global__ void __launch_bounds__(NW * 32)
decode_kernel(const DecodeParams p) {
    constexpr int KPL = K / LPR;       // floats of a row held by one lane
    constexpr int NCH = KPL / 4;       // 16-byte chunks of a row held by one lane
    constexpr int RPW = 32 / LPR;      // rows covered by one warp instruction
    constexpr int TV = NW * NR * RPW;  // rows per CTA
    static_assert(KPL % 4 == 0 && NCH >= 1, "a lane holds whole 16-byte chunks");
    static_assert(32 % LPR == 0, "row groups tile the warp");

    extern __shared__ __align__(16) float smem[];
    const int T = p.T;
    float* sq = smem;                                   // [T][K] q (raw)
    float* sk = sq + T * K;                             // [T][K] k (raw)
    float* sd = sk + T * K;                             // [T][K] KDA exp(g)
    float* sc = sd + (FORM == FORM_KDA ? T * K : 0);    // [5][T] beta, decay, 1/|q|, 1/|k|, k.q

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int j = lane % LPR;
    const int gi = lane / LPR;
    const int b = blockIdx.z;
    const int hv = blockIdx.y;
    const int h = hv / p.group;
    const int v0 = blockIdx.x * TV;

    const int64_t r = ld_idx(p.ridx, b * p.ri_s, p.ri_dt);
    const int64_t w = p.widx ? ld_idx(p.widx, b * p.wi_s, p.wi_dt) : r;
    const bool rd = r >= 0 && r < p.P;
    const bool wr = w >= 0 && w < p.P;
    if (threadIdx.x == 0 && blockIdx.x == 0 && hv == 0 && p.dev_err) {
        const int e = (r >= p.P ? LAR_DEVERR_READ_SLOT : 0) | (w >= p.P ? LAR_DEVERR_WRITE_SLOT : 0);
        if (e) atomicOr(p.dev_err, e);
    }

    // ---- state load: issued first so the preamble overlaps its latency
    float4 s[NR][NCH];
    {
        const float* src = p.pool + (rd ? r : 0) * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int row = v0 + (warp * NR + i) * RPW + gi;
            const bool ok = rd && row < p.V;
            const float4* rp = reinterpret_cast<const float4*>(src + row * p.ps[2]) + j;
#pragma unroll
            for (int c = 0; c < NCH; ++c)
                s[i][c] = ok ? __ldcs(rp + c * LPR) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    // ---- preamble: per-token vectors and scalars into shared memory
    const bool gate_raw = (p.flags & LAR_GATE_RAW) != 0;
    for (int i = threadIdx.x; i < T * K; i += NW * 32) {
        const int t = i / K;
        const int c = i - t * K;
        sq[i] = ld_in(p.q, b * p.qs[0] + t * p.qs[1] + h * p.qs[2] + c * p.qs[3], p.q_dt);
        sk[i] = ld_in(p.k, b * p.ks[0] + t * p.ks[1] + h * p.ks[2] + c * p.ks[3], p.k_dt);
        if constexpr (FORM == FORM_KDA) {
            float x = ld_in(p.g, b * p.gs[0] + t * p.gs[1] + hv * p.gs[2] + c * p.gs[3], p.g_dt);
            if (gate_raw) {
                const float bias =
                    p.dt_bias ? p.dt_bias[(static_cast<int64_t>(hv) * K + c) * p.dtb_s] : 0.f;
                x = -expf(p.A_log[hv * p.A_s]) * softplus_f(x + bias);
            }
            sd[i] = expf(x);
        }
    }
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
    const bool l2 = FORM != FORM_LA && (p.flags & LAR_QK_L2NORM) != 0;
    for (int t = warp; t < T; t += NW) {
        float qq = 0.f, kk = 0.f, kq = 0.f;
        for (int c = lane; c < K; c += 32) {
            const float a = sq[t * K + c], bb = sk[t * K + c];
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
    __syncthreads();

    // ---- token loop: the state never leaves registers between tokens
    const float scale = p.scale;
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
        const float bt = sc[t], dec = sc[T + t];
        const float iq = sc[2 * T + t], ik = sc[3 * T + t], kq = sc[4 * T + t];
        float4 kv[NCH], qv[NCH], dv[NCH];
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int kidx = (c * LPR + j) * 4;
            const float4 a = *reinterpret_cast<const float4*>(sk + t * K + kidx);
            const float4 bq = *reinterpret_cast<const float4*>(sq + t * K + kidx);
            kv[c] = make_float4(a.x * ik, a.y * ik, a.z * ik, a.w * ik);
            qv[c] = make_float4(bq.x * iq, bq.y * iq, bq.z * iq, bq.w * iq);
            if constexpr (FORM == FORM_KDA) dv[c] = *reinterpret_cast<const float4*>(sd + t * K + kidx);
        }
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int row = v0 + (warp * NR + i) * RPW + gi;
            const bool rv = row < p.V;
            const float vval =
                rv ? ld_in(p.v, b * p.vs[0] + t * p.vs[1] + hv * p.vs[2] + row * p.vs[3], p.v_dt) : 0.f;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                if constexpr (FORM == FORM_KDA) {
                    s[i][c].x *= dv[c].x; s[i][c].y *= dv[c].y;
                    s[i][c].z *= dv[c].z; s[i][c].w *= dv[c].w;
                } else {
                    s[i][c].x *= dec; s[i][c].y *= dec; s[i][c].z *= dec; s[i][c].w *= dec;
                }
            }
            float o;
            if constexpr (FORM == FORM_LA) {
                float pp = 0.f;
#pragma unroll
                for (int c = 0; c < NCH; ++c) pp = dot4(s[i][c], qv[c], pp);
                pp = group_sum<LPR>(pp);
#pragma unroll
                for (int c = 0; c < NCH; ++c) axpy4(s[i][c], vval, kv[c]);
                o = fmaf(vval, kq, pp);
            } else {
                float u = 0.f, pp = 0.f;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    u = dot4(s[i][c], kv[c], u);
                    pp = dot4(s[i][c], qv[c], pp);
                }
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) {
                    u += __shfl_xor_sync(0xffffffffu, u, off);
                    pp += __shfl_xor_sync(0xffffffffu, pp, off);
                }
                const float delta = bt * (vval - u);
#pragma unroll
                for (int c = 0; c < NCH; ++c) axpy4(s[i][c], delta, kv[c]);
                o = fmaf(delta, kq, pp);
            }
            if (j == 0 && rv)
                st_out(p.out, b * p.os[0] + t * p.os[1] + hv * p.os[2] + row * p.os[3], p.out_dt, o * scale);
            if (p.inter != nullptr && rv) {
                float4* ip = reinterpret_cast<float4*>(p.inter + b * p.is[0] + t * p.is[1] +
                                                       hv * p.is[2] + row * p.is[3]) + j;
#pragma unroll
                for (int c = 0; c < NCH; ++c) __stcs(ip + c * LPR, s[i][c]);
            }
        }
    }

    // ---- writeback to the write slot (skipped for negative / out-of-range slots)
    if (wr) {
        float* dst = p.pool + w * p.ps[0] + static_cast<int64_t>(hv) * p.ps[1];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int row = v0 + (warp * NR + i) * RPW + gi;
            if (row < p.V) {
                float4* wp = reinterpret_cast<float4*>(dst + row * p.ps[2]) + j;
#pragma unroll
                for (int c = 0; c < NCH; ++c) __stcs(wp + c * LPR, s[i][c]);
            }
        }
    }
}

template <int FORM, int K, int LPR, int NR, int NW>
lar_status launch_tile(const DecodeParams& p, cudaStream_t stream) {
    constexpr int TV = NW * NR * (32 / LPR);
    const dim3 grid(static_cast<unsigned>((p.V + TV - 1) / TV), static_cast<unsigned>(p.HV),
                    static_cast<unsigned>(p.B));
    const size_t smem = decode_smem_bytes<FORM, K>(p.T);
    decode_kernel<FORM, K, LPR, NR, NW><<<grid, NW * 32, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? LAR_OK : LAR_ERR_LAUNCH;
}

// Tile shapes per key size: 8 lanes per 512-byte row at K = 128 (one full line
// per lane group per instruction), 32 rows per CTA of 4 warps.
template <int FORM>
lar_status launch_form(const DecodeParams& p, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (p.K) {
        case 16: return launch_tile<FORM, 16, 4, 2, 2>(p, st);
        case 32: return launch_tile<FORM, 32, 8, 2, 4>(p, st);
        case 64: return launch_tile<FORM, 64, 8, 2, 4>(p, st);
        case 128: return launch_tile<FORM, 128, 8, 2, 4>(p, st);
        default: return LAR_ERR_SHAPE;
    }
}

}  // namespace lar
