// prefill_common.cuh -- what the two tensor-core prefill kernels (prefill_tc.cu,
// prefill_ws.cu) share: the chunk geometry, the tensor-memory columns both give
// the same role, the layout of the M tile (the B operand of O = D M^T, tf32
// halves), and small helpers: the tf32 split into tensor memory, the CTA-wide
// barrier that orders tensor-core work, the decay table, and the launch.
#pragma once

#include "decode_kernel.cuh"
#include "tc_util.cuh"

namespace lar {

// The warp-specialised tensor-core prefill for GDN and LA with bf16 q / k / v
// rows that can be staged (prefill_ws.cu); *launched false: the call does not
// qualify and nothing was launched.
lar_status launch_prefill_ws(const DecodeParams& p, void* stream, bool* launched);

namespace pf {

inline constexpr int TK = 128;       // key channels
inline constexpr int TVV = 128;      // value channels (the M of every product)
inline constexpr int TC = 32;        // tokens per chunk
inline constexpr uint32_t LBO = 144;                      // fp32 tiles: between K-adjacent core matrices
inline constexpr uint32_t MT_SBO = (TC / 4) * LBO + 16;   // M tile: 32 tokens x 32 tokens
inline constexpr uint32_t MT_BYTES = (TC / 8) * MT_SBO;
inline constexpr int TROW = TC + 4;                       // C x C tables (rows 16-byte aligned)
inline constexpr uint32_t STG_ROW = TK * 2;               // one staged bf16 row (TK = TVV)
// sequences ranked by span length in every CTA (at most this many; the ranking
// costs each thread one pass over the spans)
inline constexpr int kLptMax = 256;
// tensor-memory columns: [U | P], [K ; Q] K^T, the state increment; all 512 allocated
inline constexpr uint32_t COL_UP = 256, COL_KK = 320, COL_DS = 384, TMEM_COLS = 512;
static_assert(TVV == TK, "one staged row size for q, k and v");
static_assert(tc::kmaj(TC - 1, TC - 1, LBO, MT_SBO) + 4 <= MT_BYTES, "the M tile holds its elements");

// x (N values, a multiple of 16) into tensor memory as its tf32 halves
template <int N>
__device__ __forceinline__ void split_store(uint32_t taddr_hi, uint32_t taddr_lo, const float* x) {
#pragma unroll
    for (int i0 = 0; i0 < N; i0 += 16) {
        float hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            hi[i] = tc::tf32_hi(x[i0 + i]);
            lo[i] = x[i0 + i] - hi[i];
        }
        tc::tmem_st16(taddr_hi + i0, hi);
        tc::tmem_st16(taddr_lo + i0, lo);
    }
}

// all threads of the CTA: a barrier that also orders tensor-core work around it
__device__ __forceinline__ void tc_sync() {
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Row t of the decay table for lane t of one warp: P[t][s] = a_{s+1} ... a_t
// (products, as the recurrence applies them; 0 above the diagonal),
// E_t = a_0 ... a_t and W_s = P[31][s].
__device__ __forceinline__ void decay_table(int lane, const float* Af, float* Pt, float* E, float* Wd) {
    const int t = lane;
    float f = 1.f;
#pragma unroll 1
    for (int s2 = TC - 1; s2 >= 0; --s2) {
        if (s2 <= t) {
            Pt[t * TROW + s2] = f;
            f *= Af[s2];
        } else {
            Pt[t * TROW + s2] = 0.f;
        }
    }
    E[t] = f;
    __syncwarp();
    Wd[t] = Pt[(TC - 1) * TROW + t];
}

// Launch `kern` over (HV, B) CTAs: one per (v-head, sequence).
template <typename Arg>
inline lar_status launch_kernel(void (*kern)(Arg), int threads, uint32_t smem_bytes, const Arg& a,
                                const DecodeParams& p, cudaStream_t stream) {
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes)) != cudaSuccess)
        return LAR_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.HV), static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
#if LAR_PDL
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
#endif
    return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? LAR_OK : LAR_ERR_LAUNCH;
}

}  // namespace pf
}  // namespace lar
