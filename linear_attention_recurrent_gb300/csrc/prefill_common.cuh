// prefill_common.cuh -- what the two tensor-core prefill kernels (prefill_tc.cu,
// prefill_ws.cu) share: the chunk geometry, the tensor-memory columns both give
// the same role, the layout of the M tile (the B operand of O = D M^T, tf32
// halves), and small helpers: the tf32 split into tensor memory, the CTA-wide
// barrier that orders tensor-core work, the decay table, and the launch.
#pragma once

#include <algorithm>
#include <climits>

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

// Length of span n if it is valid (not reversed, inside the token arrays), else 0.
__device__ __forceinline__ int span_len(const DecodeParams& p, int n, bool& reversed) {
    const int64_t a = ld_idx(p.cu, n * p.cu_s, p.cu_dt), e = ld_idx(p.cu, (n + 1) * p.cu_s, p.cu_dt);
    reversed = e < a;
    return a >= 0 && e >= a && e <= p.ntok ? static_cast<int>(e - a < INT_MAX ? e - a : INT_MAX) : 0;
}

// The sequence of grid row blockIdx.y, or -1 for none; every thread of the
// block calls it and gets the same answer.  Up to kLptMax sequences: the row's
// rank in a longest-first order of the valid spans (ties by index) -- CTAs start
// in blockIdx order, so the longest spans go first and the short ones fill the
// grid's tail (on 16 spans of 256-1024 tokens the simulated makespan drops from
// 1.21x to 1.12x the ideal).  More sequences: row y is sequence y.
// In a split variable-length call (split_len > 0) this kernel takes only the
// valid spans of split_len tokens or more, and only when no span is reversed:
// then the valid spans are disjoint, there are at most ntok / split_len long
// ones, and the launch gives the grid that many rows (not one per sequence).
// A row past the long spans returns -1; with more than kLptMax sequences row y
// takes the y-th long span in index order.  A reversed span anywhere leaves
// every span to the token-by-token kernel (which applies the same test).
// `scratch`: max(kLptMax, NTH / 32) ints of shared memory not otherwise in use
// yet, `pick` one more.
template <int NTH>
__device__ __forceinline__ int pick_sequence(const DecodeParams& p, int* scratch, int* pick) {
    const int tid = threadIdx.x, y = static_cast<int>(blockIdx.y);
    const bool split = p.split_len > 0;
    bool rev = false, r = false;
    if (p.B <= kLptMax) {
        static_assert(NTH >= kLptMax, "one span per thread: the block-wide counts below see every span");
        bool is_long = false;
        if (tid < p.B) {
            const int li = span_len(p, tid, r);
            scratch[tid] = li;
            rev = r;
            is_long = li >= p.split_len;
        }
        const bool any_rev = __syncthreads_or(rev) != 0;
        // a row past the long spans leaves before the ranking (the common case
        // when the call's spans are short); the count needs no further barrier
        // since every thread returns or goes on alike
        if (split && (any_rev || y >= __syncthreads_count(is_long))) return -1;
        for (int i = tid; i < p.B; i += NTH) {
            const int li = scratch[i];
            int rank = 0;
            for (int m = 0; m < p.B; ++m) rank += scratch[m] > li || (scratch[m] == li && m < i);
            if (rank == y) *pick = split && (any_rev || li < p.split_len) ? -1 : i;
        }
        __syncthreads();
        const int n = *pick;
        __syncthreads();   // scratch and pick may be reused
        return n;
    }
    if (!split) return y;
    // count the long spans in index order, blocks of NTH spans at a time (the
    // whole array is read: one reversed span anywhere cancels the split)
    const int lane = tid & 31, warp = tid >> 5;
    int before = 0, n = -1;
    for (int i0 = 0; i0 < p.B; i0 += NTH) {
        const int i = i0 + tid;
        const bool f = i < p.B && span_len(p, i, r) >= p.split_len;
        rev |= i < p.B && r;
        const unsigned m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) scratch[warp] = __popc(m);
        __syncthreads();
        int ahead = before + __popc(m & ((1u << lane) - 1u)), total = 0;
        for (int w = 0; w < NTH / 32; ++w) {
            const int c = scratch[w];
            if (w < warp) ahead += c;
            total += c;
        }
        if (f && ahead == y) *pick = i;
        before += total;
        __syncthreads();   // scratch is rewritten for the next block; pick is final once written
        if (before > y && n < 0) n = *pick;
    }
    const bool any_rev = __syncthreads_or(rev) != 0;
    return any_rev ? -1 : n;
}

// Launch `kern` over (HV, B) CTAs: one per (v-head, sequence); in a split
// variable-length call (v-head, long span) for at most ntok / split_len long
// spans (see pick_sequence), and no launch when no span can be that long.
template <typename Arg>
inline lar_status launch_kernel(void (*kern)(Arg), int threads, uint32_t smem_bytes, const Arg& a,
                                const DecodeParams& p, cudaStream_t stream) {
    int64_t rows = p.B;
    if (p.split_len > 0) rows = std::min<int64_t>(rows, p.ntok / p.split_len);
    if (rows <= 0) return LAR_OK;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(kern), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes)) != cudaSuccess)
        return LAR_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.HV), static_cast<unsigned>(rows));
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
