// decode_params.h -- the validated, flattened argument block handed from the
// C ABI layer (lar_abi.cpp) to the kernel launchers (decode_*.cu).
#pragma once

#include <stdint.h>

#include "lar.h"

namespace lar {

enum Form : int { FORM_GDN = 0, FORM_KDA = 1, FORM_LA = 2 };

// Every stride is in elements.  Per-token tensors are indexed (b, t, head, x);
// a rank-3 input (T = 1) has its t stride set to 0 by the ABI layer.
struct DecodeParams {
    int form;
    int B, T, H, HV, K, V;
    int group;             // HV / H
    int64_t P;             // pool slots

    const void* q;    int64_t qs[4];  int q_dt;
    const void* k;    int64_t ks[4];  int k_dt;
    const void* v;    int64_t vs[4];  int v_dt;
    const void* g;    int64_t gs[4];  int g_dt;    // GDN uses gs[0..2]
    const void* beta; int64_t bs[3];  int beta_dt;
    const float* A_log;   int64_t A_s;            // [HV]
    const float* dt_bias; int64_t dtb_s;          // GDN [HV]; KDA [HV*K]
    const float* decay;   int64_t dec_s;          // LA [H]

    void* pool; int64_t ps[3]; int pool_dt;       // fp32 or bf16; slot, head, row strides (innermost stride 1)
    int state_kv;                                 // 0: rows are v (S^T, k fastest); 1: rows are k (v fastest)
    const void* ridx; int64_t ri_s; int ri_dt;
    const void* widx; int64_t wi_s; int wi_dt;    // NULL: write to the read slot

    const void* nacc;  int64_t na_s; int na_dt;     // accepted-token counts [B] or NULL (seed selection)
    const void* tslot; int64_t tsl_s[2]; int tsl_dt; // per-token write slots [B, T] or NULL

    const void* cu;    int64_t cu_s; int cu_dt;    // varlen: token spans [N+1] or NULL (fixed T)
    int64_t ntok;                                   // varlen: tokens in the q/k/v arrays
    // varlen: spans (valid ones) of at least this many tokens run in the chunked
    // form -- the prefill kernels take only those, the token-by-token kernel skips
    // them; 0: one kernel takes every span
    int split_len;

    void* out;    int64_t os[4]; int out_dt;
    void* inter; int64_t is[4]; int inter_dt;     // fp32 or bf16; b, t, head, row (same layout as the pool); may be NULL

    float scale;
    uint32_t flags;
    int32_t* dev_err;
};

lar_status launch_gdn(const DecodeParams& p, void* stream);
lar_status launch_kda(const DecodeParams& p, void* stream);
lar_status launch_la(const DecodeParams& p, void* stream);
// chunked form over variable-length spans (GDN, KDA and LA, K = V = 128; prefill.cu)
lar_status launch_prefill(const DecodeParams& p, void* stream);
// the same for GDN and LA with the chunk products on the tensor cores (prefill_tc.cu)
lar_status launch_prefill_tc(const DecodeParams& p, void* stream);

// Largest T a call may use (per-pair token tables are sized for it).
constexpr int kMaxTokens = 16;
// Tokens of a variable-length span staged per chunk (at most kMaxTokens): the
// per-token vectors of one chunk live in shared memory, so the chunk size sets
// the CTA's footprint and with it the CTAs per SM.  At K = V = 128, 16-token
// chunks leave room for 2 fp32-pool CTAs per SM, 12 for 3 (18 % faster on a
// mix of short and long spans), and 8 for 4 of the bf16 pool's (16 %).
#ifndef LAR_VL_CHUNK
#define LAR_VL_CHUNK 12
#endif
#ifndef LAR_VL_CHUNK_BF16
#define LAR_VL_CHUNK_BF16 8
#endif
constexpr int kVarlenChunk = LAR_VL_CHUNK;
constexpr int kVarlenChunkBf16 = LAR_VL_CHUNK_BF16;
static_assert(kVarlenChunk >= 1 && kVarlenChunk <= kMaxTokens && kVarlenChunkBf16 >= 1 &&
                  kVarlenChunkBf16 <= kMaxTokens,
              "chunks within the staging capacity");
// A variable-length call without a state cache (K = V = 128) sends spans of at
// least this many tokens to the chunked tensor-core kernels and the rest to the
// token-by-token kernel; 0 keeps every span token by token.
#ifndef LAR_VL_SPLIT
#define LAR_VL_SPLIT 16
#endif
constexpr int kVarlenSplit = LAR_VL_SPLIT;

}  // namespace lar
