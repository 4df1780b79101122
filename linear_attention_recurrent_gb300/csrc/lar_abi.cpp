// lar_abi.cpp -- the exported C entry points: validate every descriptor on the
// host, flatten it into a DecodeParams block and enqueue one kernel.  Nothing
// is launched (and nothing written) unless every check passes.
#include <stdint.h>

#include "decode_params.h"
#include "lar.h"

namespace {

using lar::DecodeParams;

bool is_float(const lar_tensor* t) { return t->dtype == LAR_F32 || t->dtype == LAR_BF16; }
bool is_index(const lar_tensor* t) { return t->dtype == LAR_I32 || t->dtype == LAR_I64; }

int64_t elem_size(int32_t dt) {
    switch (dt) {
        case LAR_F32: return 4;
        case LAR_BF16: return 2;
        case LAR_I32: return 4;
        case LAR_I64: return 8;
        default: return 0;
    }
}

// Rank in 1..5, non-negative sizes and strides.
lar_status check_header(const lar_tensor* t) {
    if (t->ndim < 1 || t->ndim > 5) return LAR_ERR_RANK;
    for (int i = 0; i < t->ndim; ++i) {
        if (t->shape[i] < 0) return LAR_ERR_SHAPE;
        if (t->stride[i] < 0) return LAR_ERR_STRIDE;
    }
    return LAR_OK;
}

// A view with a zero-sized dimension holds no elements and may carry a NULL
// data pointer (torch gives empty tensors one).
bool empty(const lar_tensor* t) {
    for (int i = 0; i < t->ndim && i < 5; ++i)
        if (t->shape[i] == 0) return true;
    return false;
}

bool missing(const lar_tensor* t) { return !t || (!t->data && !empty(t)); }

// Half-open byte range [lo, hi) that a view can touch (empty views touch nothing).
struct Span {
    uintptr_t lo = 0, hi = 0;
};

Span span_of(const lar_tensor* t) {
    Span s;
    if (!t || !t->data) return s;
    int64_t last = 0;
    for (int i = 0; i < t->ndim; ++i) {
        if (t->shape[i] == 0) return s;
        last += (t->shape[i] - 1) * t->stride[i];
    }
    const uintptr_t base = reinterpret_cast<uintptr_t>(t->data);
    s.lo = base;
    s.hi = base + static_cast<uintptr_t>((last + 1) * elem_size(t->dtype));
    return s;
}

bool overlap(const Span& a, const Span& b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// A per-token tensor of logical shape [B, T, heads, X] given at rank `full`
// or rank `full - 1` (T = 1).  Writes strides (b, t, head, x), with t stride 0
// for the short form.  X < 0 means the tensor has no trailing x dimension.
bool per_token_view(const lar_tensor* t, int full, int64_t B, int64_t T, int64_t heads, int64_t X,
                    int64_t st[4]) {
    const bool has_x = X >= 0;
    int64_t shp[4] = {0, 0, 0, 0};
    int64_t str[4] = {0, 0, 0, 0};
    if (t->ndim == full) {
        for (int i = 0; i < full; ++i) { shp[i] = t->shape[i]; str[i] = t->stride[i]; }
    } else if (t->ndim == full - 1 && T == 1) {
        shp[0] = t->shape[0]; str[0] = t->stride[0];
        shp[1] = 1; str[1] = 0;
        for (int i = 1; i < full - 1; ++i) { shp[i + 1] = t->shape[i]; str[i + 1] = t->stride[i]; }
    } else {
        return false;
    }
    if (shp[0] != B || shp[1] != T || shp[2] != heads) return false;
    if (has_x && shp[3] != X) return false;
    for (int i = 0; i < 4; ++i) st[i] = str[i];
    if (!has_x) st[3] = 0;
    return true;
}

// pool: [P, HV, V, K] or flat [P*HV, V, K] (kv: [P, HV, K, V] / [P*HV, K, V]);
// innermost dimension contiguous, 16-byte chunks.  Fills the pool fields of p.
lar_status check_pool(const lar_tensor* pl, int form, int64_t HV, int64_t K, int64_t V, bool kv, DecodeParams& p) {
    const int64_t R1 = kv ? K : V;   // rows of one state
    const int64_t R2 = kv ? V : K;   // elements of one row
    p.state_kv = kv ? 1 : 0;
    if (kv && (R2 * elem_size(pl->dtype)) % 16 != 0) return LAR_ERR_SHAPE;
    int64_t P;
    if (pl->ndim == 4) {
        if (pl->shape[1] != HV || pl->shape[2] != R1 || pl->shape[3] != R2) return LAR_ERR_SHAPE;
        if (pl->stride[3] != 1) return LAR_ERR_STRIDE;
        P = pl->shape[0];
        p.ps[0] = pl->stride[0];
        p.ps[1] = pl->stride[1];
        p.ps[2] = pl->stride[2];
        if (form == lar::FORM_LA && P > 1 && pl->stride[0] != HV * pl->stride[1]) return LAR_ERR_STRIDE;
    } else if (pl->ndim == 3) {
        if (pl->shape[1] != R1 || pl->shape[2] != R2) return LAR_ERR_SHAPE;
        if (pl->shape[0] % HV != 0) return LAR_ERR_SHAPE;
        if (pl->stride[2] != 1) return LAR_ERR_STRIDE;
        P = pl->shape[0] / HV;
        p.ps[0] = pl->stride[0] * HV;
        p.ps[1] = pl->stride[0];
        p.ps[2] = pl->stride[1];
    } else {
        return LAR_ERR_RANK;
    }
    // state rows move as 16-byte chunks: aligned base, strides in whole chunks
    const int64_t pes = elem_size(pl->dtype);
    if (reinterpret_cast<uintptr_t>(pl->data) % 16 != 0) return LAR_ERR_ALIGN;
    if ((p.ps[0] * pes) % 16 || (p.ps[1] * pes) % 16 || (p.ps[2] * pes) % 16) return LAR_ERR_ALIGN;
    p.P = P;
    p.pool = pl->data;
    p.pool_dt = pl->dtype;
    return LAR_OK;
}

// read / write slot vectors [B] (write may be NULL: the read slot).
lar_status check_slots(const lar_tensor* read_idx, const lar_tensor* write_idx, int64_t B, DecodeParams& p) {
    if (read_idx->ndim != 1) return LAR_ERR_RANK;
    if (read_idx->shape[0] != B) return LAR_ERR_SHAPE;
    if (!is_index(read_idx)) return LAR_ERR_DTYPE;
    p.ridx = read_idx->data; p.ri_s = read_idx->stride[0]; p.ri_dt = read_idx->dtype;
    if (write_idx) {
        if (missing(write_idx)) return LAR_ERR_NULL;
        if (write_idx->ndim != 1) return LAR_ERR_RANK;
        if (write_idx->shape[0] != B) return LAR_ERR_SHAPE;
        if (!is_index(write_idx)) return LAR_ERR_DTYPE;
        p.widx = write_idx->data; p.wi_s = write_idx->stride[0]; p.wi_dt = write_idx->dtype;
    } else {
        p.widx = nullptr; p.wi_s = 0; p.wi_dt = LAR_I32;
    }
    return LAR_OK;
}

struct Common {
    const lar_tensor *q, *k, *v, *pool, *read_idx, *write_idx, *out, *inter;
};

// Checks shared by every form; fills sizes, q/k/v/out/pool/index/inter fields.
// kv: the state is stored [k][v] (LAR_STATE_KV) instead of [v][k].
lar_status check_common(const Common& c, int form, DecodeParams& p, bool kv = false) {
    if (missing(c.q) || missing(c.k) || missing(c.v) || missing(c.pool) || missing(c.read_idx) ||
        missing(c.out))
        return LAR_ERR_NULL;
    const lar_tensor* all[] = {c.q, c.k, c.v, c.pool, c.read_idx, c.write_idx, c.out, c.inter};
    for (const lar_tensor* t : all) {
        if (!t) continue;
        const lar_status st = check_header(t);
        if (st != LAR_OK) return st;
    }

    if (c.q->ndim != 3 && c.q->ndim != 4) return LAR_ERR_RANK;
    if (c.k->ndim != c.q->ndim || c.v->ndim != c.q->ndim || c.out->ndim != c.q->ndim) return LAR_ERR_RANK;
    if (!is_float(c.q) || !is_float(c.k) || !is_float(c.v) || !is_float(c.out)) return LAR_ERR_DTYPE;
    if (!is_float(c.pool)) return LAR_ERR_DTYPE;

    const bool short_form = c.q->ndim == 3;
    const int64_t B = c.q->shape[0];
    const int64_t T = short_form ? 1 : c.q->shape[1];
    const int64_t H = c.q->shape[short_form ? 1 : 2];
    const int64_t K = c.q->shape[short_form ? 2 : 3];
    const int64_t HV = c.v->shape[short_form ? 1 : 2];
    const int64_t V = c.v->shape[short_form ? 2 : 3];
    if (K != 16 && K != 32 && K != 64 && K != 128) return LAR_ERR_SHAPE;
    if (T < 1 || T > 16 || H < 1 || HV < 1 || V < 1 || B > 65535 || HV > 65535 || V > (1 << 24))
        return LAR_ERR_SHAPE;
    if (HV % H != 0) return LAR_ERR_SHAPE;
    if (form == lar::FORM_LA && HV != H) return LAR_ERR_SHAPE;

    p.form = form;
    p.B = static_cast<int>(B);
    p.T = static_cast<int>(T);
    p.H = static_cast<int>(H);
    p.HV = static_cast<int>(HV);
    p.K = static_cast<int>(K);
    p.V = static_cast<int>(V);
    p.group = static_cast<int>(HV / H);

    if (!per_token_view(c.q, 4, B, T, H, K, p.qs)) return LAR_ERR_SHAPE;
    if (!per_token_view(c.k, 4, B, T, H, K, p.ks)) return LAR_ERR_SHAPE;
    if (!per_token_view(c.v, 4, B, T, HV, V, p.vs)) return LAR_ERR_SHAPE;
    if (!per_token_view(c.out, 4, B, T, HV, V, p.os)) return LAR_ERR_SHAPE;
    p.q = c.q->data; p.q_dt = c.q->dtype;
    p.k = c.k->data; p.k_dt = c.k->dtype;
    p.v = c.v->data; p.v_dt = c.v->dtype;
    p.out = c.out->data; p.out_dt = c.out->dtype;

    lar_status st = check_pool(c.pool, form, HV, K, V, kv, p);
    if (st != LAR_OK) return st;
    st = check_slots(c.read_idx, c.write_idx, B, p);
    if (st != LAR_OK) return st;
    const int64_t R1 = kv ? K : V;   // rows of one state
    const int64_t R2 = kv ? V : K;   // elements of one row

    // intermediate-state cache: [B, T, HV, V, K] (rank 4 [B, HV, V, K] for T = 1)
    p.inter = nullptr;
    p.inter_dt = LAR_F32;
    for (int i = 0; i < 4; ++i) p.is[i] = 0;
    if (c.inter) {
        const lar_tensor* it = c.inter;
        if (missing(it)) return LAR_ERR_NULL;
        if (!is_float(it)) return LAR_ERR_DTYPE;
        int64_t shp[5], str[5];
        if (it->ndim == 5) {
            for (int i = 0; i < 5; ++i) { shp[i] = it->shape[i]; str[i] = it->stride[i]; }
        } else if (it->ndim == 4 && T == 1) {
            shp[0] = it->shape[0]; str[0] = it->stride[0];
            shp[1] = 1; str[1] = 0;
            for (int i = 1; i < 4; ++i) { shp[i + 1] = it->shape[i]; str[i + 1] = it->stride[i]; }
        } else {
            return LAR_ERR_RANK;
        }
        if (shp[0] != B || shp[1] != T || shp[2] != HV || shp[3] != R1 || shp[4] != R2) return LAR_ERR_SHAPE;
        if (str[4] != 1) return LAR_ERR_STRIDE;
        // cached rows are written in aligned runs of 8 or 16 bytes: aligned base, 16-byte strides
        const int64_t ies = elem_size(it->dtype);
        if (reinterpret_cast<uintptr_t>(it->data) % 16 != 0) return LAR_ERR_ALIGN;
        if ((str[0] * ies) % 16 || (str[1] * ies) % 16 || (str[2] * ies) % 16 || (str[3] * ies) % 16)
            return LAR_ERR_ALIGN;
        p.inter = it->data;
        p.inter_dt = it->dtype;
        for (int i = 0; i < 4; ++i) p.is[i] = str[i];
    }
    return LAR_OK;
}

// Outputs overlap neither each other nor any input.  The device error word
// (written with atomicOr by the kernels) is a 4-byte output too: aligned to 4
// bytes and clear of every tensor of the call.
lar_status check_aliasing(const lar_tensor* const* outs, int n_out, const lar_tensor* const* ins, int n_in,
                          const int32_t* dev_err) {
    if (dev_err) {
        if (reinterpret_cast<uintptr_t>(dev_err) % alignof(int32_t) != 0) return LAR_ERR_ALIGN;
        Span e;
        e.lo = reinterpret_cast<uintptr_t>(dev_err);
        e.hi = e.lo + sizeof(int32_t);
        for (int i = 0; i < n_out; ++i)
            if (outs[i] && overlap(e, span_of(outs[i]))) return LAR_ERR_ALIAS;
        for (int j = 0; j < n_in; ++j)
            if (ins[j] && overlap(e, span_of(ins[j]))) return LAR_ERR_ALIAS;
    }
    for (int i = 0; i < n_out; ++i) {
        if (!outs[i]) continue;
        const Span a = span_of(outs[i]);
        for (int j = i + 1; j < n_out; ++j)
            if (outs[j] && overlap(a, span_of(outs[j]))) return LAR_ERR_ALIAS;
        for (int j = 0; j < n_in; ++j)
            if (ins[j] && overlap(a, span_of(ins[j]))) return LAR_ERR_ALIAS;
    }
    return LAR_OK;
}

// A 1-D fp32 parameter vector of length n (A_log, dt_bias, decay).
lar_status check_vec(const lar_tensor* t, int64_t n, const float** ptr, int64_t* stride) {
    const lar_status st = check_header(t);
    if (st != LAR_OK) return st;
    if (missing(t)) return LAR_ERR_NULL;
    if (t->ndim != 1) return LAR_ERR_RANK;
    if (t->shape[0] != n) return LAR_ERR_SHAPE;
    if (t->dtype != LAR_F32) return LAR_ERR_DTYPE;
    *ptr = static_cast<const float*>(t->data);
    *stride = t->stride[0];
    return LAR_OK;
}

// num_accepted / state_idx select the per-token-slot mode (state_idx != NULL).
lar_status delta_rule(int form, const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                      const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                      const lar_tensor* dt_bias, const lar_tensor* pool, const lar_tensor* read_idx,
                      const lar_tensor* write_idx, const lar_tensor* num_accepted,
                      const lar_tensor* state_idx, const lar_tensor* out, const lar_tensor* inter,
                      float scale, uint32_t flags, int32_t* dev_err, void* stream) {
    DecodeParams p{};
    if (flags & ~static_cast<uint32_t>(LAR_QK_L2NORM | LAR_GATE_RAW | LAR_BETA_RAW | LAR_STATE_KV))
        return LAR_ERR_ARG;
    const bool tok = state_idx != nullptr;
    const bool kv = (flags & LAR_STATE_KV) != 0;
    if (tok && kv) return LAR_ERR_ARG;   // per-token slots are served for the [v][k] layout only
    if (tok && (read_idx == nullptr) == (num_accepted == nullptr)) return LAR_ERR_ARG;
    // the seed source ([B] index vector) goes through the common checks as the read index
    const lar_tensor* seed = read_idx ? read_idx : num_accepted;
    lar_status st = check_common(Common{q, k, v, pool, seed, write_idx, out, inter}, form, p, kv);
    if (st != LAR_OK) return st;
    p.nacc = nullptr; p.na_s = 0; p.na_dt = LAR_I32;
    p.tslot = nullptr; p.tsl_s[0] = p.tsl_s[1] = 0; p.tsl_dt = LAR_I32;
    if (tok) {
        if (missing(state_idx)) return LAR_ERR_NULL;
        if ((st = check_header(state_idx)) != LAR_OK) return st;
        // rank 2 only: a flat table read with a guessed row stride is the bug the aiter review found
        if (state_idx->ndim != 2) return LAR_ERR_RANK;
        if (state_idx->shape[0] != p.B || state_idx->shape[1] != p.T) return LAR_ERR_SHAPE;
        if (!is_index(state_idx)) return LAR_ERR_DTYPE;
        p.tslot = state_idx->data;
        p.tsl_s[0] = state_idx->stride[0];
        p.tsl_s[1] = state_idx->stride[1];
        p.tsl_dt = state_idx->dtype;
        if (num_accepted) {
            p.nacc = num_accepted->data;
            p.na_s = num_accepted->stride[0];
            p.na_dt = num_accepted->dtype;
            p.ridx = nullptr;
        }
    }
    if (missing(g) || missing(beta)) return LAR_ERR_NULL;
    if ((st = check_header(g)) != LAR_OK) return st;
    if ((st = check_header(beta)) != LAR_OK) return st;
    if (!is_float(g) || !is_float(beta)) return LAR_ERR_DTYPE;
    const bool kda = form == lar::FORM_KDA;
    if (!per_token_view(g, kda ? 4 : 3, p.B, p.T, p.HV, kda ? p.K : -1, p.gs)) return LAR_ERR_SHAPE;
    int64_t bst[4];
    if (!per_token_view(beta, 3, p.B, p.T, p.HV, -1, bst)) return LAR_ERR_SHAPE;
    for (int i = 0; i < 3; ++i) p.bs[i] = bst[i];
    p.g = g->data; p.g_dt = g->dtype;
    p.beta = beta->data; p.beta_dt = beta->dtype;

    // Gate parameters only make sense with the in-kernel gate: the aiter review
    // found a wrapper that accepted them without the flag and silently ran
    // ungated decay.
    const bool raw = (flags & LAR_GATE_RAW) != 0;
    if (!raw && (A_log || dt_bias)) return LAR_ERR_ARG;
    if (raw && !A_log) return LAR_ERR_NULL;
    p.A_log = nullptr; p.A_s = 0; p.dt_bias = nullptr; p.dtb_s = 0;
    if (raw) {
        st = check_vec(A_log, p.HV, &p.A_log, &p.A_s);
        if (st != LAR_OK) return st;
        if (dt_bias) {
            st = check_vec(dt_bias, kda ? static_cast<int64_t>(p.HV) * p.K : p.HV, &p.dt_bias, &p.dtb_s);
            if (st != LAR_OK) return st;
        }
    }
    p.decay = nullptr; p.dec_s = 0;
    p.scale = scale;
    p.flags = flags;
    p.dev_err = dev_err;

    const lar_tensor* outs[] = {pool, out, inter};
    const lar_tensor* ins[] = {q, k, v, g, beta, A_log, dt_bias, read_idx, write_idx, num_accepted, state_idx};
    st = check_aliasing(outs, 3, ins, 11, dev_err);
    if (st != LAR_OK) return st;
    if (p.B == 0) return LAR_OK;
    return kda ? lar::launch_kda(p, stream) : lar::launch_gdn(p, stream);
}

// Variable-length spans: token-major q/k [Ntok, H, K], v / out [Ntok, HV, V],
// g [Ntok, HV] (KDA [Ntok, HV, K]), beta [Ntok, HV], cu_seqlens [N+1], slots
// [N], cache [Ntok, HV, V, K] or NULL.  Sequence n owns tokens
// cu_seqlens[n] .. cu_seqlens[n+1] - 1.  g / beta / A_log / dt_bias are NULL
// for LA, decay NULL for GDN / KDA.
lar_status varlen(int form, const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                  const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                  const lar_tensor* dt_bias, const lar_tensor* decay, const lar_tensor* pool,
                  const lar_tensor* cu_seqlens, const lar_tensor* read_idx, const lar_tensor* write_idx,
                  const lar_tensor* out, const lar_tensor* inter, float scale, uint32_t flags,
                  int32_t* dev_err, void* stream, bool prefill = false) {
    DecodeParams p{};
    const bool delta = form != lar::FORM_LA;
    if (flags & ~static_cast<uint32_t>(LAR_QK_L2NORM | LAR_GATE_RAW | LAR_BETA_RAW)) return LAR_ERR_ARG;
    if (missing(q) || missing(k) || missing(v) || missing(pool) || missing(cu_seqlens) || missing(read_idx) ||
        missing(out))
        return LAR_ERR_NULL;
    if (delta && (missing(g) || missing(beta))) return LAR_ERR_NULL;
    const lar_tensor* all[] = {q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx, out, inter};
    for (const lar_tensor* t : all) {
        if (!t) continue;
        const lar_status st = check_header(t);
        if (st != LAR_OK) return st;
    }
    if (q->ndim != 3 || k->ndim != 3 || v->ndim != 3 || out->ndim != 3) return LAR_ERR_RANK;
    if (!is_float(q) || !is_float(k) || !is_float(v) || !is_float(out) || !is_float(pool)) return LAR_ERR_DTYPE;
    const int64_t NT = q->shape[0], H = q->shape[1], K = q->shape[2];
    const int64_t HV = v->shape[1], V = v->shape[2];
    if (k->shape[0] != NT || k->shape[1] != H || k->shape[2] != K) return LAR_ERR_SHAPE;
    if (v->shape[0] != NT || out->shape[0] != NT || out->shape[1] != HV || out->shape[2] != V) return LAR_ERR_SHAPE;
    if (K != 16 && K != 32 && K != 64 && K != 128) return LAR_ERR_SHAPE;
    if (H < 1 || HV < 1 || V < 1 || HV > 65535 || V > (1 << 24) || NT > INT32_MAX) return LAR_ERR_SHAPE;
    if (HV % H != 0) return LAR_ERR_SHAPE;
    if (!delta && HV != H) return LAR_ERR_SHAPE;
    // the chunked prefill kernel is built for K = V = 128 and keeps no per-token states
    if (prefill && (K != 128 || V != 128)) return LAR_ERR_SHAPE;
    if (prefill && inter) return LAR_ERR_ARG;
    if (cu_seqlens->ndim != 1) return LAR_ERR_RANK;
    if (!is_index(cu_seqlens)) return LAR_ERR_DTYPE;
    const int64_t N = cu_seqlens->shape[0] - 1;
    if (N < 0 || N > 65535) return LAR_ERR_SHAPE;

    p.form = form;
    p.B = static_cast<int>(N);
    // tokens staged per chunk (set below, once the pool type is known)
    p.H = static_cast<int>(H);
    p.HV = static_cast<int>(HV);
    p.K = static_cast<int>(K);
    p.V = static_cast<int>(V);
    p.group = static_cast<int>(HV / H);
    // (sequence, token, head, x) strides: the sequence term is 0, tokens are
    // addressed through cu_seqlens
    const lar_tensor* tv[] = {q, k, v, out};
    int64_t* dst[] = {p.qs, p.ks, p.vs, p.os};
    for (int i = 0; i < 4; ++i) {
        dst[i][0] = 0;
        for (int d = 0; d < 3; ++d) dst[i][d + 1] = tv[i]->stride[d];
    }
    p.q = q->data; p.q_dt = q->dtype;
    p.k = k->data; p.k_dt = k->dtype;
    p.v = v->data; p.v_dt = v->dtype;
    p.out = out->data; p.out_dt = out->dtype;
    lar_status st = check_pool(pool, form, HV, K, V, false, p);
    if (st != LAR_OK) return st;
    p.T = p.pool_dt == LAR_BF16 ? lar::kVarlenChunkBf16 : lar::kVarlenChunk;
    if ((st = check_slots(read_idx, write_idx, N, p)) != LAR_OK) return st;
    p.cu = cu_seqlens->data; p.cu_s = cu_seqlens->stride[0]; p.cu_dt = cu_seqlens->dtype;
    p.ntok = NT;

    // per-token state cache [Ntok, HV, V, K]
    p.inter = nullptr; p.inter_dt = LAR_F32;
    for (int i = 0; i < 4; ++i) p.is[i] = 0;
    if (inter) {
        if (missing(inter)) return LAR_ERR_NULL;
        if (!is_float(inter)) return LAR_ERR_DTYPE;
        if (inter->ndim != 4) return LAR_ERR_RANK;
        if (inter->shape[0] != NT || inter->shape[1] != HV || inter->shape[2] != V || inter->shape[3] != K)
            return LAR_ERR_SHAPE;
        if (inter->stride[3] != 1) return LAR_ERR_STRIDE;
        const int64_t ies = elem_size(inter->dtype);
        if (reinterpret_cast<uintptr_t>(inter->data) % 16 != 0) return LAR_ERR_ALIGN;
        for (int d = 0; d < 3; ++d)
            if ((inter->stride[d] * ies) % 16) return LAR_ERR_ALIGN;
        p.inter = inter->data;
        p.inter_dt = inter->dtype;
        p.is[1] = inter->stride[0]; p.is[2] = inter->stride[1]; p.is[3] = inter->stride[2];
    }

    p.nacc = nullptr; p.tslot = nullptr;
    p.A_log = nullptr; p.A_s = 0; p.dt_bias = nullptr; p.dtb_s = 0;
    p.decay = nullptr; p.dec_s = 0;
    if (delta) {
        const bool kda = form == lar::FORM_KDA;
        if (!is_float(g) || !is_float(beta)) return LAR_ERR_DTYPE;
        if (g->ndim != (kda ? 3 : 2) || beta->ndim != 2) return LAR_ERR_RANK;
        if (g->shape[0] != NT || g->shape[1] != HV || (kda && g->shape[2] != K)) return LAR_ERR_SHAPE;
        if (beta->shape[0] != NT || beta->shape[1] != HV) return LAR_ERR_SHAPE;
        p.gs[0] = 0; p.gs[1] = g->stride[0]; p.gs[2] = g->stride[1]; p.gs[3] = kda ? g->stride[2] : 0;
        p.bs[0] = 0; p.bs[1] = beta->stride[0]; p.bs[2] = beta->stride[1];
        p.g = g->data; p.g_dt = g->dtype;
        p.beta = beta->data; p.beta_dt = beta->dtype;
        const bool raw = (flags & LAR_GATE_RAW) != 0;
        if (!raw && (A_log || dt_bias)) return LAR_ERR_ARG;
        if (raw && !A_log) return LAR_ERR_NULL;
        if (raw) {
            if ((st = check_vec(A_log, HV, &p.A_log, &p.A_s)) != LAR_OK) return st;
            if (dt_bias && (st = check_vec(dt_bias, kda ? HV * K : HV, &p.dt_bias, &p.dtb_s)) != LAR_OK) return st;
        }
    } else {
        if (g || beta || A_log || dt_bias || flags) return LAR_ERR_ARG;
        if (!decay) return LAR_ERR_NULL;
        if ((st = check_vec(decay, H, &p.decay, &p.dec_s)) != LAR_OK) return st;
        p.g = nullptr; p.beta = nullptr;
    }
    p.scale = scale;
    p.flags = flags;
    p.dev_err = dev_err;

    const lar_tensor* outs[] = {pool, out, inter};
    const lar_tensor* ins[] = {q, k, v, g, beta, A_log, dt_bias, decay, cu_seqlens, read_idx, write_idx};
    if ((st = check_aliasing(outs, 3, ins, 11, dev_err)) != LAR_OK) return st;
    if (N == 0) return LAR_OK;
    if (prefill) return lar::launch_prefill(p, stream);
    // Without a state cache, spans of kVarlenSplit tokens or more run in the
    // chunked form (several times cheaper per token from about a dozen tokens on)
    // and the token-by-token kernel skips them: two launches, each deciding per
    // span on the device from cu_seqlens.
    if (!inter && K == 128 && V == 128 && lar::kVarlenSplit > 0) {
        p.split_len = lar::kVarlenSplit;
        if ((st = lar::launch_prefill(p, stream)) != LAR_OK) return st;
    }
    switch (form) {
        case lar::FORM_GDN: return lar::launch_gdn(p, stream);
        case lar::FORM_KDA: return lar::launch_kda(p, stream);
        default: return lar::launch_la(p, stream);
    }
}

}  // namespace

extern "C" {

lar_status gdn_decode(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                      const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                      const lar_tensor* dt_bias, const lar_tensor* pool,
                      const lar_tensor* read_idx, const lar_tensor* write_idx,
                      const lar_tensor* out, const lar_tensor* inter, float scale, uint32_t flags,
                      int32_t* dev_err, void* stream) {
    return delta_rule(lar::FORM_GDN, q, k, v, g, beta, A_log, dt_bias, pool, read_idx, write_idx,
                      nullptr, nullptr, out, inter, scale, flags, dev_err, stream);
}

lar_status kda_decode(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                      const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                      const lar_tensor* dt_bias, const lar_tensor* pool,
                      const lar_tensor* read_idx, const lar_tensor* write_idx,
                      const lar_tensor* out, const lar_tensor* inter, float scale, uint32_t flags,
                      int32_t* dev_err, void* stream) {
    return delta_rule(lar::FORM_KDA, q, k, v, g, beta, A_log, dt_bias, pool, read_idx, write_idx,
                      nullptr, nullptr, out, inter, scale, flags, dev_err, stream);
}

lar_status gdn_decode_tokens(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                             const lar_tensor* dt_bias, const lar_tensor* pool,
                             const lar_tensor* read_idx, const lar_tensor* num_accepted,
                             const lar_tensor* state_idx, const lar_tensor* out, float scale,
                             uint32_t flags, int32_t* dev_err, void* stream) {
    if (!state_idx) return LAR_ERR_NULL;
    return delta_rule(lar::FORM_GDN, q, k, v, g, beta, A_log, dt_bias, pool, read_idx, nullptr,
                      num_accepted, state_idx, out, nullptr, scale, flags, dev_err, stream);
}

lar_status kda_decode_tokens(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                             const lar_tensor* dt_bias, const lar_tensor* pool,
                             const lar_tensor* read_idx, const lar_tensor* num_accepted,
                             const lar_tensor* state_idx, const lar_tensor* out, float scale,
                             uint32_t flags, int32_t* dev_err, void* stream) {
    if (!state_idx) return LAR_ERR_NULL;
    return delta_rule(lar::FORM_KDA, q, k, v, g, beta, A_log, dt_bias, pool, read_idx, nullptr,
                      num_accepted, state_idx, out, nullptr, scale, flags, dev_err, stream);
}

lar_status la_decode(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                     const lar_tensor* decay, const lar_tensor* pool, const lar_tensor* read_idx,
                     const lar_tensor* write_idx, const lar_tensor* out, const lar_tensor* inter,
                     float scale, int32_t* dev_err, void* stream) {
    DecodeParams p{};
    lar_status st = check_common(Common{q, k, v, pool, read_idx, write_idx, out, inter}, lar::FORM_LA, p);
    if (st != LAR_OK) return st;
    if (!decay) return LAR_ERR_NULL;
    st = check_vec(decay, p.H, &p.decay, &p.dec_s);
    if (st != LAR_OK) return st;
    p.g = nullptr; p.beta = nullptr; p.A_log = nullptr; p.dt_bias = nullptr;
    p.nacc = nullptr; p.tslot = nullptr;
    p.scale = scale;
    p.flags = 0;
    p.dev_err = dev_err;
    const lar_tensor* outs[] = {pool, out, inter};
    const lar_tensor* ins[] = {q, k, v, decay, read_idx, write_idx};
    st = check_aliasing(outs, 3, ins, 6, dev_err);
    if (st != LAR_OK) return st;
    if (p.B == 0) return LAR_OK;
    return lar::launch_la(p, stream);
}

lar_status gdn_decode_varlen(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                             const lar_tensor* dt_bias, const lar_tensor* pool, const lar_tensor* cu_seqlens,
                             const lar_tensor* read_idx, const lar_tensor* write_idx, const lar_tensor* out,
                             const lar_tensor* inter, float scale, uint32_t flags, int32_t* dev_err,
                             void* stream) {
    return varlen(lar::FORM_GDN, q, k, v, g, beta, A_log, dt_bias, nullptr, pool, cu_seqlens, read_idx,
                  write_idx, out, inter, scale, flags, dev_err, stream);
}

lar_status kda_decode_varlen(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta, const lar_tensor* A_log,
                             const lar_tensor* dt_bias, const lar_tensor* pool, const lar_tensor* cu_seqlens,
                             const lar_tensor* read_idx, const lar_tensor* write_idx, const lar_tensor* out,
                             const lar_tensor* inter, float scale, uint32_t flags, int32_t* dev_err,
                             void* stream) {
    return varlen(lar::FORM_KDA, q, k, v, g, beta, A_log, dt_bias, nullptr, pool, cu_seqlens, read_idx,
                  write_idx, out, inter, scale, flags, dev_err, stream);
}

lar_status la_decode_varlen(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                            const lar_tensor* decay, const lar_tensor* pool, const lar_tensor* cu_seqlens,
                            const lar_tensor* read_idx, const lar_tensor* write_idx, const lar_tensor* out,
                            const lar_tensor* inter, float scale, int32_t* dev_err, void* stream) {
    return varlen(lar::FORM_LA, q, k, v, nullptr, nullptr, nullptr, nullptr, decay, pool, cu_seqlens, read_idx,
                  write_idx, out, inter, scale, 0, dev_err, stream);
}

lar_status gdn_prefill(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v, const lar_tensor* g,
                       const lar_tensor* beta, const lar_tensor* A_log, const lar_tensor* dt_bias,
                       const lar_tensor* pool, const lar_tensor* cu_seqlens, const lar_tensor* read_idx,
                       const lar_tensor* write_idx, const lar_tensor* out, float scale, uint32_t flags,
                       int32_t* dev_err, void* stream) {
    return varlen(lar::FORM_GDN, q, k, v, g, beta, A_log, dt_bias, nullptr, pool, cu_seqlens, read_idx, write_idx,
                  out, nullptr, scale, flags, dev_err, stream, true);
}

lar_status kda_prefill(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v, const lar_tensor* g,
                       const lar_tensor* beta, const lar_tensor* A_log, const lar_tensor* dt_bias,
                       const lar_tensor* pool, const lar_tensor* cu_seqlens, const lar_tensor* read_idx,
                       const lar_tensor* write_idx, const lar_tensor* out, float scale, uint32_t flags,
                       int32_t* dev_err, void* stream) {
    return varlen(lar::FORM_KDA, q, k, v, g, beta, A_log, dt_bias, nullptr, pool, cu_seqlens, read_idx, write_idx,
                  out, nullptr, scale, flags, dev_err, stream, true);
}

lar_status la_prefill(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v, const lar_tensor* decay,
                      const lar_tensor* pool, const lar_tensor* cu_seqlens, const lar_tensor* read_idx,
                      const lar_tensor* write_idx, const lar_tensor* out, float scale, int32_t* dev_err,
                      void* stream) {
    return varlen(lar::FORM_LA, q, k, v, nullptr, nullptr, nullptr, nullptr, decay, pool, cu_seqlens, read_idx,
                  write_idx, out, nullptr, scale, 0, dev_err, stream, true);
}

const char* lar_status_string(lar_status status) {
    switch (status) {
        case LAR_OK: return "ok";
        case LAR_ERR_NULL: return "a required tensor or pointer is NULL";
        case LAR_ERR_DTYPE: return "unsupported dtype";
        case LAR_ERR_RANK: return "wrong tensor rank";
        case LAR_ERR_SHAPE: return "shapes disagree or a size is outside the supported range";
        case LAR_ERR_STRIDE: return "unsupported strides (k stride of pool/inter must be 1; no negative strides)";
        case LAR_ERR_ALIGN:
            return "pool/inter must be 16-byte aligned with strides that are multiples of 16 bytes; "
                   "dev_err 4-byte aligned";
        case LAR_ERR_ARG: return "inconsistent arguments or flags";
        case LAR_ERR_ALIAS: return "an output (dev_err included) overlaps another output or an input";
        case LAR_ERR_LAUNCH: return "kernel launch failed";
    }
    return "unknown status";
}

}  // extern "C"
