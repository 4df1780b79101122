/*
 * lar.h -- C ABI of the recurrent linear-attention decode library (GB300, sm_103a).
 *
 * One decode step of linear attention with a fixed-size recurrent state per
 * (sequence, value head), kept in a paged fp32 state pool.  Three forms:
 *
 *   gdn_decode  gated delta rule, scalar decay per (token, v-head)
 *   kda_decode  gated delta rule, decay per key channel
 *   la_decode   Lightning Attention: decay per head, no delta term
 *
 * with variants for per-token pool slots (gdn_decode_tokens, kda_decode_tokens),
 * token-major spans of any length per sequence (gdn_decode_varlen,
 * kda_decode_varlen, la_decode_varlen) and the chunked form of the latter for
 * long spans (gdn_prefill, kda_prefill, la_prefill).  The chunked calls also set their
 * kernel's shared-memory limit (a function attribute) on every call; capturing
 * them into a CUDA graph has not been tested (the other calls' capture and
 * replay are).
 *
 * The delta-rule recurrence is the one the ROCm/aiter PR #4584 "Fused Gluon KDA
 * decode path" advisory review states: per token
 *     S <- exp(g_t) S;   S <- S + beta_t k_t (x) (v_t - S^T k_t);   o_t = S^T q_t
 * with S a K x V matrix (for KDA exp(g_t) scales key channel k by exp(g_t[k])).
 * Lightning Attention: S <- lambda_h S + k_t (x) v_t;  o_t = S^T q_t.
 * Every output is multiplied by `scale`.
 *
 * Pool addressing (flashinfer "fp32 sibling of #3268" 4D-pool page; cuLA PR #75):
 *   the state of batch entry b and v-head hv is read from slot read_idx[b] and
 *   written to slot write_idx[b] (NULL write_idx: the read slot).  A negative
 *   read index means a zero initial state; a negative write index skips the
 *   writeback.  Every pool byte outside the written (slot, head) states is left
 *   bit-identical.  The pool is read and written in place through its strides.
 *
 * Layouts (all strides in ELEMENTS and non-negative; shape[] is logical):
 *   S is stored transposed: pool[slot][hv][v][k] = S[k][v], k fastest.
 *   pool   fp32 or bf16, rank 4 [P, HV, V, K] (any slot/head/row strides), or
 *          rank 3 [P*HV, V, K] (slot p, head hv at row p*HV + hv).  k stride
 *          must be 1; the data pointer 16-byte aligned; slot, head and row
 *          strides multiples of 16 bytes (rows move as 16-byte chunks).  The
 *          arithmetic is fp32 either way: a bf16 state is widened on load and
 *          rounded to nearest even once per store.
 *   q, k   [B, T, H, K]  (rank 3 [B, H, K] means T = 1); fp32 or bf16, any strides
 *          (so q/k/v may be head-dim slices of one fused buffer).
 *   v      [B, T, HV, V] (rank 3 [B, HV, V]); fp32 or bf16, any strides.
 *   out    [B, T, HV, V] (rank 3 [B, HV, V]); fp32 or bf16 (round to nearest even).
 *          With LAR_STATE_KV (gdn_decode / kda_decode only) the state is held
 *          untransposed, pool[slot][hv][k][v] = S[k][v] with v fastest (the
 *          "nontranspose" layout of the flashinfer GDN decode kernels): rank 4
 *          [P, HV, K, V] or rank 3 [P*HV, K, V], v stride 1, V a multiple of
 *          16 bytes of elements (4 fp32 or 8 bf16); inter is [B, T, HV, K, V].
 *   inter  NULL, or fp32 or bf16 [B, T, HV, V, K] (rank 4 [B, HV, V, K] when
 *          T = 1): the state after each token; same alignment rules as the
 *          pool; its type is independent of the pool's.
 *   read_idx, write_idx  rank 1 [B], int32 or int64, any stride.
 *   H divides HV; v-head hv reads q/k head hv / (HV / H).
 *   K must be 16, 32, 64 or 128; V from 1 to 2^24; T from 1 to 16;
 *   B and HV at most 65535.
 *
 * Ownership and execution: the caller owns every buffer (device memory).
 * Every pointer of a call (tensor data and dev_err) must be memory of the
 * CUDA device that is current on the calling thread, and `stream` a stream of
 * that device: the kernel is launched there and dereferences the pointers
 * as given (memory of another device is not checked here, and a kernel that
 * touches it without peer access faults).  The library allocates nothing, keeps no state between calls and never
 * synchronises: each call validates on the host and then enqueues one kernel
 * on `stream` (a cudaStream_t; NULL is the legacy default stream).  The kernel
 * is launched with programmatic dependent launch: it may be scheduled while
 * the previous kernel on the stream drains, but it reads no memory before that
 * kernel has completed, so stream order is kept.  Calls may be made from
 * several host threads at once (the only host-side state is a per-device cache
 * of occupancy figures, filled under a lock on a kernel's first call) and may
 * be captured into CUDA graphs; make one uncaptured call of a configuration
 * first so that the one-time setup does not fall inside the capture.
 *
 * Errors: a host-detectable problem returns a status other than LAR_OK BEFORE
 * anything is launched (nothing is written).  Slot indices >= P are caught on
 * the device: that entry's state is not read (zero state) / not written, and
 * the bits LAR_DEVERR_* are OR-ed into *dev_err when dev_err is not NULL (a
 * caller-owned device int32, 4-byte aligned (else LAR_ERR_ALIGN) and clear of
 * every tensor of the call (else LAR_ERR_ALIAS); never cleared by the
 * library).  No kernel traps or asserts.
 *
 * Aliasing: pool, out and inter must not overlap one another or any input
 * (checked on the host by address range).  Entries must not read a slot that
 * another entry writes, and write slots must be distinct; such calls are
 * undefined (the kernels run entries concurrently).  In-place update (write
 * slot == read slot of the same entry) is allowed.
 */
#ifndef LAR_H_
#define LAR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LAR_F32 = 0,
    LAR_BF16 = 1,
    LAR_I32 = 2,
    LAR_I64 = 3
} lar_dtype;

/* A strided view of device memory.  data points at element [0, ..., 0]. */
typedef struct {
    void* data;
    int32_t dtype;      /* lar_dtype */
    int32_t ndim;       /* 1..5 */
    int64_t shape[5];
    int64_t stride[5];  /* in elements */
} lar_tensor;

typedef enum {
    LAR_OK = 0,
    LAR_ERR_NULL = 1,        /* a required tensor or pointer is NULL */
    LAR_ERR_DTYPE = 2,       /* unsupported dtype for that argument */
    LAR_ERR_RANK = 3,        /* wrong ndim */
    LAR_ERR_SHAPE = 4,       /* shapes disagree, or a size outside the supported range */
    LAR_ERR_STRIDE = 5,      /* k stride of pool/inter not 1, or negative strides */
    LAR_ERR_ALIGN = 6,       /* pool/inter pointer or strides not multiples of 16 bytes, or dev_err
                                not 4-byte aligned */
    LAR_ERR_ARG = 7,         /* inconsistent flags/arguments (e.g. A_log without LAR_GATE_RAW) */
    LAR_ERR_ALIAS = 8,       /* an output (dev_err included) overlaps another output or an input */
    LAR_ERR_LAUNCH = 9       /* the CUDA launch itself failed */
} lar_status;

/* flags for gdn_decode / kda_decode */
enum {
    LAR_QK_L2NORM = 1u << 0, /* q, k <- x / sqrt(sum x^2 + 1e-6) over K, in kernel */
    LAR_GATE_RAW = 1u << 1,  /* g <- -exp(A_log[hv]) * softplus(g + dt_bias), in kernel */
    LAR_BETA_RAW = 1u << 2,  /* beta <- 1 / (1 + exp(-beta)), in kernel */
    LAR_STATE_KV = 1u << 3   /* pool and inter hold S as [k][v] (v fastest), see below */
};

/* bits OR-ed into *dev_err */
enum {
    LAR_DEVERR_READ_SLOT = 1,  /* some read_idx[b] >= P (that entry started from zero) */
    LAR_DEVERR_WRITE_SLOT = 2, /* some write slot >= P (that writeback was skipped) */
    LAR_DEVERR_ACCEPTED = 4,   /* some num_accepted[b] outside [1, T] (that entry started from zero) */
    LAR_DEVERR_SEQLEN = 8,     /* varlen: some span cu_seqlens[n]..[n+1] reversed or past the token
                                  arrays (treated as empty: the read state goes to the write slot) */
    LAR_DEVERR_TIMEOUT = 16    /* chunked prefill: a bounded wait for the tensor cores gave up; that
                                  (sequence, head) skipped the rest of its span and its writeback */
};

/*
 * Gated delta rule, scalar decay (GDN).  Interface of flashinfer's
 * `gated_delta_rule_mtp` (initial_state = pool, initial_state_indices =
 * read_idx, output_state_indices = write_idx, cache_intermediate_states =
 * inter), recurrence from the aiter review.
 *   g       [B, T, HV] (rank 2 [B, HV] when T = 1): log-decay, or the raw gate
 *           input when LAR_GATE_RAW; fp32 or bf16, any strides.
 *   beta    [B, T, HV] (rank 2 when T = 1): fp32 or bf16; a logit when LAR_BETA_RAW.
 *   A_log   fp32 [HV]; required with LAR_GATE_RAW, must be NULL without it.
 *   dt_bias fp32 [HV]; optional with LAR_GATE_RAW (zero), must be NULL without it.
 */
lar_status gdn_decode(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                      const lar_tensor* g, const lar_tensor* beta,
                      const lar_tensor* A_log, const lar_tensor* dt_bias,
                      const lar_tensor* pool,
                      const lar_tensor* read_idx, const lar_tensor* write_idx,
                      const lar_tensor* out, const lar_tensor* inter,
                      float scale, uint32_t flags, int32_t* dev_err, void* stream);

/*
 * Gated delta rule, per-key-channel decay (KDA, "Kimi Delta Attention" in the
 * aiter review; its wrapper consumes A_log, dt_bias and use_gate_in_kernel).
 * Same as gdn_decode except:
 *   g       [B, T, HV, K] (rank 3 [B, HV, K] when T = 1)
 *   dt_bias fp32 [HV * K], channel k of head hv at hv * K + k
 */
lar_status kda_decode(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                      const lar_tensor* g, const lar_tensor* beta,
                      const lar_tensor* A_log, const lar_tensor* dt_bias,
                      const lar_tensor* pool,
                      const lar_tensor* read_idx, const lar_tensor* write_idx,
                      const lar_tensor* out, const lar_tensor* inter,
                      float scale, uint32_t flags, int32_t* dev_err, void* stream);

/*
 * Lightning-Attention decode (cuLA PR #75): S <- lambda_h S + k (x) v, o = S^T q.
 * HV == H here: q, k [B, T, H, K], v and out [B, T, H, V] (rank 3 for T = 1).
 *   decay  fp32 [H]: lambda_h.
 *   pool   rank 3 [P*H, V, K] (the page's layout; the state of entry b, head h
 *          is row read_idx[b] * H + h), or rank 4 [P, H, V, K] whose slot
 *          stride equals H times its head stride.  The first dimension of a
 *          rank-3 pool must be a multiple of H.
 */
lar_status la_decode(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                     const lar_tensor* decay, const lar_tensor* pool,
                     const lar_tensor* read_idx, const lar_tensor* write_idx,
                     const lar_tensor* out, const lar_tensor* inter,
                     float scale, int32_t* dev_err, void* stream);

/*
 * Multi-token decode with per-token pool slots (speculative / MTP verify).
 * The aiter KDA review describes these paged per-token state slots and the
 * seed chosen by the number of accepted draft tokens, and lists the two ways
 * such a wrapper went wrong (a flat index table read with the wrong row
 * stride; an accepted count of 0 reading before its row); both are closed here.
 *
 *   state_idx     int32/int64 [B, T] (rank 2 only): the state after token t of
 *                 entry b is written to pool slot state_idx[b][t]; a negative
 *                 slot skips that store.  There is no other writeback.
 *   num_accepted  int32/int64 [B] or NULL: the seed state of entry b is read
 *                 from slot state_idx[b][num_accepted[b] - 1] (the state after
 *                 the last accepted token of the previous step, which stored
 *                 its token states in the same row).  A count outside [1, T]
 *                 starts that entry from a zero state and sets
 *                 LAR_DEVERR_ACCEPTED.
 *   read_idx      [B] or NULL: the seed slot when num_accepted is NULL.
 *                 Exactly one of read_idx and num_accepted must be given.
 * All other arguments as gdn_decode / kda_decode (no write_idx, no inter).
 * The seed of an entry may be one of its own per-token slots (each state row
 * is read before it is overwritten); across entries the aliasing rules of
 * gdn_decode apply.
 */
lar_status gdn_decode_tokens(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta,
                             const lar_tensor* A_log, const lar_tensor* dt_bias,
                             const lar_tensor* pool, const lar_tensor* read_idx,
                             const lar_tensor* num_accepted, const lar_tensor* state_idx,
                             const lar_tensor* out, float scale, uint32_t flags,
                             int32_t* dev_err, void* stream);

lar_status kda_decode_tokens(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta,
                             const lar_tensor* A_log, const lar_tensor* dt_bias,
                             const lar_tensor* pool, const lar_tensor* read_idx,
                             const lar_tensor* num_accepted, const lar_tensor* state_idx,
                             const lar_tensor* out, float scale, uint32_t flags,
                             int32_t* dev_err, void* stream);

/*
 * Variable-length spans (the "varlen" mode of the aiter KDA decode path): N
 * sequences whose tokens are packed token-major, sequence n owning tokens
 * cu_seqlens[n] .. cu_seqlens[n+1] - 1 (any length, 0 included; long spans are
 * a fused-recurrent prefill that leaves its final state in the pool).  Each
 * sequence starts from slot read_idx[n] (negative: zero state), runs the same
 * recurrence token by token, writes o for each of its tokens and its final
 * state to write_idx[n] (negative: skipped; an empty span copies the read
 * state there).  Tokens outside every span are not written.
 *   q, k        [Ntok, H, K];  v, out  [Ntok, HV, V];  any strides, fp32 or bf16
 *   g, beta     [Ntok, HV] (KDA g: [Ntok, HV, K])
 *   cu_seqlens  [N + 1], int32 or int64, non-decreasing from 0 to at most Ntok
 *               (a span that is reversed or runs past Ntok is treated as empty
 *               and sets LAR_DEVERR_SEQLEN in *dev_err; spans that overlap,
 *               which non-decreasing offsets rule out, write the shared output
 *               rows in an unspecified order)
 *   read_idx, write_idx  [N] (write_idx NULL: the read slot)
 *   inter       NULL, or [Ntok, HV, V, K] fp32 or bf16: the state after each token
 *   pool        as for gdn_decode, [v][k] layout only (LAR_STATE_KV is rejected)
 * Flags, A_log, dt_bias and decay as for the fixed-T calls.  N <= 65535,
 * Ntok < 2^31.
 * Without a state cache (inter NULL) and at K = V = 128, spans of 16 tokens or
 * more are computed in the chunked form of gdn_prefill / kda_prefill /
 * la_prefill below (equal to the recurrence up to rounding, and several times
 * cheaper per token on such spans) and the shorter ones token by token: two
 * kernels on `stream`, each choosing its spans on the device from cu_seqlens.
 * The chunked kernel's grid has a row per possible long span (at most
 * Ntok / 16 when the valid spans are disjoint) and is not launched when Ntok <
 * 16; if any span is reversed (then valid spans may overlap) every span runs
 * token by token.  With a state cache every span runs token by token.
 */
lar_status gdn_decode_varlen(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta,
                             const lar_tensor* A_log, const lar_tensor* dt_bias,
                             const lar_tensor* pool, const lar_tensor* cu_seqlens,
                             const lar_tensor* read_idx, const lar_tensor* write_idx,
                             const lar_tensor* out, const lar_tensor* inter,
                             float scale, uint32_t flags, int32_t* dev_err, void* stream);

lar_status kda_decode_varlen(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                             const lar_tensor* g, const lar_tensor* beta,
                             const lar_tensor* A_log, const lar_tensor* dt_bias,
                             const lar_tensor* pool, const lar_tensor* cu_seqlens,
                             const lar_tensor* read_idx, const lar_tensor* write_idx,
                             const lar_tensor* out, const lar_tensor* inter,
                             float scale, uint32_t flags, int32_t* dev_err, void* stream);

lar_status la_decode_varlen(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                            const lar_tensor* decay, const lar_tensor* pool,
                            const lar_tensor* cu_seqlens, const lar_tensor* read_idx,
                            const lar_tensor* write_idx, const lar_tensor* out,
                            const lar_tensor* inter, float scale, int32_t* dev_err, void* stream);

/*
 * Chunked prefill over variable-length spans (the form of the recurrence for
 * long spans): the same operation and arguments as gdn_decode_varlen /
 * la_decode_varlen, computed 32 tokens at a time with the recurrence unrolled
 * over each chunk into matrix products and a unit lower-triangular solve (the
 * per-token recurrence of the aiter KDA review, rearranged; equal up to
 * rounding).  Every output row of a token inside a span and every written state
 * is produced; there is no per-token state cache (the chunked form never forms
 * the intermediate states).
 *   K = V = 128 only (other shapes: LAR_ERR_SHAPE; use *_decode_varlen).
 * One CTA per (sequence, v-head) pair keeps the state on chip (registers and
 * tensor memory) for the whole span and runs the chunk's products on the
 * tensor cores; the work of a sequence is spread over its heads, so a span
 * shorter than a chunk costs a whole chunk (the *_decode_varlen calls send
 * such spans token by token).
 *
 * kda_prefill: KDA's per-key-channel decay moves into the chunk's dot
 * products: with P[t][s][c] = exp(g_{s+1}[c]) ... exp(g_t[c]) (products of the
 * per-token factors, never exponentials of differences),
 *     A[t][s] = beta_t sum_c k_t[c] k_s[c] P[t][s][c]  (s < t),
 *     o_t = sum_c q_t[c] E_t[c] (S0 column) + sum_{s<=t} (sum_c q_t[c] k_s[c] P[t][s][c]) d_s,
 *     S   = diag(E_last) S0 + sum_s (P[last][s] o k_s) d_s^T,
 * E_t[c] = exp(g_0[c]) ... exp(g_t[c]); arguments as kda_decode_varlen
 * (g [Ntok, HV, K], dt_bias [HV * K]) without the state cache.
 */
lar_status gdn_prefill(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                       const lar_tensor* g, const lar_tensor* beta,
                       const lar_tensor* A_log, const lar_tensor* dt_bias,
                       const lar_tensor* pool, const lar_tensor* cu_seqlens,
                       const lar_tensor* read_idx, const lar_tensor* write_idx,
                       const lar_tensor* out, float scale, uint32_t flags, int32_t* dev_err,
                       void* stream);

lar_status kda_prefill(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                       const lar_tensor* g, const lar_tensor* beta,
                       const lar_tensor* A_log, const lar_tensor* dt_bias,
                       const lar_tensor* pool, const lar_tensor* cu_seqlens,
                       const lar_tensor* read_idx, const lar_tensor* write_idx,
                       const lar_tensor* out, float scale, uint32_t flags, int32_t* dev_err,
                       void* stream);

lar_status la_prefill(const lar_tensor* q, const lar_tensor* k, const lar_tensor* v,
                      const lar_tensor* decay, const lar_tensor* pool,
                      const lar_tensor* cu_seqlens, const lar_tensor* read_idx,
                      const lar_tensor* write_idx, const lar_tensor* out, float scale,
                      int32_t* dev_err, void* stream);

/* Static, human-readable name of a status code. */
const char* lar_status_string(lar_status status);

#ifdef __cplusplus
}
#endif

#endif /* LAR_H_ */
