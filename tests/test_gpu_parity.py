"""GPU parity: the sm_103a kernels through the C ABI against the fp64 oracle,
plus GPU-vs-GPU invariants that must hold bit for bit.

Replicated test plans from the pages:
  * cuLA PR #75 pool tests: identity / non-identity (pool 6, offsets
    [2,0,5,1]) / reversed offsets, writeback (active slots updated, inactive
    untouched), big batch (B=33, pool 40).
  * flashinfer fp32 MTP pool tests: B in {1,4,16} x T in {2,4} x separate
    write slots x intermediate caching; strided pools B in {1,4} x T in {2,4} x
    stride_multiplier in {2,3}.
  * flashinfer packed-QKV regression: q/k/v as head-dim slices of a fused
    buffer give bit-identical results to contiguous copies.
Tolerances are in tests/_parity.py.
"""
import zlib

import pytest
import torch

import _parity as P
import workloads as W

pytestmark = pytest.mark.gpu
F32 = torch.float32

SWEEP = {
    "gdn_gqa_t1": ("gdn", dict(B=4, T=1, H=2, HV=4, K=128, V=128)),
    "gdn_ragged_sep_skip": ("gdn", dict(B=3, T=3, H=1, HV=2, K=64, V=40, separate_write=True,
                                         skip_frac=0.34, cache_intermediate=True)),
    "gdn_f32_stride3_i64": ("gdn", dict(B=5, T=2, H=2, HV=2, K=32, V=70, in_dtype=F32,
                                         out_dtype=F32, stride_mult=3, index_dtype=torch.int64)),
    "gdn_k16_t8_raw": ("gdn", dict(B=2, T=8, H=2, HV=6, K=16, V=16, raw_gates=True,
                                    cache_intermediate=True)),
    "gdn_big_batch": ("gdn", dict(B=33, T=1, H=2, HV=2, K=128, V=128, P=40)),
    "gdn_t16": ("gdn", dict(B=2, T=16, H=1, HV=1, K=128, V=64, cache_intermediate=True)),
    "kda_raw_t1": ("kda", dict(B=4, T=1, H=2, HV=2, K=128, V=128, raw_gates=True)),
    "kda_mtp_strided": ("kda", dict(B=3, T=4, H=1, HV=3, K=64, V=100, separate_write=True,
                                    skip_frac=0.34, cache_intermediate=True, stride_mult=2)),
    "kda_packed_raw": ("kda", dict(B=2, T=2, H=2, HV=2, K=128, V=96, packed=True, raw_gates=True)),
    "kda_f32_k32": ("kda", dict(B=6, T=1, H=4, HV=4, K=32, V=33, in_dtype=F32, out_dtype=F32)),
    "la_packed_flat": ("la", dict(B=4, T=1, H=3, K=128, V=128, packed=True, flat_pool=True)),
    "la_mtp_sep_skip": ("la", dict(B=3, T=4, H=2, K=64, V=50, cache_intermediate=True,
                                   separate_write=True, skip_frac=0.34)),
    "la_f32_k16": ("la", dict(B=2, T=2, H=2, K=16, V=24, in_dtype=F32, out_dtype=F32,
                              flat_pool=True)),
    # T * V > 4096: v is read from global memory in the token loop instead of staged
    "gdn_unstaged_v": ("gdn", dict(B=2, T=16, H=1, HV=2, K=64, V=300, cache_intermediate=True)),
    "kda_unstaged_v": ("kda", dict(B=2, T=9, H=1, HV=1, K=128, V=520, raw_gates=True)),
    "la_unstaged_v": ("la", dict(B=2, T=11, H=2, K=32, V=400, separate_write=True)),
    "kda_t16_gqa": ("kda", dict(B=3, T=16, H=2, HV=4, K=128, V=64, raw_gates=True,
                                cache_intermediate=True)),
    # bfloat16 state pool (fp32 arithmetic, state rounded once per store)
    "gdn_bf16_t1": ("gdn", dict(B=5, T=1, H=2, HV=4, K=128, V=128, state_dtype=torch.bfloat16)),
    "gdn_bf16_mtp_strided": ("gdn", dict(B=4, T=4, H=2, HV=4, K=128, V=96, state_dtype=torch.bfloat16,
                                         stride_mult=2, separate_write=True, skip_frac=0.25,
                                         cache_intermediate=True)),
    "gdn_bf16_pool_f32_cache": ("gdn", dict(B=3, T=3, H=1, HV=2, K=64, V=70, state_dtype=torch.bfloat16,
                                            cache_intermediate=True, inter_dtype=torch.float32)),
    "gdn_f32_pool_bf16_cache": ("gdn", dict(B=3, T=3, H=1, HV=2, K=64, V=70, cache_intermediate=True,
                                            inter_dtype=torch.bfloat16)),
    "kda_bf16_raw": ("kda", dict(B=4, T=2, H=2, HV=2, K=128, V=128, raw_gates=True,
                                 state_dtype=torch.bfloat16, cache_intermediate=True)),
    "kda_bf16_k32": ("kda", dict(B=3, T=1, H=2, HV=2, K=32, V=33, state_dtype=torch.bfloat16)),
    # single-token K = 128 instances with ragged V, skipped and separate writes
    "gdn_t1_ragged_skip": ("gdn", dict(B=5, T=1, H=2, HV=4, K=128, V=100, separate_write=True,
                                       skip_frac=0.3)),
    "kda_bf16_t1_ragged": ("kda", dict(B=4, T=1, H=2, HV=2, K=128, V=72, raw_gates=True,
                                       state_dtype=torch.bfloat16, separate_write=True, skip_frac=0.3)),
    "gdn_bf16_t1_ragged": ("gdn", dict(B=4, T=1, H=1, HV=3, K=128, V=100, state_dtype=torch.bfloat16,
                                       stride_mult=2)),
    "la_k128_t2_cache": ("la", dict(B=3, T=2, H=2, K=128, V=96, cache_intermediate=True,
                                    separate_write=True, skip_frac=0.34)),
    # multi-token GDN without a cache, raw gates, odd token counts
    "gdn_t6_nocache": ("gdn", dict(B=3, T=6, H=2, HV=4, K=128, V=96, separate_write=True, skip_frac=0.34)),
    "gdn_t16_nocache_raw": ("gdn", dict(B=2, T=16, H=1, HV=2, K=64, V=64, raw_gates=True)),
    "gdn_bf16_t5_nocache": ("gdn", dict(B=3, T=5, H=1, HV=3, K=128, V=128, state_dtype=torch.bfloat16)),
    "gdn_t7_cache_k32": ("gdn", dict(B=2, T=7, H=2, HV=2, K=32, V=40, cache_intermediate=True,
                                     in_dtype=F32, out_dtype=F32)),
    # single-token calls with a state cache (served by the general instances)
    "gdn_t1_cache": ("gdn", dict(B=4, T=1, H=2, HV=4, K=128, V=128, cache_intermediate=True)),
    "gdn_kv_t1_cache_bf16": ("gdn", dict(B=3, T=1, H=1, HV=2, K=128, V=96, state_kv=True,
                                         state_dtype=torch.bfloat16, cache_intermediate=True)),
    "kda_t1_cache_bf16_pool": ("kda", dict(B=3, T=1, H=2, HV=2, K=128, V=64, raw_gates=True,
                                           state_dtype=torch.bfloat16, cache_intermediate=True,
                                           inter_dtype=F32)),
    # more tiles than resident CTAs: every CTA streams several tiles across pair boundaries
    "gdn_split_tiles": ("gdn", dict(B=48, T=1, H=2, HV=4, K=128, V=100, separate_write=True,
                                    skip_frac=0.25)),
    "gdn_bf16_split_tiles": ("gdn", dict(B=48, T=1, H=2, HV=4, K=128, V=128, P=60,
                                         state_dtype=torch.bfloat16)),
    "gdn_split_mtp_cache": ("gdn", dict(B=40, T=4, H=2, HV=4, K=128, V=112, cache_intermediate=True,
                                        separate_write=True, skip_frac=0.25, stride_mult=2)),
    "kda_split_tiles": ("kda", dict(B=40, T=2, H=4, HV=4, K=128, V=128, raw_gates=True)),
    "la_split_tiles": ("la", dict(B=64, T=1, H=4, K=128, V=128, flat_pool=True)),
    "la_bf16_packed": ("la", dict(B=4, T=1, H=3, K=128, V=128, packed=True, flat_pool=True,
                                  state_dtype=torch.bfloat16)),
    "la_bf16_k16": ("la", dict(B=2, T=2, H=2, K=16, V=24, flat_pool=True, state_dtype=torch.bfloat16)),
    "gdn_bf16_unstaged_v": ("gdn", dict(B=2, T=16, H=1, HV=1, K=64, V=300, state_dtype=torch.bfloat16)),
    # [k][v] ("nontranspose") state layout
    "gdn_kv_t1": ("gdn", dict(B=5, T=1, H=2, HV=4, K=128, V=128, state_kv=True)),
    "gdn_kv_mtp_strided": ("gdn", dict(B=4, T=4, H=2, HV=4, K=128, V=96, state_kv=True, stride_mult=2,
                                       separate_write=True, skip_frac=0.25, cache_intermediate=True)),
    "gdn_kv_ragged_k64": ("gdn", dict(B=3, T=3, H=1, HV=2, K=64, V=72, state_kv=True,
                                      cache_intermediate=True)),
    "gdn_kv_k16": ("gdn", dict(B=2, T=2, H=2, HV=2, K=16, V=16, state_kv=True)),
    "gdn_kv_k32_f32": ("gdn", dict(B=3, T=1, H=1, HV=3, K=32, V=40, state_kv=True, in_dtype=F32,
                                   out_dtype=F32)),
    "kda_kv_raw": ("kda", dict(B=4, T=2, H=2, HV=2, K=128, V=128, raw_gates=True, state_kv=True,
                               cache_intermediate=True)),
    "gdn_kv_bf16": ("gdn", dict(B=4, T=2, H=2, HV=4, K=128, V=128, state_kv=True,
                                state_dtype=torch.bfloat16, cache_intermediate=True)),
    "gdn_kv_bf16_t1_ragged": ("gdn", dict(B=5, T=1, H=2, HV=4, K=128, V=96, state_kv=True,
                                          state_dtype=torch.bfloat16, separate_write=True, skip_frac=0.2)),
    "kda_kv_bf16_t1": ("kda", dict(B=3, T=1, H=2, HV=2, K=128, V=128, state_kv=True, raw_gates=True,
                                   state_dtype=torch.bfloat16)),
    "kda_kv_bf16_k16": ("kda", dict(B=3, T=1, H=1, HV=2, K=16, V=24, state_kv=True,
                                    state_dtype=torch.bfloat16)),
    "gdn_kv_unstaged_v": ("gdn", dict(B=2, T=16, H=1, HV=1, K=64, V=320, state_kv=True)),
}


def test_gdn_tiny_config(cuda_device):
    P.full_check(W.make("gdn_tiny"), cuda_device)


@pytest.mark.parametrize("name", list(SWEEP))
def test_sweep(name, cuda_device):
    form, kw = SWEEP[name]
    P.full_check(W.make_custom(form, seed=zlib.crc32(name.encode()) % 1000, **kw), cuda_device)


def test_scale_argument(cuda_device):
    w = W.make_custom("gdn", B=2, T=2, H=2, HV=2, K=128, V=64, seed=3)
    w.scale = 128 ** -0.5
    P.full_check(w, cuda_device)


# ---------------------------------------------------------------- cuLA PR #75 pool tests

def _la_states(n, H, V, K, seed):
    return torch.randn(n, H, V, K, generator=torch.Generator().manual_seed(seed)) * 0.1


@pytest.mark.parametrize("slots,pool_size", [([0, 1, 2, 3], 4), ([2, 0, 5, 1], 6), ([3, 2, 1, 0], 4)])
def test_la_pool_offsets(slots, pool_size, cuda_device):
    """Same sequences placed at different pool slots give bit-identical outputs
    and states; inactive slots are untouched."""
    B, H, K, V = 4, 2, 128, 64
    w = W.make_custom("la", B=B, T=1, H=H, K=K, V=V, P=pool_size, flat_pool=True, seed=5)
    states = _la_states(B, H, V, K, 6)

    def place(sl, P_):
        pool = torch.full((P_ * H, V, K), -7.0)
        for i, s in enumerate(sl):
            pool[s * H:(s + 1) * H] = states[i]
        return pool

    ident = place([0, 1, 2, 3], 4).to(cuda_device)
    out_ref = P.run_gpu(w, cuda_device, pool=ident, read_idx=torch.arange(4), write_idx=None)[0]
    pool = place(slots, pool_size).to(cuda_device)
    before = pool.clone()
    ri = torch.tensor(slots, dtype=torch.int32)
    out = P.run_gpu(w, cuda_device, pool=pool, read_idx=ri, write_idx=None)[0]
    torch.cuda.synchronize()
    assert torch.equal(out, out_ref)
    for i, s in enumerate(slots):
        assert torch.equal(pool[s * H:(s + 1) * H], ident[i * H:(i + 1) * H])
    inactive = [s for s in range(pool_size) if s not in slots]
    for s in inactive:
        assert torch.equal(pool[s * H:(s + 1) * H], before[s * H:(s + 1) * H])
    # and against the oracle
    host = place(slots, pool_size)
    ref = P.run_oracle(w, host, read_idx=ri, write_idx=None)
    P.assert_out_close(out, ref["out"])
    P.assert_state_close(pool.cpu(), host.double().numpy(), "pool")


def test_la_big_batch(cuda_device):
    w = W.make_custom("la", B=33, T=1, H=2, K=128, V=128, P=40, flat_pool=True, seed=7)
    P.full_check(w, cuda_device)


# ---------------------------------------------------------------- flashinfer fp32 MTP pool tests

@pytest.mark.parametrize("B", [1, 4, 16])
@pytest.mark.parametrize("T", [2, 4])
@pytest.mark.parametrize("separate", [False, True])
@pytest.mark.parametrize("cache", [False, True])
def test_mtp_fp32_state_pool(B, T, separate, cache, cuda_device):
    w = W.make_custom("gdn", B=B, T=T, H=4, HV=8, K=128, V=128, P=2 * B + 2,
                      separate_write=separate, cache_intermediate=cache, seed=B * 10 + T)
    P.full_check(w, cuda_device)


@pytest.mark.parametrize("B", [1, 4])
@pytest.mark.parametrize("T", [2, 4])
@pytest.mark.parametrize("mult", [2, 3])
def test_mtp_fp32_state_pool_non_contiguous(B, T, mult, cuda_device):
    w = W.make_custom("gdn", B=B, T=T, H=4, HV=8, K=128, V=128, P=2 * B + 2, stride_mult=mult,
                      separate_write=True, cache_intermediate=True, seed=B + T + mult)
    assert not w.pool.is_contiguous()
    P.full_check(w, cuda_device)


# ---------------------------------------------------------------- packed QKV regression

@pytest.mark.parametrize("form", ["gdn", "kda", "la"])
@pytest.mark.parametrize("T", [1, 3])
def test_packed_equals_contiguous(form, T, cuda_device):
    kw = dict(flat_pool=True) if form == "la" else dict(raw_gates=form == "kda")
    w = W.make_custom(form, B=5, T=T, H=3, HV=3, K=128, V=128, packed=True, seed=T, **kw)
    q, k, v = P.qkv_dev(w, cuda_device)    # slices of one fused device buffer (asserted)
    qc, kc, vc = (x.contiguous() for x in (q, k, v))
    assert qc.is_contiguous() and qc.data_ptr() != q.data_ptr()
    pa, pb = w.pool.to(cuda_device), w.pool.to(cuda_device)
    oa = P.run_gpu(w, cuda_device, pool=pa, q=q, k=k, v=v)[0]
    ob = P.run_gpu(w, cuda_device, pool=pb, q=qc, k=kc, v=vc)[0]
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    assert torch.equal(pa, pb)


def test_any_input_strides(cuda_device):
    """q/k/v/g/beta read through arbitrary strides (here every other element and
    a transposed batch/head order) give bit-identical results."""
    w = W.make_custom("gdn", B=3, T=2, H=2, HV=4, K=64, V=64, seed=12)
    dev = cuda_device

    def spread(t):
        big = torch.zeros(*t.shape[:-1], 2 * t.shape[-1], dtype=t.dtype)
        big[..., ::2] = t
        return big.to(dev)[..., ::2]

    pa, pb = w.pool.to(dev), w.pool.to(dev)
    oa = P.run_gpu(w, dev, pool=pa)[0]
    ob = P.run_gpu(w, dev, pool=pb, q=spread(w.q), k=spread(w.k),
                   v=w.v.transpose(0, 2).contiguous().transpose(0, 2).to(dev))[0]
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and torch.equal(pa, pb)


# ---------------------------------------------------------------- GPU-vs-GPU invariants

@pytest.mark.parametrize("form", ["gdn", "kda", "la"])
def test_multi_token_equals_chained_launches(form, cuda_device):
    """A T-token launch equals T one-token launches chained through the pool
    (the state is fp32 in registers and in the pool alike: bit-exact)."""
    kw = dict(flat_pool=True) if form == "la" else dict(raw_gates=form == "kda")
    w = W.make_custom(form, B=4, T=4, H=2, HV=2, K=128, V=96, cache_intermediate=True, seed=21, **kw)
    dev = cuda_device
    pa, pb = w.pool.to(dev), w.pool.to(dev)
    out_multi, inter = P.run_gpu(w, dev, pool=pa)
    outs = []
    for t in range(w.T):
        sub = W.make_custom(form, B=4, T=4, H=2, HV=2, K=128, V=96, seed=21, **kw)
        for name in ("q", "k", "v", "g", "beta"):
            x = getattr(w, name)
            if x is not None:
                setattr(sub, name, x[:, t:t + 1])
        sub.T = 1
        sub.cache_intermediate = False
        outs.append(P.run_gpu(sub, dev, pool=pb)[0])
        torch.cuda.synchronize()
        for b, s in enumerate(w.write_idx.tolist()):
            assert torch.equal(inter[b, t], P.slot_state(pb, w, s))
    assert torch.equal(out_multi, torch.cat(outs, dim=1))
    assert torch.equal(pa, pb)


def test_batch_permutation(cuda_device):
    w = W.make_custom("kda", B=8, T=2, H=2, HV=4, K=128, V=64, raw_gates=True, seed=4)
    dev = cuda_device
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(1))
    pa, pb = w.pool.to(dev), w.pool.to(dev)
    oa = P.run_gpu(w, dev, pool=pa)[0]
    for name in ("q", "k", "v", "g", "beta", "read_idx", "write_idx"):
        setattr(w, name, getattr(w, name)[perm])
    ob = P.run_gpu(w, dev, pool=pb)[0]
    torch.cuda.synchronize()
    assert torch.equal(oa[perm], ob)
    assert torch.equal(pa, pb)


def test_index_dtypes_agree(cuda_device):
    w = W.make_custom("gdn", B=4, T=1, H=2, HV=2, K=128, V=128, seed=8)
    dev = cuda_device
    pa, pb = w.pool.to(dev), w.pool.to(dev)
    oa = P.run_gpu(w, dev, pool=pa, read_idx=w.read_idx.int(), write_idx=w.write_idx.int())[0]
    ob = P.run_gpu(w, dev, pool=pb, read_idx=w.read_idx.long(), write_idx=w.write_idx.long())[0]
    torch.cuda.synchronize()
    assert torch.equal(oa, ob) and torch.equal(pa, pb)


@pytest.mark.parametrize("form,T,state_dtype", [("gdn", 2, F32), ("gdn", 1, F32), ("gdn", 1, torch.bfloat16),
                                                ("kda", 1, F32), ("kda", 1, torch.bfloat16)])
def test_negative_and_out_of_range_slots(form, T, state_dtype, cuda_device):
    """read -1: zero initial state; write -1: no writeback; slots >= P: the
    same, plus the device error bits; every other byte untouched."""
    w = W.make_custom(form, B=4, T=T, H=1, HV=2, K=128, V=64, P=6, seed=9, raw_gates=form == "kda",
                      state_dtype=state_dtype)
    dev = cuda_device
    ri = torch.tensor([-1, 2, 6, 4], dtype=torch.int32)
    wi = torch.tensor([0, -1, 1, 9], dtype=torch.int32)
    pool = w.pool.to(dev)
    before = pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = P.run_gpu(w, dev, pool=pool, read_idx=ri, write_idx=wi, dev_err=err)[0]
    torch.cuda.synchronize()
    assert int(err.item()) == 3                     # LAR_DEVERR_READ_SLOT | LAR_DEVERR_WRITE_SLOT
    host = w.pool.clone()
    ref = P.run_oracle(w, host, read_idx=ri, write_idx=wi)
    assert ref["n_bad"] == 2
    P.assert_out_close(out, ref["out"])
    for s in (2, 3, 4, 5):                          # only slots 0 and 1 are written
        assert torch.equal(pool[s], before[s])
    P.assert_state_close(pool[0], ref["final_state"][0])
    P.assert_state_close(pool[1], ref["final_state"][2])
    P.assert_state_close(pool.cpu(), host.double().numpy(), "pool")


def test_empty_batch_changes_nothing(cuda_device):
    w = W.make_custom("gdn", B=2, T=1, H=1, HV=1, K=128, V=32, seed=2)
    dev = cuda_device
    pool = w.pool.to(dev)
    before = pool.clone()
    for name in ("q", "k", "v", "g", "beta", "read_idx", "write_idx"):
        setattr(w, name, getattr(w, name)[:0])
    w.B = 0
    out = P.run_gpu(w, dev, pool=pool)[0]
    torch.cuda.synchronize()
    assert out.shape[0] == 0 and torch.equal(pool, before)


# ---------------------------------------------------------------- per-token pool slots

def _token_case(form, B, T, seed, state_dtype=F32, HV=4, H=2):
    w = W.make_custom(form, B=B, T=T, H=H, HV=HV, K=128, V=96, P=B * T + B + 3, seed=seed,
                      raw_gates=form == "kda", state_dtype=state_dtype)
    g = torch.Generator().manual_seed(seed + 1)
    perm = torch.randperm(w.P, generator=g)
    table = perm[:B * T].view(B, T).clone()
    seeds = perm[B * T:B * T + B].clone()
    table[0, -1] = -1                                    # a skipped token store
    return w, table, seeds


@pytest.mark.parametrize("form", ["gdn", "kda"])
@pytest.mark.parametrize("state_dtype", [F32, torch.bfloat16])
@pytest.mark.parametrize("use_accepted", [False, True])
def test_token_slots_against_oracle(form, state_dtype, use_accepted, cuda_device):
    import linear_attention_recurrent_gb300 as lar
    import oracle
    dev = cuda_device
    B, T = 5, 4
    w, table, seeds = _token_case(form, B, T, seed=30 + T, state_dtype=state_dtype)
    host = w.pool.clone()
    pool = w.pool.to(dev)
    before = pool.clone()
    kw = dict(A_log=w.A_log, dt_bias=w.dt_bias, qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw,
              beta_raw=w.beta_raw)
    if use_accepted:
        acc = torch.tensor([1, 4, 2, 3, 4])
        acc_seed = {"num_accepted": acc}
        # the seeds live in the table row: make them valid states first (they are: pool slots)
    else:
        acc_seed = {"read_idx": seeds}
    ofn = oracle.kda_decode_tokens if form == "kda" else oracle.gdn_decode_tokens
    gfn = lar.kda_decode_tokens if form == "kda" else lar.gdn_decode_tokens
    ref = ofn(w.q, w.k, w.v, w.g, w.beta, host, table, cache_intermediate=True, **acc_seed, **kw)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cu = {n: (t.to(dev) if isinstance(t, torch.Tensor) else t) for n, t in kw.items()}
    cu_seed = {n: t.to(dev) for n, t in acc_seed.items()}
    out = gfn(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), pool, table.to(dev),
              out_dtype=w.out_dtype, dev_err=err, **cu_seed, **cu)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and ref["n_bad"] == 0
    P.assert_out_close(out, ref["out"])
    # each written slot holds the state after its token (fp64 reference, before any rounding)
    written = {}
    for b in range(B):
        for t in range(T):
            if int(table[b, t]) >= 0:
                written[int(table[b, t])] = (b, t)
    for s in range(w.P):
        if s in written:
            b, t = written[s]
            P.assert_state_close(pool[s], ref["inter"][b, t], f"slot {s} (entry {b}, token {t})")
        else:
            assert torch.equal(pool[s], before[s]), f"slot {s} changed"


def test_token_slots_bad_accepted_count(cuda_device):
    import linear_attention_recurrent_gb300 as lar
    import oracle
    dev = cuda_device
    w, table, _ = _token_case("gdn", 3, 4, seed=50)
    host = w.pool.clone()
    pool = w.pool.to(dev)
    acc = torch.tensor([0, 5, 2])
    ref = oracle.gdn_decode_tokens(w.q, w.k, w.v, w.g, w.beta, host, table, num_accepted=acc)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = lar.gdn_decode_tokens(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), pool,
                                table.to(dev), num_accepted=acc.to(dev), out_dtype=w.out_dtype, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4 and ref["n_bad"] == 2   # LAR_DEVERR_ACCEPTED
    P.assert_out_close(out, ref["out"])
    P.assert_state_close(pool.cpu(), host.double().numpy(), "pool")


def test_token_slots_two_step_speculative_flow(cuda_device):
    """Step 1 stores every token's state in the row; step 2 seeds from the
    accepted count; both on the GPU and in the oracle, pools compared at the end."""
    import linear_attention_recurrent_gb300 as lar
    import oracle
    dev = cuda_device
    w1, table, seeds = _token_case("gdn", 4, 4, seed=60)
    w2, _, _ = _token_case("gdn", 4, 4, seed=61)
    host = w1.pool.clone()
    pool = w1.pool.to(dev)
    oracle.gdn_decode_tokens(w1.q, w1.k, w1.v, w1.g, w1.beta, host, table, read_idx=seeds)
    lar.gdn_decode_tokens(w1.q.to(dev), w1.k.to(dev), w1.v.to(dev), w1.g.to(dev), w1.beta.to(dev), pool,
                          table.to(dev), read_idx=seeds.to(dev), out_dtype=w1.out_dtype)
    acc = torch.tensor([3, 1, 4, 2])
    table2 = table.clone()                               # the same slot row serves every step
    ref = oracle.gdn_decode_tokens(w2.q, w2.k, w2.v, w2.g, w2.beta, host, table2, num_accepted=acc)
    out = lar.gdn_decode_tokens(w2.q.to(dev), w2.k.to(dev), w2.v.to(dev), w2.g.to(dev), w2.beta.to(dev), pool,
                                table2.to(dev), num_accepted=acc.to(dev), out_dtype=w2.out_dtype)
    torch.cuda.synchronize()
    P.assert_out_close(out, ref["out"])
    P.assert_state_close(pool.cpu(), host.double().numpy(), "pool")
