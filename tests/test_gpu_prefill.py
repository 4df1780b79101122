"""The chunked prefill calls (gdn_prefill, la_prefill) against the oracle.

The chunked form rearranges the per-token recurrence over 32-token chunks
(matrix products plus a unit lower-triangular solve), so it equals the
recurrence up to rounding; it is compared with the same fp64 oracle and the
same tolerances as the token-by-token calls: outputs of every token inside a
span, written states, untouched pool bytes, rows of tokens outside every span
left as allocated.  Span lengths straddle the chunk size (31, 32, 33, 64, 65)
and run to several chunks; empty and bad spans, bf16 pools, in-kernel gates,
separate and skipped write slots, packed, fp32 and unaligned inputs are
covered.
"""
import pytest
import torch

import _parity as P
import workloads as W
import linear_attention_recurrent_gb300 as lar

pytestmark = pytest.mark.gpu
F32, BF16 = torch.float32, torch.bfloat16

SPANS = [31, 1, 32, 0, 33, 64, 65, 100, 257]

CASES = {
    "gdn": dict(form="gdn", lengths=SPANS, H=2, HV=4),
    "gdn_raw_gates": dict(form="gdn", lengths=SPANS, H=1, HV=2, raw_gates=True),
    "gdn_bf16_pool": dict(form="gdn", lengths=SPANS, H=2, HV=4, state_dtype=BF16),
    "gdn_separate_skip_fp32_io": dict(form="gdn", lengths=[40, 5, 96, 0, 70, 3], H=2, HV=2, separate_write=True,
                                      skip_frac=0.34, in_dtype=F32, out_dtype=F32),
    "gdn_strided_pool": dict(form="gdn", lengths=[50, 129], H=1, HV=3, stride_mult=2),
    "gdn_int64": dict(form="gdn", lengths=[65, 2, 31], H=1, HV=2, index_dtype=torch.int64),
    "gdn_long": dict(form="gdn", lengths=[1000], H=1, HV=2),
    "la": dict(form="la", lengths=SPANS, H=3),
    "la_flat_bf16": dict(form="la", lengths=[33, 0, 64, 7], H=2, flat_pool=True, state_dtype=BF16),
    "la_packed": dict(form="la", lengths=[45, 90], H=2, packed=True),
    # KDA: per-key-channel decay inside the chunk products (raw gates: in-kernel gate chain,
    # l2 norm and sigmoid, decays down to exp(-16 softplus(.)) per token, whose products underflow)
    "kda_raw_gates": dict(form="kda", lengths=SPANS, H=2, HV=2, raw_gates=True),
    "kda_activated_gqa": dict(form="kda", lengths=SPANS, H=1, HV=3),
    "kda_bf16_pool": dict(form="kda", lengths=SPANS, H=2, HV=2, raw_gates=True, state_dtype=BF16),
    "kda_long": dict(form="kda", lengths=[1000], H=1, HV=2, raw_gates=True),
    "kda_separate_skip_fp32_io": dict(form="kda", lengths=[40, 5, 96, 0, 70, 3], H=2, HV=2, separate_write=True,
                                      skip_frac=0.34, in_dtype=F32, out_dtype=F32, raw_gates=True),
    "kda_packed_strided": dict(form="kda", lengths=[50, 129], H=2, HV=2, packed=True, raw_gates=True, stride_mult=2),
}


def _run_prefill(w, dev, pool, cu_seqlens=None, dev_err=None):
    cu = P.to_dev(w.cu_seqlens if cu_seqlens is None else cu_seqlens, dev)
    out = torch.full(tuple(w.v.shape), float("nan"), dtype=w.out_dtype, device=dev)
    q, k, v = P.qkv_dev(w, dev)
    ri, wi = P.to_dev(w.read_idx, dev), P.to_dev(w.write_idx, dev)
    if w.form == "la":
        lar.la_prefill(q, k, v, P.to_dev(w.decay, dev), pool, cu, ri, wi, out=out, scale=w.scale, dev_err=dev_err)
    else:
        fn = lar.gdn_prefill if w.form == "gdn" else lar.kda_prefill
        fn(q, k, v, P.to_dev(w.g, dev), P.to_dev(w.beta, dev), pool, cu, ri, wi, out=out,
                        A_log=P.to_dev(w.A_log, dev), dt_bias=P.to_dev(w.dt_bias, dev), scale=w.scale,
                        qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw, dev_err=dev_err)
    return out


def prefill_check(w, dev, cu_seqlens=None, expect_err=0):
    st_host = P.storage(w)
    dev_storage = st_host.to(dev)
    before = dev_storage.clone()
    if w.backing is not None:
        mult = w.pool.stride(0) // w.backing.stride(0)
        pool_dev, host_view = dev_storage[::mult], st_host.clone()[::mult]
    else:
        pool_dev, host_view = dev_storage, st_host.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = _run_prefill(w, dev, pool_dev, cu_seqlens, err)
    torch.cuda.synchronize()
    ref = P.run_oracle_varlen(w, host_view, cu_seqlens)
    import numpy as np
    covered = ~np.isnan(ref["out"]).all(axis=(1, 2))
    cov = torch.from_numpy(covered).to(dev)
    if covered.any():
        P.assert_out_close(out[cov], ref["out"][covered])
    if (~covered).any():
        assert torch.isnan(out[~cov].float()).all(), "output rows outside every span written"
    mask = P.written_mask(w).to(dev)
    assert torch.equal(dev_storage[~mask], before[~mask]), "untouched pool bytes changed"
    for n, s in enumerate(w.write_idx.tolist()):
        if 0 <= s < w.P:
            P.assert_state_close(P.slot_state(pool_dev, w, s), ref["final_state"][n], f"slot {s} (sequence {n})")
    assert int(err.item()) == expect_err


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_parity(name, cuda_device):
    kw = dict(CASES[name])
    form, lengths = kw.pop("form"), kw.pop("lengths")
    w = W.make_varlen(form, lengths, K=128, V=128, seed=71, **kw)
    prefill_check(w, cuda_device)


@pytest.mark.parametrize("form", ["gdn", "kda"])
def test_prefill_many_sequences(form, cuda_device):
    """More sequences than the longest-first ranking takes (256): the grid
    keeps the sequences' own order; short and chunk-straddling spans."""
    lengths = [(7 * i) % 41 for i in range(300)]
    w = W.make_varlen(form, lengths, H=1, HV=1, K=128, V=128, P=320, seed=78, raw_gates=form == "kda")
    prefill_check(w, cuda_device)


@pytest.mark.parametrize("form", ["gdn", "kda"])
def test_prefill_bad_spans(form, cuda_device):
    w = W.make_varlen(form, [40, 6, 3, 5], H=1, HV=2, K=128, V=128, seed=72, separate_write=True,
                      raw_gates=form == "kda")
    cu = torch.tensor([0, 40, 46, 3, 80], dtype=torch.int32)       # [0,40) [40,46) [46,3) [3,80)
    prefill_check(w, cuda_device, cu_seqlens=cu, expect_err=lar.LAR_DEVERR_SEQLEN)


def test_kda_prefill_then_decode_equals_one_recurrence(cuda_device):
    """KDA: the chunked call over 300 tokens, then the multi-token decode of the
    next 4 from the state it left, against the oracle on all 304 tokens."""
    dev = cuda_device
    w = W.make_varlen("kda", [304], H=2, HV=2, K=128, V=128, P=4, seed=76, raw_gates=True)
    slot = torch.tensor([2], dtype=torch.int32, device=dev)
    pool = w.pool.to(dev)
    part = lambda x, a, b: P.to_dev(x[a:b], dev)
    kw = dict(A_log=P.to_dev(w.A_log, dev), dt_bias=P.to_dev(w.dt_bias, dev), qk_l2norm=True, gate_raw=True,
              beta_raw=True, scale=w.scale)
    lar.kda_prefill(part(w.q, 0, 300), part(w.k, 0, 300), part(w.v, 0, 300), part(w.g, 0, 300),
                    part(w.beta, 0, 300), pool, torch.tensor([0, 300], dtype=torch.int32, device=dev), slot, slot,
                    **kw)
    tail = lambda x: P.to_dev(x[300:304][None], dev)
    out = lar.kda_decode(tail(w.q), tail(w.k), tail(w.v), tail(w.g), tail(w.beta), pool, slot, slot, **kw)
    torch.cuda.synchronize()
    import oracle
    host = w.pool.clone()
    ref = oracle.kda_decode_varlen(w.q, w.k, w.v, w.g, w.beta, host, torch.tensor([0, 304]), torch.tensor([2]),
                                   torch.tensor([2]), A_log=w.A_log, dt_bias=w.dt_bias, qk_l2norm=True,
                                   gate_raw=True, beta_raw=True, scale=w.scale)
    P.assert_out_close(out[0], ref["out"][300:304])
    P.assert_state_close(pool[2].cpu(), ref["final_state"][0], "slot 2")


def test_prefill_then_decode_equals_one_recurrence(cuda_device):
    """Prefill 300 tokens of a sequence with the chunked call, then decode the
    next 4 tokens with the multi-token call reading the state it left: the
    outputs of the 4 decode tokens and the final state match the oracle run on
    all 304 tokens."""
    dev = cuda_device
    w = W.make_varlen("gdn", [304], H=2, HV=4, K=128, V=128, P=4, seed=73)
    slot = torch.tensor([1], dtype=torch.int32, device=dev)
    pool = w.pool.to(dev)
    part = lambda x, a, b: P.to_dev(x[a:b], dev)
    lar.gdn_prefill(part(w.q, 0, 300), part(w.k, 0, 300), part(w.v, 0, 300), part(w.g, 0, 300),
                    part(w.beta, 0, 300), pool, torch.tensor([0, 300], dtype=torch.int32, device=dev), slot, slot,
                    scale=w.scale)
    tail = lambda x: P.to_dev(x[300:304][None], dev)
    out = lar.gdn_decode(tail(w.q), tail(w.k), tail(w.v), tail(w.g), tail(w.beta), pool, slot, slot, scale=w.scale)
    torch.cuda.synchronize()
    import oracle
    host = w.pool.clone()
    ref = oracle.gdn_decode_varlen(w.q, w.k, w.v, w.g, w.beta, host, torch.tensor([0, 304]), torch.tensor([1]),
                                   torch.tensor([1]), scale=w.scale)
    P.assert_out_close(out[0], ref["out"][300:304])
    P.assert_state_close(pool[1].cpu(), ref["final_state"][0], "slot 1")


def test_prefill_close_to_token_by_token(cuda_device):
    """The chunked and the token-by-token calls on the same spans agree to
    within the oracle tolerances of each other (both are checked against the
    oracle elsewhere; this ties them together on a mixed batch)."""
    dev = cuda_device
    w = W.make_varlen("gdn", [1, 4, 40, 200, 0, 77], H=2, HV=4, K=128, V=128, seed=74, in_dtype=F32, out_dtype=F32)
    pa, pb = w.pool.to(dev), w.pool.to(dev)
    args = lambda: (*P.qkv_dev(w, dev), P.to_dev(w.g, dev), P.to_dev(w.beta, dev))
    cu, ri = P.to_dev(w.cu_seqlens, dev), P.to_dev(w.read_idx, dev)
    oa = lar.gdn_prefill(*args(), pa, cu, ri, scale=w.scale)
    ob = lar.gdn_decode_varlen(*args(), pb, cu, ri, scale=w.scale)
    torch.cuda.synchronize()
    P.assert_out_close(oa, ob.double().cpu().numpy())
    P.assert_state_close(pa.cpu(), pb.double().cpu().numpy(), "pool")


@pytest.mark.parametrize("form", ["gdn", "la"])
def test_prefill_unaligned_rows(form, cuda_device):
    """bf16 q / k / v rows that do not start on a 16-byte boundary cannot be
    staged through shared memory; such a call runs the general kernel (rows read
    element by element) and meets the same oracle tolerances as the aligned
    call, which runs the warp-specialised one."""
    dev = cuda_device
    w = W.make_varlen(form, [31, 70, 0, 129, 5], H=2, HV=2 if form == "gdn" else None, K=128, V=128, seed=77,
                      raw_gates=form == "gdn")
    q, k, v = (x.to(dev) for x in (w.q, w.k, w.v))

    def shifted(x):                      # the same values, rows starting 2 bytes past a 16-byte boundary
        buf = torch.zeros(*x.shape[:-1], x.shape[-1] + 1, dtype=x.dtype, device=dev)
        buf[..., 1:].copy_(x)
        return buf[..., 1:]

    def run(q_, k_, v_):
        pool = w.pool.to(dev)
        cu, ri = P.to_dev(w.cu_seqlens, dev), P.to_dev(w.read_idx, dev)
        if form == "la":
            out = lar.la_prefill(q_, k_, v_, P.to_dev(w.decay, dev), pool, cu, ri, scale=w.scale)
        else:
            out = lar.gdn_prefill(q_, k_, v_, P.to_dev(w.g, dev), P.to_dev(w.beta, dev), pool, cu, ri,
                                  A_log=P.to_dev(w.A_log, dev), dt_bias=P.to_dev(w.dt_bias, dev), scale=w.scale,
                                  qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw)
        return out, pool

    qs, ks, vs = shifted(q), shifted(k), shifted(v)
    assert qs.data_ptr() % 16 != 0 and torch.equal(qs, q)
    runs = [run(q, k, v), run(qs, ks, vs)]
    torch.cuda.synchronize()
    ref = P.run_oracle_varlen(w, w.pool.clone())
    import numpy as np
    covered = ~np.isnan(ref["out"]).all(axis=(1, 2))
    cov = torch.from_numpy(covered).to(dev)
    for out, pool in runs:
        P.assert_out_close(out[cov], ref["out"][covered])
        for n, slot in enumerate(w.read_idx.tolist()):
            P.assert_state_close(P.slot_state(pool, w, slot), ref["final_state"][n], f"slot {slot}")


def test_prefill_rejects_unsupported_shapes(cuda_device):
    dev = cuda_device
    w = W.make_varlen("gdn", [5, 3], H=1, HV=2, K=64, V=64, seed=75)
    with pytest.raises(RuntimeError):
        lar.gdn_prefill(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), w.pool.to(dev),
                        w.cu_seqlens.to(dev), w.read_idx.to(dev))
