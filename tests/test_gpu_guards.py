"""Canary checks: the pool, the output and the state cache are carved out of
larger buffers whose surrounding bytes hold a sentinel (a NaN bit pattern), and
the slots a decode writes include the pool's last one, so any write past the
end of a row, a tile, a slot or a tensor lands in a guard.  After the call the
guards must be bit-identical and the results must match the oracle.
"""
import math

import pytest
import torch

import _parity as P
import workloads as W
import linear_attention_recurrent_gb300 as lar

pytestmark = pytest.mark.gpu
F32, BF16 = torch.float32, torch.bfloat16
GUARD = 4096   # elements on each side
_PATTERN = {F32: (torch.int32, 0x7FC0DEAD), BF16: (torch.int16, 0x7FC1)}


def _guarded(shape, dtype, dev):
    n = math.prod(shape)
    big = torch.empty(GUARD + n + GUARD, dtype=dtype, device=dev)
    idt, pat = _PATTERN[dtype]
    big.view(idt).fill_(pat)
    return big, big[GUARD:GUARD + n].view(shape)


def _guards_intact(big, dtype):
    idt, pat = _PATTERN[dtype]
    raw = big.view(idt)
    return bool((raw[:GUARD] == pat).all()) and bool((raw[-GUARD:] == pat).all())


def _with_last_slot(w):
    """Entry 0 reads and writes the pool's last slot (the one next to the
    guard); the other entries use distinct slots below it, in place."""
    gen = torch.Generator().manual_seed(7)
    others = torch.randperm(w.P - 1, generator=gen)[:w.B - 1]
    ri = torch.cat([torch.tensor([w.P - 1]), others]).to(w.read_idx.dtype)
    w.read_idx, w.write_idx = ri, ri.clone()
    return w


CASES = {
    "gdn_ragged_v": dict(form="gdn", B=4, T=1, H=2, HV=4, K=128, V=100),
    "gdn_bf16_ragged_cache": dict(form="gdn", B=3, T=3, H=1, HV=2, K=64, V=72, state_dtype=BF16,
                                  cache_intermediate=True),
    "gdn_kv_ragged": dict(form="gdn", B=3, T=2, H=1, HV=2, K=128, V=100, state_kv=True,
                          cache_intermediate=True),
    "kda_cache_k32": dict(form="kda", B=5, T=2, H=2, HV=2, K=32, V=33, raw_gates=True,
                          cache_intermediate=True, in_dtype=F32, out_dtype=F32),
    "la_flat": dict(form="la", B=4, T=2, H=3, K=128, V=96, flat_pool=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_guards_and_parity(name, cuda_device):
    dev = cuda_device
    kw = dict(CASES[name])
    form = kw.pop("form")
    w = _with_last_slot(W.make_custom(form, seed=51, **kw))
    sdt = w.pool.dtype
    big_pool, pool = _guarded(tuple(w.pool.shape), sdt, dev)
    pool.copy_(w.pool.to(dev))
    before = pool.clone()
    big_out, out = _guarded(tuple(w.v.shape), w.out_dtype, dev)
    inter = big_inter = None
    if w.cache_intermediate:
        ishape = (w.B, w.T, w.HV, w.K, w.V) if w.state_kv else (w.B, w.T, w.HV, w.V, w.K)
        big_inter, inter = _guarded(ishape, w.inter_dtype, dev)
    cu = lambda t: None if t is None else t.to(dev)
    q, k, v = P.qkv_dev(w, dev)
    if form == "la":
        lar.la_decode(q, k, v, cu(w.decay), pool, cu(w.read_idx), cu(w.write_idx),
                      out=out, inter=inter, scale=w.scale)
    else:
        fn = lar.gdn_decode if form == "gdn" else lar.kda_decode
        fn(q, k, v, cu(w.g), cu(w.beta), pool, cu(w.read_idx), cu(w.write_idx),
           out=out, inter=inter, A_log=cu(w.A_log), dt_bias=cu(w.dt_bias), scale=w.scale,
           qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw, state_kv=w.state_kv)
    torch.cuda.synchronize()
    assert _guards_intact(big_pool, sdt), "pool guard overwritten"
    assert _guards_intact(big_out, w.out_dtype), "output guard overwritten"
    if big_inter is not None:
        assert _guards_intact(big_inter, w.inter_dtype), "cache guard overwritten"

    host = w.pool.clone()
    ref = P.run_oracle(w, host)
    P.assert_out_close(out, ref["out"])
    tr = (lambda x: x.transpose(-1, -2)) if w.state_kv else (lambda x: x)
    if inter is not None:
        P.assert_state_close(tr(inter), ref["inter"], "inter")
    written = set()
    for b, s in enumerate(w.write_idx.tolist()):
        if 0 <= s < w.P:
            written.add(s)
            P.assert_state_close(tr(P.slot_state(pool, w, s)), ref["final_state"][b], f"slot {s}")
    for s in range(w.P):
        if s not in written:
            assert torch.equal(P.slot_state(pool, w, s), P.slot_state(before, w, s)), f"slot {s} changed"


def test_guards_token_slots(cuda_device):
    """Per-token slots: the last token of entry 0 is stored to the pool's last
    slot; guards around the pool and the output stay intact."""
    dev = cuda_device
    w = W.make_custom("gdn", B=3, T=3, H=1, HV=2, K=128, V=100, P=12, seed=52)
    gen = torch.Generator().manual_seed(8)
    table = torch.randperm(w.P - 1, generator=gen)[:w.B * w.T].view(w.B, w.T)
    table[0, w.T - 1] = w.P - 1
    accepted = torch.tensor([w.T, 1, 2], dtype=torch.int32)
    big_pool, pool = _guarded(tuple(w.pool.shape), w.pool.dtype, dev)
    pool.copy_(w.pool.to(dev))
    big_out, out = _guarded(tuple(w.v.shape), w.out_dtype, dev)
    lar.gdn_decode_tokens(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), pool,
                          table.to(torch.int32).to(dev), num_accepted=accepted.to(dev), out=out, scale=w.scale)
    torch.cuda.synchronize()
    assert _guards_intact(big_pool, w.pool.dtype), "pool guard overwritten"
    assert _guards_intact(big_out, w.out_dtype), "output guard overwritten"
    import oracle
    host = w.pool.clone()
    ref = oracle.gdn_decode_tokens(w.q, w.k, w.v, w.g, w.beta, host, table.to(torch.int64),
                                   num_accepted=accepted.to(torch.int64), scale=w.scale)
    P.assert_out_close(out, ref["out"])
    P.assert_state_close(pool.cpu(), host.double().numpy(), "pool")


def test_guards_varlen(cuda_device):
    """Variable-length spans with an empty span and three trailing tokens that
    belong to no span: sequence 0 updates the pool's last slot in place; the
    guards around the pool, the output and the cache stay intact, and the
    output and cache rows of the trailing tokens keep their sentinel bits."""
    dev = cuda_device
    w = W.make_varlen("gdn", [5, 0, 14, 1, 3], H=1, HV=2, K=128, V=100, P=12, seed=53, cache_intermediate=True)
    N = 4
    w.cu_seqlens = w.cu_seqlens[:N + 1].clone()
    ri = torch.tensor([w.P - 1, 3, 7, 0], dtype=torch.int32)
    w.read_idx, w.write_idx = ri, torch.tensor([w.P - 1, 5, 7, -1], dtype=torch.int32)
    big_pool, pool = _guarded(tuple(w.pool.shape), w.pool.dtype, dev)
    pool.copy_(w.pool.to(dev))
    ntok = w.v.shape[0]
    big_out, out = _guarded((ntok, w.HV, w.V), w.out_dtype, dev)
    big_inter, inter = _guarded((ntok, w.HV, w.V, w.K), w.inter_dtype, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    lar.gdn_decode_varlen(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), pool,
                          w.cu_seqlens.to(dev), w.read_idx.to(dev), w.write_idx.to(dev), out=out, inter=inter,
                          scale=w.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _guards_intact(big_pool, w.pool.dtype), "pool guard overwritten"
    assert _guards_intact(big_out, w.out_dtype), "output guard overwritten"
    assert _guards_intact(big_inter, w.inter_dtype), "cache guard overwritten"
    idt, pat = _PATTERN[w.out_dtype]
    assert bool((out[20:].contiguous().view(idt) == pat).all()), "output rows outside every span written"
    idt, pat = _PATTERN[w.inter_dtype]
    assert bool((inter[20:].contiguous().view(idt) == pat).all()), "cache rows outside every span written"
    import oracle
    host = w.pool.clone()
    ref = oracle.gdn_decode_varlen(w.q, w.k, w.v, w.g, w.beta, host, w.cu_seqlens, w.read_idx, w.write_idx,
                                   scale=w.scale, cache_intermediate=True)
    P.assert_out_close(out[:20], ref["out"][:20])
    P.assert_state_close(inter[:20], ref["inter"][:20], "inter")
    P.assert_state_close(pool.cpu(), host.double().numpy(), "pool")
