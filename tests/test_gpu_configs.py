"""The named workloads at full size, in the launch configuration bench.py
times: sampled batch entries (first, last and six seeded others) against the
fp64 oracle, every untouched pool byte bit-identical, written states finite."""
import pytest
import torch

import _parity as P
import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample(B, seed=0, n=6):
    rest = torch.randperm(B - 2, generator=torch.Generator().manual_seed(seed))[:n] + 1
    return sorted({0, B - 1, *rest.tolist()})


@pytest.mark.parametrize("name", ["gdn_b64", "gdn_mtp_strided", "kda_b256", "la_b512_packed",
                                  "gdn_b64_bf16", "gdn_b64_kv", "gdn_b64_kv_bf16", "kda_b256_bf16",
                                  "la_b512_bf16"])
def test_full_size(name, cuda_device):
    dev = cuda_device
    w = W.make(name, pool_device=dev)
    storage = P.storage(w)
    before = storage.clone()
    mult = w.pool.stride(0) // w.backing.stride(0) if w.backing is not None else 1
    before_view = before[::mult] if w.backing is not None else before
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, inter = P.run_gpu(w, dev, pool=w.pool, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    mask = P.written_mask(w).to(dev)
    assert torch.equal(storage[~mask], before[~mask]), "untouched pool bytes changed"
    assert torch.isfinite(storage[mask]).all()

    sample = _sample(w.B)
    n = len(sample)
    ri = w.read_idx.long()
    shape = (n * w.HV,) + tuple(w.pool.shape[1:]) if w.pool.dim() == 3 else (n,) + tuple(w.pool.shape[1:])
    sub = torch.zeros(shape, dtype=w.pool.dtype)
    for i, b in enumerate(sample):
        r = int(ri[b])
        if 0 <= r < w.P:
            if w.pool.dim() == 3:
                sub[i * w.HV:(i + 1) * w.HV] = P.slot_state(before_view, w, r).cpu()
            else:
                sub[i] = before_view[r].cpu()
    ri_sub = torch.full((w.B,), -1, dtype=torch.int64)
    ri_sub[sample] = torch.arange(n)
    wi_sub = torch.full((w.B,), -1, dtype=torch.int64)
    ref = P.run_oracle(w, sub, read_idx=ri_sub, write_idx=wi_sub, batch=sample)
    P.assert_out_close(out[sample], ref["out"].reshape(out[sample].shape))
    tr = (lambda x: x.transpose(-1, -2)) if w.state_kv else (lambda x: x)
    if inter is not None:
        P.assert_state_close(tr(inter[sample]), ref["inter"], "inter")
    wi = (w.write_idx if w.write_idx is not None else w.read_idx).tolist()
    for i, b in enumerate(sample):
        if 0 <= wi[b] < w.P:
            P.assert_state_close(tr(P.slot_state(w.pool, w, wi[b])), ref["final_state"][i],
                                 f"slot {wi[b]} (entry {b})")


def test_full_size_speculative_token_slots(cuda_device):
    """gdn_spec_b64 at full size: outputs of sampled entries and the state in
    every written slot of those entries against the oracle; every other pool
    byte bit-identical."""
    import linear_attention_recurrent_gb300 as lar
    import oracle
    dev = cuda_device
    w = W.make("gdn_spec_b64", pool_device=dev)
    before = w.pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = lar.gdn_decode_tokens(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), w.pool,
                                w.state_idx.to(dev), num_accepted=w.num_accepted.to(dev),
                                out_dtype=w.out_dtype, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    written = w.state_idx.view(-1).long()
    mask = torch.zeros(w.P, dtype=torch.bool)
    mask[written] = True
    assert torch.equal(w.pool[~mask.to(dev)], before[~mask.to(dev)])
    sample = _sample(w.B)
    n = len(sample)
    # sub-problem: the sampled rows of the slot table, renumbered into a small host pool
    sub_tab = torch.arange(n * w.T).view(n, w.T)
    sub = torch.zeros((n * w.T,) + tuple(w.pool.shape[1:]))
    for i, b in enumerate(sample):
        for t in range(w.T):
            sub[i * w.T + t] = before[int(w.state_idx[b, t])].cpu()
    idx = torch.tensor(sample)
    ref = oracle.gdn_decode_tokens(w.q[idx], w.k[idx], w.v[idx], w.g[idx], w.beta[idx], sub, sub_tab,
                                   num_accepted=w.num_accepted[idx], cache_intermediate=True)
    P.assert_out_close(out[idx], ref["out"])
    for i, b in enumerate(sample):
        for t in range(w.T):
            P.assert_state_close(w.pool[int(w.state_idx[b, t])], ref["inter"][i, t], f"entry {b} token {t}")


def test_full_size_varlen(cuda_device):
    """gdn_varlen_b64 at full size: every untouched pool byte bit-identical;
    sampled sequences (first, last, the longest and seeded others) against the
    oracle, outputs of their tokens and their written states."""
    import linear_attention_recurrent_gb300 as lar
    import oracle
    dev = cuda_device
    w = W.make("gdn_varlen_b64", pool_device=dev)
    before = w.pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = lar.gdn_decode_varlen(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), w.pool,
                                w.cu_seqlens.to(dev), w.read_idx.to(dev), w.write_idx.to(dev), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    mask = P.written_mask(w).to(dev)
    assert torch.equal(w.pool[~mask], before[~mask]), "untouched pool bytes changed"
    cu = w.cu_seqlens.long()
    lengths = cu[1:] - cu[:-1]
    # the longest span, the shortest one the chunked kernel takes (16 tokens or
    # more) and the longest one left to the token-by-token kernel, beside the
    # seeded sample
    long_ = (lengths >= 16).nonzero().flatten()
    short = (lengths < 16).nonzero().flatten()
    picks = {int(lengths.argmax()), int(long_[lengths[long_].argmin()]), int(short[lengths[short].argmax()])}
    sample = sorted(set(_sample(w.B)) | picks)
    for n in sample:
        lo, hi = int(cu[n]), int(cu[n + 1])
        sub = before[int(w.read_idx[n])].cpu()[None].clone()
        tok = lambda t: t[lo:hi]
        ref = oracle.gdn_decode_varlen(tok(w.q), tok(w.k), tok(w.v), tok(w.g), tok(w.beta), sub,
                                       torch.tensor([0, hi - lo]), torch.tensor([0]), torch.tensor([-1]))
        P.assert_out_close(out[lo:hi], ref["out"], f"sequence {n} out")
        P.assert_state_close(w.pool[int(w.write_idx[n])], ref["final_state"][0], f"sequence {n} state")


@pytest.mark.parametrize("name", ["gdn_prefill_n16", "kda_prefill_n16"])
def test_full_size_prefill(name, cuda_device):
    """The prefill workloads at full size through the chunked call: every
    untouched pool byte bit-identical; sampled sequences (first, last, the
    longest and seeded others) against the oracle, outputs of their tokens and
    their written states."""
    import linear_attention_recurrent_gb300 as lar
    import oracle
    dev = cuda_device
    w = W.make(name, pool_device=dev)
    before = w.pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    fn = lar.gdn_prefill if w.form == "gdn" else lar.kda_prefill
    ofn = oracle.gdn_decode_varlen if w.form == "gdn" else oracle.kda_decode_varlen
    gates = dict(A_log=w.A_log, dt_bias=w.dt_bias, qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw,
                 beta_raw=w.beta_raw)
    dev_gates = {n: (x.to(dev) if isinstance(x, torch.Tensor) else x) for n, x in gates.items()}
    out = fn(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), w.pool,
             w.cu_seqlens.to(dev), w.read_idx.to(dev), w.write_idx.to(dev), dev_err=err, **dev_gates)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    mask = P.written_mask(w).to(dev)
    assert torch.equal(w.pool[~mask], before[~mask]), "untouched pool bytes changed"
    cu = w.cu_seqlens.long()
    lengths = cu[1:] - cu[:-1]
    sample = sorted({0, w.B - 1, int(lengths.argmax()), 5, 9})
    for n in sample:
        lo, hi = int(cu[n]), int(cu[n + 1])
        sub = before[int(w.read_idx[n])].cpu()[None].clone()
        tok = lambda t: t[lo:hi]
        ref = ofn(tok(w.q), tok(w.k), tok(w.v), tok(w.g), tok(w.beta), sub,
                  torch.tensor([0, hi - lo]), torch.tensor([0]), torch.tensor([-1]), **gates)
        P.assert_out_close(out[lo:hi], ref["out"], f"sequence {n} out")
        P.assert_state_close(w.pool[int(w.write_idx[n])], ref["final_state"][0], f"sequence {n} state")
