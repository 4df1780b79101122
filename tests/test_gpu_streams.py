"""The decode call under the execution models a serving loop uses: capture into
a CUDA graph and replay, concurrent calls on independent streams, and launches
back to back on one stream (the kernels use programmatic dependent launch, so a
launch may start while the previous one drains).  Every result is compared bit
for bit with plain eager launches of the same calls.
"""
import pytest
import torch

import _parity as P
import workloads as W
import linear_attention_recurrent_gb300 as lar

pytestmark = pytest.mark.gpu


def _call(w, dev, pool, out, stream):
    kw = dict(zip("qkv", P.qkv_dev(w, dev)), pool=pool,
              read_idx=P.to_dev(w.read_idx, dev), write_idx=P.to_dev(w.write_idx, dev), out=out)
    if w.form == "la":
        kw["decay"] = P.to_dev(w.decay, dev)
    else:
        kw.update(g=P.to_dev(w.g, dev), beta=P.to_dev(w.beta, dev), A_log=P.to_dev(w.A_log, dev),
                  dt_bias=P.to_dev(w.dt_bias, dev), qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw,
                  beta_raw=w.beta_raw)
    return lar.PreparedCall(w.form, scale=w.scale, stream=stream, **kw), kw


@pytest.mark.parametrize("form,T", [("gdn", 1), ("gdn", 3), ("kda", 1), ("la", 2)])
def test_graph_replay_equals_eager(form, T, cuda_device):
    """Three decode steps captured in one CUDA graph, replayed twice, against
    six eager steps on a copy of the pool: outputs and pool bit-identical."""
    dev = cuda_device
    w = W.make_custom(form, B=8, T=T, H=2, HV=4, K=128, V=128, seed=41, raw_gates=form == "kda",
                      flat_pool=form == "la")
    pool_g, pool_e = w.pool.to(dev), w.pool.to(dev)
    out_g = torch.empty(w.v.shape, dtype=w.out_dtype, device=dev)
    out_e = torch.empty_like(out_g)
    side = torch.cuda.Stream(device=dev)
    call_g, _ = _call(w, dev, pool_g, out_g, side)
    call_e, _ = _call(w, dev, pool_e, out_e, side)
    with torch.cuda.stream(side):
        call_g()                       # first launch outside capture: one-time attribute setup
        call_e()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(3):
            call_g()
    outs_g, outs_e = [], []
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        outs_g.append(out_g.clone())
    with torch.cuda.stream(side):
        for i in range(6):
            call_e()
            if i % 3 == 2:
                side.synchronize()
                outs_e.append(out_e.clone())
    torch.cuda.synchronize()
    for a, b in zip(outs_g, outs_e):
        assert torch.equal(a, b)
    assert torch.equal(pool_g, pool_e)


def test_independent_streams_equal_serial(cuda_device):
    """Two decode calls on disjoint slot sets of one pool, launched on two
    streams at once, give the same bytes as the same calls run one after the
    other."""
    dev = cuda_device
    w = W.make_custom("gdn", B=16, T=2, H=2, HV=4, K=128, V=128, P=40, seed=42, cache_intermediate=False)
    sets = W.disjoint_index_sets(w.P, w.B, 2, seed=7)
    pool_c, pool_s = w.pool.to(dev), w.pool.to(dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    outs = {}
    for tag, pool, streams in (("conc", pool_c, (s1, s2)), ("ser", pool_s, (s1, s1))):
        res = []
        for idx, st in zip(sets, streams):
            w.read_idx = idx
            w.write_idx = idx.clone()
            out = torch.empty(w.v.shape, dtype=w.out_dtype, device=dev)
            call, _ = _call(w, dev, pool, out, st)
            with torch.cuda.stream(st):
                call()
            res.append(out)
        torch.cuda.synchronize()
        outs[tag] = res
    for a, b in zip(outs["conc"], outs["ser"]):
        assert torch.equal(a, b)
    assert torch.equal(pool_c, pool_s)


def test_back_to_back_dependent_launches(cuda_device):
    """Ten in-place steps on the same slots, launched back to back on one
    stream without host synchronisation: each step reads the state the
    previous one wrote, so any overlap of dependent launches would show as a
    difference from ten steps with a synchronize between them."""
    dev = cuda_device
    w = W.make_custom("gdn", B=64, T=1, H=4, HV=8, K=128, V=128, seed=43)
    pool_a, pool_b = w.pool.to(dev), w.pool.to(dev)
    out_a = torch.empty(w.v.shape, dtype=w.out_dtype, device=dev)
    out_b = torch.empty_like(out_a)
    st = torch.cuda.Stream(device=dev)
    call_a, _ = _call(w, dev, pool_a, out_a, st)
    call_b, _ = _call(w, dev, pool_b, out_b, st)
    with torch.cuda.stream(st):
        for _ in range(10):
            call_a()
    torch.cuda.synchronize()
    for _ in range(10):
        with torch.cuda.stream(st):
            call_b()
        torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(pool_a, pool_b)


def test_calls_from_several_host_threads(cuda_device):
    """Four host threads, each with its own stream and its own disjoint slots,
    issue ten in-place steps at once (the first call of a configuration from
    any thread sets up the launch cache under its lock); the pool ends up as
    forty serial steps leave it."""
    import threading
    dev = cuda_device
    w = W.make_custom("gdn", B=8, T=1, H=2, HV=4, K=64, V=96, P=40, seed=44)
    sets = W.disjoint_index_sets(w.P, w.B, 4, seed=9)
    pool_t, pool_s = w.pool.to(dev), w.pool.to(dev)

    def steps(pool, idx, stream, n=10):
        w2 = W.make_custom("gdn", B=8, T=1, H=2, HV=4, K=64, V=96, P=40, seed=44)
        w2.read_idx, w2.write_idx = idx, idx.clone()
        out = torch.empty(w2.v.shape, dtype=w2.out_dtype, device=dev)
        call, _ = _call(w2, dev, pool, out, stream)
        with torch.cuda.stream(stream):
            for _ in range(n):
                call()
        stream.synchronize()

    errors = []

    def guarded(*args):
        try:
            steps(*args)
        except Exception as e:   # surfaced below: a thread's exception does not fail the test by itself
            errors.append(e)

    threads = [threading.Thread(target=guarded, args=(pool_t, idx, torch.cuda.Stream(device=dev)))
               for idx in sets]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    st = torch.cuda.Stream(device=dev)
    for idx in sets:
        steps(pool_s, idx, st)
    torch.cuda.synchronize()
    assert torch.equal(pool_t, pool_s)
