"""StepGraph: a serving step (input copies, the call, output copies) captured
once as a CUDA graph.  Replays must equal the same steps run eagerly, bit for
bit, and pick up the host buffers' new contents on every replay."""
import pytest
import torch

import workloads as W
import linear_attention_recurrent_gb300 as lar

pytestmark = pytest.mark.gpu


def test_stepgraph_replays_equal_eager_steps(cuda_device):
    dev = cuda_device
    ws = [W.make_custom("gdn", B=8, T=1, H=2, HV=4, K=128, V=128, P=16, seed=90 + i) for i in range(3)]
    w0 = ws[0]
    stream = torch.cuda.Stream(dev)

    def staged(w):
        return {"q": w.q, "k": w.k, "v": w.v, "g": w.g, "beta": w.beta}

    # pinned host inputs and their device copies (the graph copies host -> device)
    host = {n: t.contiguous().pin_memory() for n, t in staged(w0).items()}
    devb = {n: torch.empty_like(t, device=dev) for n, t in host.items()}
    ri, wi = w0.read_idx.to(dev), w0.write_idx.to(dev)
    pool_g = w0.pool.to(dev)
    out_dev = torch.empty(w0.v.shape, dtype=w0.out_dtype, device=dev)
    out_host = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    call = lar.PreparedCall("gdn", scale=w0.scale, stream=stream, pool=pool_g, read_idx=ri, write_idx=wi,
                            out=out_dev, **devb)
    # the constructor's warm-up runs one eager step on pool_g; the eager reference
    # repeats it on its own pool
    graph = lar.StepGraph(call, copies_in=[(devb[n], host[n]) for n in host], copies_out=[(out_host, out_dev)],
                          stream=stream)
    pool_e = w0.pool.to(dev)
    lar.gdn_decode(*(staged(w0)[n].to(dev) for n in ("q", "k", "v", "g", "beta")), pool_e, ri, wi,
                   scale=w0.scale)
    torch.cuda.synchronize()
    for w in ws[1:]:
        for n, t in staged(w).items():
            host[n].copy_(t)
        graph.replay()
        stream.synchronize()
        out_e = lar.gdn_decode(*(staged(w)[n].to(dev) for n in ("q", "k", "v", "g", "beta")), pool_e, ri, wi,
                               scale=w0.scale)
        torch.cuda.synchronize()
        assert torch.equal(out_host, out_e.cpu())
        assert torch.equal(pool_g, pool_e)


def test_stepgraph_needs_its_own_stream(cuda_device):
    dev = cuda_device
    w = W.make_custom("gdn", B=2, T=1, H=1, HV=1, K=128, V=128, P=4, seed=95)
    call = lar.PreparedCall("gdn", scale=w.scale, q=w.q.to(dev), k=w.k.to(dev), v=w.v.to(dev), g=w.g.to(dev),
                            beta=w.beta.to(dev), pool=w.pool.to(dev), read_idx=w.read_idx.to(dev),
                            write_idx=w.write_idx.to(dev), out=torch.empty(w.v.shape, dtype=w.out_dtype, device=dev))
    with pytest.raises(ValueError):
        lar.StepGraph(call, stream=torch.cuda.default_stream(dev))
