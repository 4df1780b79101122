"""Variable-length spans through *_decode_varlen against the oracle.

N sequences packed token-major, sequence n owning tokens cu_seqlens[n] ..
cu_seqlens[n+1]-1 (the "varlen" mode the aiter KDA decode review names).  A
span longer than the kernel's chunk (12 tokens with an fp32 pool, 8 with a bf16
pool) is staged chunk by chunk, so long spans (a fused-recurrent prefill that
leaves its final state in the pool) exercise the chunk loop, and spans of
exactly one or two chunks its boundaries; short and empty spans, spans over several V tiles, GQA, bf16 pools
and caches, in-kernel gates, Lightning Attention, skipped and separate write
slots, reversed and overlong spans are all compared with the oracle.
"""
import pytest
import torch

import _parity as P
import workloads as W
import linear_attention_recurrent_gb300 as lar

pytestmark = pytest.mark.gpu
F32, BF16 = torch.float32, torch.bfloat16

MIXED = [1, 5, 0, 16, 17, 40, 3, 33, 2, 0, 64, 7]

CASES = {
    "gdn_mixed": dict(form="gdn", lengths=MIXED, H=2, HV=4, K=128, V=128),
    "gdn_mixed_cache": dict(form="gdn", lengths=MIXED, H=2, HV=4, K=128, V=128, cache_intermediate=True,
                            separate_write=True, skip_frac=0.25),
    "gdn_ragged_v_fp32": dict(form="gdn", lengths=[3, 18, 1, 0, 31], H=1, HV=2, K=64, V=100,
                              in_dtype=F32, out_dtype=F32),
    "gdn_bf16_pool": dict(form="gdn", lengths=MIXED, H=2, HV=4, K=128, V=128, state_dtype=BF16,
                          cache_intermediate=True),
    "gdn_single_tokens": dict(form="gdn", lengths=[1] * 37, H=4, HV=8, K=128, V=128),
    "gdn_one_long": dict(form="gdn", lengths=[200], H=2, HV=4, K=128, V=128),
    "gdn_k32_long_v": dict(form="gdn", lengths=[9, 20, 4], H=1, HV=3, K=32, V=600),
    "gdn_strided_pool": dict(form="gdn", lengths=[6, 0, 25, 16], H=2, HV=4, K=128, V=128, stride_mult=2),
    "kda_raw_gates": dict(form="kda", lengths=MIXED, H=2, HV=2, K=128, V=128, raw_gates=True),
    "kda_raw_cache_bf16": dict(form="kda", lengths=[2, 19, 0, 5], H=1, HV=2, K=64, V=72, raw_gates=True,
                               cache_intermediate=True, state_dtype=BF16, inter_dtype=F32),
    "la_mixed": dict(form="la", lengths=MIXED, H=3, K=128, V=128),
    "la_flat_bf16": dict(form="la", lengths=[4, 0, 21, 1], H=2, K=128, V=96, flat_pool=True,
                         state_dtype=BF16, cache_intermediate=True),
    "la_packed": dict(form="la", lengths=[7, 17, 3], H=2, K=128, V=128, packed=True),
    "gdn_chunk_edges": dict(form="gdn", lengths=[12, 24, 13, 25, 11, 1], H=1, HV=2, K=128, V=128),
    "gdn_chunk_edges_bf16": dict(form="gdn", lengths=[8, 16, 9, 17, 7, 1], H=1, HV=2, K=128, V=128,
                                 state_dtype=BF16, cache_intermediate=True),
    "kda_chunk_edges_k64": dict(form="kda", lengths=[12, 8, 24, 16], H=1, HV=2, K=64, V=64, raw_gates=True,
                                cache_intermediate=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_varlen_parity(name, cuda_device):
    kw = dict(CASES[name])
    form, lengths = kw.pop("form"), kw.pop("lengths")
    w = W.make_varlen(form, lengths, seed=61, **kw)
    P.varlen_check(w, cuda_device)


def test_varlen_equal_lengths_equals_batched_call(cuda_device):
    """Spans of equal length T give bit for bit what the batched call on the
    same tokens gives (the same kernel arithmetic, addressed differently)."""
    dev = cuda_device
    w = W.make_custom("gdn", B=6, T=4, H=2, HV=4, K=128, V=128, seed=62, cache_intermediate=True)
    pool_a, pool_b = w.pool.to(dev), w.pool.to(dev)
    out_a, inter_a = P.run_gpu(w, dev, pool=pool_a)
    fl = lambda x: P.to_dev(x, dev).reshape((-1,) + tuple(x.shape[2:]))
    cu = torch.arange(0, 25, 4, dtype=torch.int32, device=dev)
    inter_b = torch.empty((24, w.HV, w.V, w.K), device=dev, dtype=w.inter_dtype)
    out_b = lar.gdn_decode_varlen(fl(w.q), fl(w.k), fl(w.v), fl(w.g), fl(w.beta), pool_b, cu,
                                  P.to_dev(w.read_idx, dev), P.to_dev(w.write_idx, dev), inter=inter_b,
                                  scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_a.reshape(out_b.shape), out_b)
    assert torch.equal(inter_a.reshape(inter_b.shape), inter_b)
    assert torch.equal(pool_a, pool_b)


def test_varlen_bad_spans_flagged(cuda_device):
    """A reversed span and one past the token arrays are run as empty (the read
    state goes to the write slot) and set the SEQLEN bit; the other spans are
    unaffected."""
    w = W.make_varlen("gdn", [4, 6, 3, 5], H=1, HV=2, K=128, V=64, seed=63, separate_write=True)
    cu = torch.tensor([0, 4, 10, 3, 30], dtype=torch.int32)       # [0,4) [4,10) [10,3) [3,30)
    P.varlen_check(w, cuda_device, cu_seqlens=cu, expect_err=lar.LAR_DEVERR_SEQLEN)


def test_varlen_int64_offsets_and_indices(cuda_device):
    w = W.make_varlen("kda", [3, 0, 22], H=2, HV=4, K=128, V=128, seed=64, raw_gates=True,
                      index_dtype=torch.int64)
    P.varlen_check(w, cuda_device, cu_seqlens=w.cu_seqlens.to(torch.int64))


def test_varlen_chunked_prefill_then_decode(cuda_device):
    """A long sequence prefilled in two varlen calls (the state passing through
    the pool between them) and then decoded one token with the plain call
    matches the oracle running all tokens at once."""
    dev = cuda_device
    w = W.make_varlen("gdn", [45], H=2, HV=4, K=128, V=128, P=4, seed=65)
    slot = torch.tensor([2], dtype=torch.int32)
    pool = w.pool.to(dev)
    tok = lambda x, a, b: P.to_dev(x[a:b], dev)
    outs = []
    for a, b in ((0, 30), (30, 44)):
        cu = torch.tensor([0, b - a], dtype=torch.int32, device=dev)
        outs.append(lar.gdn_decode_varlen(tok(w.q, a, b), tok(w.k, a, b), tok(w.v, a, b), tok(w.g, a, b),
                                          tok(w.beta, a, b), pool, cu, slot.to(dev), slot.to(dev),
                                          scale=w.scale))
    last = lambda x: P.to_dev(x[44:45][None], dev)
    outs.append(lar.gdn_decode(last(w.q), last(w.k), last(w.v), last(w.g), last(w.beta), pool, slot.to(dev),
                               slot.to(dev), scale=w.scale).reshape(1, w.HV, w.V))
    torch.cuda.synchronize()
    host = w.pool.clone()
    import oracle
    ref = oracle.gdn_decode_varlen(w.q, w.k, w.v, w.g, w.beta, host, torch.tensor([0, 45]),
                                   torch.tensor([2]), torch.tensor([2]), scale=w.scale)
    P.assert_out_close(torch.cat(outs), ref["out"])
    P.assert_state_close(pool[2].cpu(), ref["final_state"][0], "slot 2")


def test_varlen_empty_batch_and_all_empty_spans(cuda_device):
    dev = cuda_device
    w = W.make_varlen("gdn", [0, 0, 0], H=1, HV=2, K=64, V=64, seed=66, separate_write=True)
    P.varlen_check(w, dev)
    cu = torch.zeros(1, dtype=torch.int32, device=dev)            # N = 0: nothing to do
    empty = torch.empty(0, dtype=torch.int32, device=dev)
    pool = w.pool.to(dev)
    before = pool.clone()
    lar.gdn_decode_varlen(*P.qkv_dev(w, dev), P.to_dev(w.g, dev), P.to_dev(w.beta, dev), pool, cu, empty, empty)
    torch.cuda.synchronize()
    assert torch.equal(pool, before)


def test_varlen_graph_replay(cuda_device):
    """A varlen call captured in a CUDA graph and replayed equals eager calls."""
    dev = cuda_device
    w = W.make_varlen("gdn", [3, 20, 1, 9], H=2, HV=4, K=128, V=128, seed=67)
    pool_g, pool_e = w.pool.to(dev), w.pool.to(dev)
    out_g = torch.empty(tuple(w.v.shape), dtype=w.out_dtype, device=dev)
    out_e = torch.empty_like(out_g)
    args = dict(zip("qkv", P.qkv_dev(w, dev)), g=P.to_dev(w.g, dev),
                beta=P.to_dev(w.beta, dev), cu_seqlens=P.to_dev(w.cu_seqlens, dev),
                read_idx=P.to_dev(w.read_idx, dev), write_idx=P.to_dev(w.write_idx, dev))
    side = torch.cuda.Stream(device=dev)
    call_g = lar.PreparedCall("gdn", scale=w.scale, stream=side, pool=pool_g, out=out_g, **args)
    call_e = lar.PreparedCall("gdn", scale=w.scale, stream=side, pool=pool_e, out=out_e, **args)
    with torch.cuda.stream(side):
        call_g()
        call_e()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        call_g()
        call_g()
    graph.replay()
    with torch.cuda.stream(side):
        call_e()
        call_e()
    torch.cuda.synchronize()
    assert torch.equal(out_g, out_e)
    assert torch.equal(pool_g, pool_e)


# Without a state cache and at K = V = 128 the spans of 16 tokens or more run in
# the chunked tensor-core kernels and the rest token by token, in one call: these
# cases put long and short spans side by side in every pool form, around the
# threshold, and with fp32 rows (the general chunked kernel instead of the
# warp-specialised one).
SPLIT_CASES = {
    "gdn_bf16_pool": dict(form="gdn", lengths=MIXED, H=2, HV=4, state_dtype=BF16),
    "kda_bf16_pool": dict(form="kda", lengths=MIXED, H=2, HV=2, raw_gates=True, state_dtype=BF16),
    "la_flat_bf16": dict(form="la", lengths=[4, 0, 21, 1, 40], H=2, flat_pool=True, state_dtype=BF16),
    "gdn_skip_write": dict(form="gdn", lengths=MIXED, H=2, HV=4, separate_write=True, skip_frac=0.25),
    "gdn_fp32_rows": dict(form="gdn", lengths=MIXED, H=2, HV=4, in_dtype=F32, out_dtype=F32),
    "gdn_threshold": dict(form="gdn", lengths=[15, 16, 17, 31, 32, 33, 1], H=1, HV=2),
    "kda_threshold": dict(form="kda", lengths=[15, 16, 17, 2], H=1, HV=2, raw_gates=True),
    # fewer tokens than one long span: the chunked kernel is not launched
    "gdn_no_long_span": dict(form="gdn", lengths=[3, 5, 2], H=1, HV=2),
    # more sequences than the chunked kernels rank by length: the long spans are
    # found in index order, and the grid has fewer rows than sequences
    "gdn_many_sequences": dict(form="gdn", lengths=[1, 2, 0, 3] * 70 + [16, 1, 33, 2, 20, 70, 1, 17],
                               H=1, HV=2, separate_write=True, skip_frac=0.1),
    "kda_many_sequences": dict(form="kda", lengths=[2, 1] * 140 + [18, 40, 1, 16], H=1, HV=1,
                               raw_gates=True),
}


@pytest.mark.parametrize("name", sorted(SPLIT_CASES))
def test_varlen_split_parity(name, cuda_device):
    kw = dict(SPLIT_CASES[name])
    form, lengths = kw.pop("form"), kw.pop("lengths")
    w = W.make_varlen(form, lengths, K=128, V=128, seed=71, **kw)
    P.varlen_check(w, cuda_device)


def test_varlen_split_bad_spans(cuda_device):
    """A reversed span and a long one past the token arrays: the chunked kernel
    leaves both alone, the token-by-token kernel runs them as empty and flags
    them; the valid long and short spans are unaffected."""
    w = W.make_varlen("gdn", [4, 20, 3, 30], H=1, HV=2, K=128, V=128, seed=72, separate_write=True)
    cu = torch.tensor([0, 4, 24, 3, 60], dtype=torch.int32)      # [0,4) [4,24) [24,3) [3,60) of 57 tokens
    P.varlen_check(w, cuda_device, cu_seqlens=cu, expect_err=lar.LAR_DEVERR_SEQLEN)


def test_varlen_split_overlong_span(cuda_device):
    """A long span past the token arrays (bad, flagged) with no span reversed:
    the split stays on and the valid long span runs in the chunked kernel."""
    w = W.make_varlen("gdn", [4, 20, 3, 30], H=1, HV=2, K=128, V=128, seed=74, separate_write=True)
    cu = torch.tensor([0, 4, 24, 24, 60], dtype=torch.int32)     # [0,4) [4,24) [24,24) [24,60) of 57 tokens
    P.varlen_check(w, cuda_device, cu_seqlens=cu, expect_err=lar.LAR_DEVERR_SEQLEN)


def test_varlen_split_many_sequences_reversed(cuda_device):
    """More sequences than the chunked kernels rank, one span reversed: every
    span runs token by token (a reversed span lets valid spans overlap, so the
    chunked kernel's grid bound would not hold)."""
    lengths = [1, 2] * 150 + [20, 3, 17]
    w = W.make_varlen("gdn", lengths, H=1, HV=2, K=128, V=128, seed=75, separate_write=True)
    cu = w.cu_seqlens.clone()
    cu[5] = int(cu[-1]) + 5                 # span 4 past the tokens, span 5 reversed; no two valid spans overlap
    P.varlen_check(w, cuda_device, cu_seqlens=cu, expect_err=lar.LAR_DEVERR_SEQLEN)


def test_varlen_split_absent_and_bad_slots(cuda_device):
    """Long spans that start from an absent slot (-1: zero state) or an
    out-of-range one (zero state, flagged), and one whose write slot is out of
    range (writeback skipped, flagged), beside short spans."""
    w = W.make_varlen("gdn", [20, 33, 5, 40, 2], H=1, HV=2, K=128, V=128, seed=73, separate_write=True)
    w.read_idx[0] = -1
    w.read_idx[1] = w.P + 3
    w.write_idx[3] = w.P + 1
    P.varlen_check(w, cuda_device, expect_err=lar.LAR_DEVERR_READ_SLOT | lar.LAR_DEVERR_WRITE_SLOT)
