"""The seeded input generator: determinism, shapes and the structure each
workload recipe promises (strided pool views, packed q/k/v views, distinct and
disjoint slots, the share of skipped writebacks)."""
import torch

import workloads as W


def test_deterministic():
    a, b = W.make("gdn_tiny"), W.make("gdn_tiny")
    for name in ("q", "k", "v", "g", "beta", "pool", "read_idx", "write_idx"):
        assert torch.equal(getattr(a, name), getattr(b, name))


def test_gdn_tiny_recipe():
    w = W.make("gdn_tiny")
    assert w.pool.shape == (4, 2, 16, 16) and w.out_dtype == torch.float32
    assert w.read_idx.tolist() == [3, 1] and w.write_idx.tolist() == [3, 1]
    assert torch.allclose(w.q.norm(dim=-1), torch.ones(2, 1, 2))
    assert (w.g < 0).all() and ((w.beta > 0) & (w.beta < 1)).all()


def test_gdn_b64_bytes():
    w = W.make("gdn_b64")
    assert w.pool.shape == (256, 32, 128, 128)
    assert len(set(w.read_idx.tolist())) == 64
    # 2048 (entry, v-head) states read and written, 64 KiB each, plus q/k/v/g/beta/out/idx
    assert w.algorithmic_bytes() == 268_435_456 + 1_589_760


def test_mtp_strided_recipe():
    w = W.make("gdn_mtp_strided")
    assert w.pool.shape == (128, 32, 128, 128) and not w.pool.is_contiguous()
    assert w.pool.data_ptr() == w.backing.data_ptr()
    assert w.pool.stride(0) == 2 * w.backing.stride(0)
    r, wr = w.read_idx.tolist(), w.write_idx.tolist()
    assert len(set(r)) == 16
    live = [x for x in wr if x >= 0]
    assert len(live) == 12 and wr.count(-1) == 4 and len(set(live)) == 12
    assert not set(live) & set(r)
    assert w.cache_intermediate


def test_la_packed_views():
    # the full LA pool is 2.7 GB; check the packed-view structure on a small custom case
    w = W.make_custom("la", B=4, T=1, H=3, K=16, V=8, packed=True, flat_pool=True)
    assert w.q.data_ptr() == w.fused.data_ptr()
    assert w.k.data_ptr() == w.fused.data_ptr() + 16 * w.fused.element_size()
    assert not w.q.is_contiguous() and w.pool.shape == (w.P * 3, 8, 16)
    lam = W.la_decay_rates(64)
    assert abs(float(lam[0]) - 0.4) < 1e-3 and abs(float(lam[-1]) - 0.99610) < 1e-4


def test_disjoint_sets():
    sets = W.disjoint_index_sets(256, 64, 4, seed=7)
    flat = torch.cat(sets).tolist()
    assert len(flat) == 256 and len(set(flat)) == 256


def test_varlen_recipe():
    w = W.make("gdn_varlen_b64")
    cu = w.cu_seqlens.long()
    lengths = (cu[1:] - cu[:-1]).tolist()
    assert cu[0] == 0 and len(lengths) == 64 and int(cu[-1]) == w.q.shape[0] == w.v.shape[0]
    assert sum(1 for x in lengths if 1 <= x <= 4) == 48 and sum(1 for x in lengths if 16 <= x <= 128) == 16
    assert w.q.shape[1:] == (16, 128) and w.v.shape[1:] == (32, 128) and w.g.shape == (w.q.shape[0], 32)
    assert w.tokens() == int(cu[-1])
    # 2 x 64 x 32 states of 64 KiB, plus q/k/v/g/beta/out of every token and the index arrays
    per_tok = 2 * (2 * 16 * 128 + 32 * 128) + 2 * 4 * 32 + 2 * 32 * 128
    assert w.algorithmic_bytes() == 2 * 64 * 32 * 65536 + w.tokens() * per_tok + 2 * 64 * 4 + 65 * 4


def test_make_varlen_layout():
    w = W.make_varlen("kda", [3, 0, 5], H=2, HV=4, K=16, V=8, seed=1, raw_gates=True, separate_write=True)
    assert w.q.shape == (8, 2, 16) and w.g.shape == (8, 4, 16) and w.beta.shape == (8, 4)
    assert w.cu_seqlens.tolist() == [0, 3, 3, 8] and w.B == 3
    assert not set(w.read_idx.tolist()) & set(w.write_idx.tolist())


def test_prefill_recipe():
    w = W.make("gdn_prefill_n16")
    cu = w.cu_seqlens.long()
    lengths = (cu[1:] - cu[:-1]).tolist()
    assert len(lengths) == 16 and all(256 <= x <= 1024 for x in lengths)
    assert w.meta["prefill"] and w.pool.shape == (64, 32, 128, 128) and w.q.shape[0] == int(cu[-1])
