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
