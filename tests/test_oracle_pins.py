"""Pins for the fp64 CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something other than itself: hand-computed
K=V=2 steps (tests/golden/hand_cases.json), an algebraically different closed
form of the recurrence, a library routine (numpy matmul, torch softplus /
sigmoid / normalize), or an invariant that the pages state (slot placement does
not change a sequence's result, untouched slots stay bit-identical, negative
write slots skip the writeback, strided pools are written in place).

Recurrence (ROCm/aiter PR #4584, advisory review): per token
    S <- exp(g_t) S;  S <- S + beta_t k_t (x) (v_t - S^T k_t);  o_t = S^T q_t.
Pool semantics: flashinfer "fp32 sibling of #3268" (read/write slots, -1 skip,
in-place strided 4D pool, intermediate-state cache) and cuLA PR #75 (LA state at
row h0_indices[n] * H + h).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _t(x, dtype=torch.float64):
    return torch.tensor(x, dtype=dtype)


# --------------------------------------------------------------------------- hand cases

def _run_hand_case(case):
    form = case["form"]
    S0 = np.array(case["S0"], dtype=np.float64)          # K x V
    K, V = S0.shape
    toks = case["tokens"]
    T = len(toks)
    pool = torch.zeros(3, 1, V, K, dtype=torch.float32)
    pool[1, 0] = torch.from_numpy(S0.T.copy()).float()   # storage is S^T
    pool[2] = 7.0                                        # a slot nobody touches
    before = pool.clone()
    q = _t([[t["q"]] for t in toks])[None]               # [1,T,1,K]
    k = _t([[t["k"]] for t in toks])[None]
    v = _t([[t["v"]] for t in toks])[None]
    ri, wi = torch.tensor([1]), torch.tensor([0])
    if form == "la":
        lam = _t([toks[0]["decay"]])
        res = oracle.la_decode(q, k, v, lam, pool.view(3, V, K), ri, wi,
                               cache_intermediate=True)
    else:
        raw = case.get("raw")
        if raw:
            g = _t([[t["g_raw"]] for t in toks])[None]
            beta = _t([[t["beta_raw"]] for t in toks])[None]
            A_log = _t([raw["A_log"]])
            dtb = raw["dt_bias"]
            dt_bias = _t(dtb if isinstance(dtb, list) else [dtb])
            kw = dict(A_log=A_log, dt_bias=dt_bias, gate_raw=True, beta_raw=True)
        else:
            g = torch.log(_t([[t["decay"]] for t in toks]))[None]
            beta = _t([[t["beta"]] for t in toks])[None]
            kw = {}
        fn = oracle.kda_decode if form == "kda" else oracle.gdn_decode
        res = fn(q, k, v, g, beta, pool, ri, wi, cache_intermediate=True, **kw)
    return res, pool, before, toks


@pytest.mark.parametrize("name", [c["name"] for c in json.load(open(GOLDEN))["cases"]])
def test_hand_cases(name):
    case = next(c for c in json.load(open(GOLDEN))["cases"] if c["name"] == name)
    # exact where only +,*,- on dyadic values occur; exp(log(d)) may cost 1-2 ulp
    tol = case.get("tol", 0.0 if case["form"] == "la" else 1e-15)
    res, pool, before, toks = _run_hand_case(case)
    for t, tok in enumerate(toks):
        np.testing.assert_allclose(res["out"][0, t, 0], tok["o"], rtol=0, atol=tol)
        np.testing.assert_allclose(res["inter"][0, t, 0], np.array(tok["S"]).T, rtol=0, atol=tol)
    S_T = np.array(toks[-1]["S"]).T
    np.testing.assert_allclose(res["final_state"][0, 0], S_T, rtol=0, atol=tol)
    np.testing.assert_allclose(pool[0, 0].double().numpy(), S_T, rtol=0, atol=max(tol, 1e-7))
    assert torch.equal(pool[1:], before[1:])             # read slot and bystander untouched
    assert res["n_bad"] == 0


# --------------------------------------------------------------------------- closed forms

def _rand_delta_case(per_channel, B=3, T=3, H=2, HV=4, K=8, V=6, P=7, seed=0):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(B, T, H, K, generator=gen, dtype=torch.float64)
    k = F.normalize(torch.randn(B, T, H, K, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(B, T, HV, V, generator=gen, dtype=torch.float64)
    gshape = (B, T, HV, K) if per_channel else (B, T, HV)
    g = -torch.rand(gshape, generator=gen, dtype=torch.float64)
    beta = torch.rand(B, T, HV, generator=gen, dtype=torch.float64)
    pool = torch.randn(P, HV, V, K, generator=gen) * 0.5
    ri = torch.tensor([4, -1, 2][:B])
    wi = torch.tensor([4, 6, -1][:B])
    return q, k, v, g, beta, pool, ri, wi


@pytest.mark.parametrize("per_channel", [False, True])
def test_delta_rule_matches_householder_product_form(per_channel):
    """Each token is S <- (I - beta k k^T) D S + beta k v^T, D = diag(exp(g)):
    the same update written as one matrix product (K x V orientation)."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(per_channel)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    pool0 = pool.clone()
    fn = oracle.kda_decode if per_channel else oracle.gdn_decode
    res = fn(q, k, v, g, beta, pool, ri, wi, cache_intermediate=True, scale=0.75)
    for b in range(B):
        for hv in range(HV):
            h = hv // (HV // H)
            r = int(ri[b])
            S = pool0[r, hv].double().numpy().T.copy() if r >= 0 else np.zeros((K, V))
            for t in range(T):
                d = g[b, t, hv].numpy() if per_channel else np.full(K, float(g[b, t, hv]))
                kk = k[b, t, h].numpy()
                bt = float(beta[b, t, hv])
                S = (np.eye(K) - bt * np.outer(kk, kk)) @ np.diag(np.exp(d)) @ S \
                    + bt * np.outer(kk, v[b, t, hv].numpy())
                np.testing.assert_allclose(res["out"][b, t, hv], 0.75 * S.T @ q[b, t, h].numpy(),
                                           rtol=0, atol=1e-12)
                np.testing.assert_allclose(res["inter"][b, t, hv], S.T, rtol=0, atol=1e-12)
            np.testing.assert_allclose(res["final_state"][b, hv], S.T, rtol=0, atol=1e-12)
    # writeback: slot 4 (b=0, in place) and 6 (b=1) written; b=2 skipped (-1)
    for b, w in ((0, 4), (1, 6)):
        np.testing.assert_allclose(pool[w].double().numpy(), res["final_state"][b],
                                   rtol=1e-7, atol=1e-7)
    untouched = [p for p in range(pool.shape[0]) if p not in (4, 6)]
    assert torch.equal(pool[untouched], pool0[untouched])


def test_la_matches_unrolled_closed_form():
    """S_t = lambda^(t+1) S_0 + sum_{s<=t} lambda^(t-s) k_s v_s^T, o_t = S_t^T q_t."""
    gen = torch.Generator().manual_seed(1)
    B, T, H, K, V, P = 2, 4, 3, 8, 5, 5
    q = torch.randn(B, T, H, K, generator=gen, dtype=torch.float64)
    k = torch.randn(B, T, H, K, generator=gen, dtype=torch.float64)
    v = torch.randn(B, T, H, V, generator=gen, dtype=torch.float64)
    lam = torch.tensor([0.5, 0.9, 1.0], dtype=torch.float64)
    pool = torch.randn(P * H, V, K, generator=gen)
    pool0 = pool.clone()
    ri = torch.tensor([3, 1])
    res = oracle.la_decode(q, k, v, lam, pool, ri, cache_intermediate=True)
    for b in range(B):
        for h in range(H):
            S0 = pool0[int(ri[b]) * H + h].double().numpy().T
            L = float(lam[h])
            for t in range(T):
                St = L ** (t + 1) * S0 + sum(
                    L ** (t - s) * np.outer(k[b, s, h].numpy(), v[b, s, h].numpy())
                    for s in range(t + 1))
                np.testing.assert_allclose(res["inter"][b, t, h], St.T, rtol=0, atol=1e-12)
                np.testing.assert_allclose(res["out"][b, t, h], St.T @ q[b, t, h].numpy(),
                                           rtol=0, atol=1e-12)
    # rows r*H + h of the flat pool were rewritten in place, nothing else
    written = [int(r) * H + h for r in ri for h in range(H)]
    other = [i for i in range(P * H) if i not in written]
    assert torch.equal(pool[other], pool0[other])
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(pool[int(ri[b]) * H + h].double().numpy(),
                                       res["final_state"][b, h], rtol=1e-7, atol=1e-7)


def test_delta_rule_projection_property():
    """With beta = 1 and a unit key, the updated state maps k exactly to v."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False, B=2, T=1)
    beta = torch.ones_like(beta)
    res = oracle.gdn_decode(q, k, v, g, beta, pool, ri, wi)
    HV, H = v.shape[2], q.shape[2]
    for b in range(2):
        for hv in range(HV):
            S = res["final_state"][b, hv].T                     # K x V
            np.testing.assert_allclose(S.T @ k[b, 0, hv // (HV // H)].numpy(),
                                       v[b, 0, hv].numpy(), rtol=0, atol=1e-12)


def test_no_gate_no_beta_is_plain_readout():
    """g = 0, beta = 0: the state is bit-unchanged and o = S0^T q (numpy matmul)."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False, B=1, T=1)
    g.zero_()
    beta.zero_()
    pool0 = pool.clone()
    res = oracle.gdn_decode(q, k, v, g, beta, pool, ri, wi)
    for hv in range(v.shape[2]):
        S0 = pool0[4, hv].double().numpy()                     # [V,K]
        assert np.array_equal(res["final_state"][0, hv], S0)
        np.testing.assert_allclose(res["out"][0, 0, hv], S0 @ q[0, 0, hv // 2].numpy(),
                                   rtol=0, atol=1e-12)
    assert torch.equal(pool, pool0)                            # rewrote the same bits


def test_zero_initial_state_for_negative_read():
    """read -1: S0 = 0, so S = beta k v^T and o = beta (k.q) v."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False, B=2, T=1)
    res = oracle.gdn_decode(q, k, v, g, beta, pool, ri, wi)
    b = 1                                                      # ri[1] == -1
    for hv in range(v.shape[2]):
        h = hv // 2
        kq = float(k[b, 0, h] @ q[b, 0, h])
        np.testing.assert_allclose(res["out"][b, 0, hv], float(beta[b, 0, hv]) * kq * v[b, 0, hv].numpy(),
                                   rtol=0, atol=1e-12)


def test_kda_with_uniform_gate_equals_gdn():
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False)
    pool_a, pool_b = pool.clone(), pool.clone()
    a = oracle.gdn_decode(q, k, v, g, beta, pool_a, ri, wi, cache_intermediate=True)
    gk = g[..., None].expand(*g.shape, q.shape[-1]).contiguous()
    b = oracle.kda_decode(q, k, v, gk, beta, pool_b, ri, wi, cache_intermediate=True)
    for key in ("out", "final_state", "inter"):
        assert np.array_equal(a[key], b[key])
    assert torch.equal(pool_a, pool_b)


@pytest.mark.parametrize("per_channel", [False, True])
def test_gate_chain_matches_torch(per_channel):
    """In-kernel gate: g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b),
    against torch's softplus (threshold 20) and sigmoid in fp64."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(per_channel, seed=3)
    B, T, H, K = q.shape
    HV = v.shape[2]
    gen = torch.Generator().manual_seed(9)
    a = torch.randn(g.shape, generator=gen, dtype=torch.float64) * 4
    a.view(-1)[:3] = torch.tensor([25.0, 19.5, -30.0], dtype=torch.float64)  # both softplus branches
    b_raw = torch.randn(beta.shape, generator=gen, dtype=torch.float64) * 3
    A_log = torch.rand(HV, generator=gen, dtype=torch.float64) * math.log(16)
    dt_bias = torch.randn(HV * K if per_channel else HV, generator=gen, dtype=torch.float64) * 0.1
    fn = oracle.kda_decode if per_channel else oracle.gdn_decode
    p1, p2 = pool.clone(), pool.clone()
    raw = fn(q, k, v, a, b_raw, p1, ri, wi, A_log=A_log, dt_bias=dt_bias, gate_raw=True,
             beta_raw=True, cache_intermediate=True)
    if per_channel:
        x = a + dt_bias.view(HV, K)
        g_ref = -torch.exp(A_log)[:, None] * F.softplus(x)
    else:
        g_ref = -torch.exp(A_log) * F.softplus(a + dt_bias)
    act = fn(q, k, v, g_ref, torch.sigmoid(b_raw), p2, ri, wi, cache_intermediate=True)
    for key in ("out", "final_state", "inter"):
        np.testing.assert_allclose(raw[key], act[key], rtol=1e-12, atol=1e-13)


def test_l2norm_matches_normalize():
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False, seed=5)
    q, k = q * 1000, k * 1000      # eps effect 1e-6 / (2 |x|^2) ~ 5e-13
    p1, p2 = pool.clone(), pool.clone()
    a = oracle.gdn_decode(q, k, v, g, beta, p1, ri, wi, qk_l2norm=True)
    b = oracle.gdn_decode(F.normalize(q, dim=-1), F.normalize(k, dim=-1), v, g, beta, p2, ri, wi)
    np.testing.assert_allclose(a["out"], b["out"], rtol=0, atol=1e-10)
    np.testing.assert_allclose(a["final_state"], b["final_state"], rtol=0, atol=1e-10)


def test_l2norm_epsilon_inside_sqrt():
    """q = [3, 4]: q_hat = q / sqrt(25 + 1e-6); with S0 = I and g = beta = 0, o = q_hat."""
    q = _t([[[[3.0, 4.0]]]])
    k = _t([[[[1.0, 0.0]]]])
    v = _t([[[[0.0, 0.0]]]])
    pool = torch.eye(2).view(1, 1, 2, 2).clone()
    res = oracle.gdn_decode(q, k, v, _t([[[0.0]]]), _t([[[0.0]]]), pool, torch.tensor([0]),
                            torch.tensor([-1]), qk_l2norm=True)
    np.testing.assert_allclose(res["out"][0, 0, 0], np.array([3.0, 4.0]) / math.sqrt(25 + 1e-6),
                               rtol=0, atol=1e-16)


# --------------------------------------------------------------------------- indexing invariants

def _pool_with_states(states, slots, P):
    """Place per-sequence states [n,HV,V,K] at the given slots of a fresh pool."""
    HV, V, K = states.shape[1:]
    pool = torch.full((P, HV, V, K), -3.0)
    for i, s in enumerate(slots):
        pool[s] = states[i]
    return pool


@pytest.mark.parametrize("slots,P", [([0, 1, 2, 3], 4), ([2, 0, 5, 1], 6), ([3, 2, 1, 0], 4)])
def test_slot_placement_does_not_change_results(slots, P):
    """cuLA PR #75 pool tests: identity, non-identity (pool 6, [2,0,5,1]) and
    reversed offsets give the same per-sequence output and state."""
    gen = torch.Generator().manual_seed(11)
    B, T, H, HV, K, V = 4, 2, 1, 2, 4, 3
    states = torch.randn(B, HV, V, K, generator=gen)
    q = torch.randn(B, T, H, K, generator=gen, dtype=torch.float64)
    k = F.normalize(torch.randn(B, T, H, K, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(B, T, HV, V, generator=gen, dtype=torch.float64)
    g = -torch.rand(B, T, HV, generator=gen, dtype=torch.float64)
    beta = torch.rand(B, T, HV, generator=gen, dtype=torch.float64)
    ref_pool = _pool_with_states(states, [0, 1, 2, 3], 4)
    ref = oracle.gdn_decode(q, k, v, g, beta, ref_pool, torch.arange(4))
    pool = _pool_with_states(states, slots, P)
    before = pool.clone()
    res = oracle.gdn_decode(q, k, v, g, beta, pool, torch.tensor(slots))
    assert np.array_equal(res["out"], ref["out"])
    assert np.array_equal(res["final_state"], ref["final_state"])
    for i, s in enumerate(slots):
        assert torch.equal(pool[s], ref_pool[i])
    inactive = [p for p in range(P) if p not in slots]
    assert torch.equal(pool[inactive], before[inactive])


def test_gqa_map_equals_repeated_heads():
    """v-head hv uses q/k head hv // (HV / H): equal to HV independent heads
    with q/k repeated consecutively."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False)
    rep = v.shape[2] // q.shape[2]
    p1, p2 = pool.clone(), pool.clone()
    a = oracle.gdn_decode(q, k, v, g, beta, p1, ri, wi, cache_intermediate=True)
    b = oracle.gdn_decode(q.repeat_interleave(rep, dim=2), k.repeat_interleave(rep, dim=2),
                          v, g, beta, p2, ri, wi, cache_intermediate=True)
    for key in ("out", "final_state", "inter"):
        assert np.array_equal(a[key], b[key])
    assert torch.equal(p1, p2)


@pytest.mark.parametrize("mult", [2, 3])
def test_strided_pool_written_in_place(mult):
    """flashinfer 4D pool fix: a strided view of a bigger backing buffer is
    updated in place; the gap slots stay bit-identical."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(True)
    P = pool.shape[0]
    backing = torch.randn(P * mult, *pool.shape[1:], generator=torch.Generator().manual_seed(2))
    backing[::mult] = pool
    view = backing[::mult]
    assert not view.is_contiguous()
    before = backing.clone()
    flat = pool.clone()
    a = oracle.kda_decode(q, k, v, g, beta, view, ri, wi)
    b = oracle.kda_decode(q, k, v, g, beta, flat, ri, wi)
    assert np.array_equal(a["out"], b["out"])
    assert torch.equal(backing[::mult], flat)
    gaps = [i for i in range(P * mult) if i % mult]
    assert torch.equal(backing[gaps], before[gaps])


def test_flat_pool_equals_4d():
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False)
    P, HV, V, K = pool.shape
    p4, p3 = pool.clone(), pool.clone().view(P * HV, V, K)
    a = oracle.gdn_decode(q, k, v, g, beta, p4, ri, wi)
    b = oracle.gdn_decode(q, k, v, g, beta, p3, ri, wi)
    assert np.array_equal(a["out"], b["out"])
    assert torch.equal(p4.view(P * HV, V, K), p3)


def test_la_reads_row_slot_times_h_plus_h():
    """lambda = 1, k = 0: o = S^T q for S at flat row read_idx * H + h."""
    gen = torch.Generator().manual_seed(4)
    B, H, K, V, P = 3, 2, 4, 3, 5
    pool = torch.randn(P * H, V, K, generator=gen)
    q = torch.randn(B, H, K, generator=gen, dtype=torch.float64)
    k = torch.zeros(B, H, K, dtype=torch.float64)
    v = torch.randn(B, H, V, generator=gen, dtype=torch.float64)
    ri = torch.tensor([4, 0, 2])
    res = oracle.la_decode(q, k, v, torch.ones(H, dtype=torch.float64), pool.clone(), ri)
    for b in range(B):
        for h in range(H):
            S = pool[int(ri[b]) * H + h].double().numpy()       # [V,K]
            np.testing.assert_allclose(res["out"][b, 0, h], S @ q[b, h].numpy(), rtol=0, atol=1e-12)


def test_multi_token_equals_chained_single_tokens():
    """A T-token call equals T one-token calls chained through the pool (the
    chained form rounds the state to fp32 between tokens, so 1e-6 relative)."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(True, T=4)
    ri = torch.tensor([4, 0, 2])          # every entry carries its state through the pool
    wi = ri.clone()
    p_multi, p_chain = pool.clone(), pool.clone()
    multi = oracle.kda_decode(q, k, v, g, beta, p_multi, ri, wi, cache_intermediate=True)
    for t in range(4):
        one = oracle.kda_decode(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], g[:, t:t + 1],
                                beta[:, t:t + 1], p_chain, ri, wi)
        np.testing.assert_allclose(one["out"][:, 0], multi["out"][:, t], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(p_chain.numpy(), p_multi.numpy(), rtol=1e-6, atol=1e-6)
    # inter[:, T-1] is the final state
    assert np.array_equal(multi["inter"][:, -1], multi["final_state"])


def test_out_of_range_slots_are_counted_and_skipped():
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(False, B=2, T=1)
    P = pool.shape[0]
    before = pool.clone()
    ri = torch.tensor([P, 3])
    wi = torch.tensor([2, P + 5])
    res = oracle.gdn_decode(q, k, v, g, beta, pool, ri, wi)
    assert res["n_bad"] == 2
    # entry 0 read out of range -> zero state, its write to slot 2 still happens
    zero = oracle.gdn_decode(q[:1], k[:1], v[:1], g[:1], beta[:1], before.clone(),
                             torch.tensor([-1]), torch.tensor([-1]))
    assert np.array_equal(res["out"][0], zero["out"][0])
    others = [p for p in range(P) if p != 2]
    assert torch.equal(pool[others], before[others])


# --------------------------------------------------------------------------- bfloat16 pool

def _bf16_bits(x32: torch.Tensor) -> list:
    return (x32.to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF).tolist()


def test_round_bf16_matches_torch():
    """The oracle's fp64 -> bf16 rounding against torch's fp32 -> bf16 (round to
    nearest even) on values exactly representable in fp32, so both see one rounding."""
    gen = torch.Generator().manual_seed(21)
    vals = torch.randn(4000, generator=gen) * torch.exp2(torch.randint(-40, 40, (4000,), generator=gen).float())
    special = torch.tensor([0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 - 2 ** -9,
                            2 ** -130, 3 * 2 ** -134, 1e-40, -1e-42, 3.0e38, 3.4028234e38, -3.4028234e38,
                            65504.0, 0.1, -0.3], dtype=torch.float32)
    x = torch.cat([vals, special])
    got = [oracle.round_bf16(float(v)) for v in x.tolist()]
    assert got == _bf16_bits(x)


def test_bf16_pool_reads_exactly_and_writes_nearest():
    """A bf16 pool gives the same fp64 results as an fp32 pool holding the
    widened values; the written slots hold the bf16 nearest to the fp64 state."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(True, seed=13)
    pb = pool.to(torch.bfloat16)
    pf = pb.float()
    a = oracle.kda_decode(q, k, v, g, beta, pb, ri, wi, cache_intermediate=True)
    b = oracle.kda_decode(q, k, v, g, beta, pf, ri, wi, cache_intermediate=True)
    for key in ("out", "final_state", "inter"):
        assert np.array_equal(a[key], b[key])
    for bidx, w in ((0, 4), (1, 6)):
        x = a["final_state"][bidx]
        got = pb[w].double().numpy()
        # nearest: no other bf16 value is closer (the two neighbours of `got`)
        bits = pb[w].view(torch.int16).to(torch.int32) & 0xFFFF
        up = (bits + 1).to(torch.int16).view(torch.bfloat16).double().numpy()
        dn = (bits - 1).to(torch.int16).view(torch.bfloat16).double().numpy()
        err = np.abs(got - x)
        assert (err <= np.abs(up - x)).all() and (err <= np.abs(dn - x)).all()
    untouched = [p for p in range(pb.shape[0]) if p not in (4, 6)]
    assert torch.equal(pb[untouched], pool.to(torch.bfloat16)[untouched])


def test_bf16_la_flat_pool():
    gen = torch.Generator().manual_seed(3)
    B, H, K, V, P = 2, 2, 8, 4, 3
    q = torch.randn(B, H, K, generator=gen, dtype=torch.float64)
    k = torch.randn(B, H, K, generator=gen, dtype=torch.float64)
    v = torch.randn(B, H, V, generator=gen, dtype=torch.float64)
    lam = torch.tensor([0.5, 0.75], dtype=torch.float64)
    pb = torch.randn(P * H, V, K, generator=gen).to(torch.bfloat16)
    pf = pb.float()
    ri = torch.tensor([2, 0])
    a = oracle.la_decode(q, k, v, lam, pb, ri)
    b = oracle.la_decode(q, k, v, lam, pf, ri)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["final_state"], b["final_state"])
    for bi in range(B):
        for h in range(H):
            row = int(ri[bi]) * H + h
            exp = [oracle.round_bf16(x) for x in a["final_state"][bi, h].ravel().tolist()]
            got = (pb[row].view(torch.int16).to(torch.int32) & 0xFFFF).ravel().tolist()
            assert got == exp


# --------------------------------------------------------------------------- per-token pool slots

def _tok_case(per_channel, seed=17, B=3, T=4, P=16):
    q, k, v, g, beta, pool, _, _ = _rand_delta_case(per_channel, B=B, T=T, P=P, seed=seed)
    slots = torch.randperm(P, generator=torch.Generator().manual_seed(seed))[:B * T].view(B, T)
    return q, k, v, g, beta, pool, slots


@pytest.mark.parametrize("per_channel", [False, True])
def test_token_slots_hold_the_cached_states(per_channel):
    """Per-token slots receive exactly the states the intermediate cache holds
    (the state after token t), rounded to the pool type; nothing else changes."""
    q, k, v, g, beta, pool, slots = _tok_case(per_channel)
    ri = torch.tensor([3, -1, 9])
    p_plain, p_tok = pool.clone(), pool.clone()
    fn = oracle.kda_decode if per_channel else oracle.gdn_decode
    tfn = oracle.kda_decode_tokens if per_channel else oracle.gdn_decode_tokens
    ref = fn(q, k, v, g, beta, p_plain, ri, torch.full((3,), -1), cache_intermediate=True)
    res = tfn(q, k, v, g, beta, p_tok, slots, read_idx=ri)
    assert np.array_equal(res["out"], ref["out"])
    for b in range(3):
        for t in range(4):
            s = int(slots[b, t])
            assert torch.equal(p_tok[s], torch.from_numpy(ref["inter"][b, t]).float())
    others = [p for p in range(pool.shape[0]) if p not in slots.view(-1).tolist()]
    assert torch.equal(p_tok[others], pool[others])


def test_seed_is_the_state_after_the_last_accepted_token():
    """Speculative flow with one slot row per sequence, reused every step.
    Step 1 (seeded from a plain slot) stores the state after each token in the
    row; with a tokens accepted, (1) slot row[a-1] holds the state of running
    only those a tokens, and (2) step 2 seeded by num_accepted = a equals step
    2 seeded explicitly from slot row[a-1]."""
    q, k, v, g, beta, pool0, _ = _tok_case(False, B=2, T=4, P=24)
    table = torch.tensor([[3, 7, 1, 12], [5, 0, 9, 2]])
    seeds = torch.tensor([20, 21])
    pool = pool0.clone()
    oracle.gdn_decode_tokens(q, k, v, g, beta, pool, table, read_idx=seeds)          # step 1
    accepted = torch.tensor([2, 4])
    for b in range(2):
        a = int(accepted[b])
        chained = oracle.gdn_decode(q[b:b + 1, :a], k[b:b + 1, :a], v[b:b + 1, :a], g[b:b + 1, :a],
                                    beta[b:b + 1, :a], pool0.clone(), seeds[b:b + 1],
                                    torch.full((1,), -1))
        np.testing.assert_allclose(pool[int(table[b, a - 1])].double().numpy(),
                                   chained["final_state"][0], rtol=1e-6, atol=1e-7)
    q2, k2, v2, g2, beta2, _, _ = _tok_case(False, seed=99, B=2, T=4, P=24)
    pa, pb = pool.clone(), pool.clone()
    tok = oracle.gdn_decode_tokens(q2, k2, v2, g2, beta2, pa, table, num_accepted=accepted)  # step 2
    explicit = oracle.gdn_decode_tokens(q2, k2, v2, g2, beta2, pb, table,
                                        read_idx=torch.tensor([int(table[0, 1]), int(table[1, 3])]))
    assert np.array_equal(tok["out"], explicit["out"])
    assert torch.equal(pa, pb)


def test_accepted_count_outside_range_is_counted_with_zero_seed():
    q, k, v, g, beta, pool, slots = _tok_case(True, B=3, T=4)
    p1, p2 = pool.clone(), pool.clone()
    res = oracle.kda_decode_tokens(q, k, v, g, beta, p1, slots, num_accepted=torch.tensor([0, 5, 4]))
    assert res["n_bad"] == 2
    zero = oracle.kda_decode_tokens(q, k, v, g, beta, p2, slots, read_idx=torch.tensor([-1, -1, int(slots[2, 3])]))
    assert np.array_equal(res["out"], zero["out"])


def test_kv_layout_equals_transposed_pool():
    """Holding S untransposed ([.., k, v]) is only a different storage order: the
    results equal those of the [.., v, k] pool holding the transposed states,
    and the written slots are the transposes of each other."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(True, seed=23)
    p_vk = pool.clone()
    p_kv = pool.transpose(2, 3).contiguous()
    a = oracle.kda_decode(q, k, v, g, beta, p_vk, ri, wi, cache_intermediate=True)
    b = oracle.kda_decode(q, k, v, g, beta, p_kv, ri, wi, cache_intermediate=True, layout="kv")
    for key in ("out", "final_state", "inter"):
        assert np.array_equal(a[key], b[key])
    assert torch.equal(p_kv, p_vk.transpose(2, 3))


# --------------------------------------------------------------------------- variable-length spans
# (the aiter KDA review names a "varlen" mode: packed sequences of mixed length,
# token-major, delimited by cumulative offsets)

def _flat(x):
    return x.reshape((-1,) + tuple(x.shape[2:]))


@pytest.mark.parametrize("per_channel", [False, True])
def test_varlen_equal_lengths_equals_batched(per_channel):
    """Spans of equal length T over the token-major flattening of a [B, T, ..]
    batch give the batched results exactly: out row b*T + t is out[b, t] and
    the written slots match."""
    q, k, v, g, beta, pool, ri, wi = _rand_delta_case(per_channel, T=3, seed=31)
    pa, pb = pool.clone(), pool.clone()
    fn = oracle.kda_decode if per_channel else oracle.gdn_decode
    vfn = oracle.kda_decode_varlen if per_channel else oracle.gdn_decode_varlen
    ref = fn(q, k, v, g, beta, pa, ri, wi, cache_intermediate=True)
    cu = torch.tensor([0, 3, 6, 9])
    res = vfn(_flat(q), _flat(k), _flat(v), _flat(g), _flat(beta), pb, cu, ri, wi, cache_intermediate=True)
    assert np.array_equal(res["out"], _flat(torch.from_numpy(ref["out"])).numpy())
    assert np.array_equal(res["inter"], _flat(torch.from_numpy(ref["inter"])).numpy())
    assert np.array_equal(res["final_state"], ref["final_state"])
    assert torch.equal(pa, pb)


def test_varlen_split_span_equals_one_span():
    """A sequence decoded as one span of 7 tokens, or as a span of 3 whose state
    goes through a pool slot into a span of the next 4 (the chunk boundary of a
    prefill), ends in the same state with the same outputs (fp32 rounding of
    the state at the boundary: 1e-6 relative)."""
    q, k, v, g, beta, pool, _, _ = _rand_delta_case(True, B=1, T=7, P=6, seed=32)
    q, k, v, g, beta = _flat(q), _flat(k), _flat(v), _flat(g), _flat(beta)
    whole = oracle.kda_decode_varlen(q, k, v, g, beta, pool.clone(), torch.tensor([0, 7]),
                                     torch.tensor([2]), torch.tensor([5]))
    p = pool.clone()
    first = oracle.kda_decode_varlen(q[:3], k[:3], v[:3], g[:3], beta[:3], p, torch.tensor([0, 3]),
                                     torch.tensor([2]), torch.tensor([4]))
    second = oracle.kda_decode_varlen(q[3:], k[3:], v[3:], g[3:], beta[3:], p, torch.tensor([0, 4]),
                                      torch.tensor([4]), torch.tensor([5]))
    np.testing.assert_allclose(np.concatenate([first["out"], second["out"]]), whole["out"],
                               rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(second["final_state"], whole["final_state"], rtol=1e-6, atol=1e-7)


def test_varlen_empty_and_bad_spans():
    """An empty span applies no token: its write slot receives the state as
    read (bit-exact for an fp32 pool) and no output row belongs to it.  A span
    that is reversed or runs past the token arrays is counted and run as
    empty; tokens outside every span keep no output (NaN here)."""
    gen = torch.Generator().manual_seed(33)
    q = torch.randn(6, 1, 4, generator=gen, dtype=torch.float64)
    k = F.normalize(torch.randn(6, 1, 4, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(6, 1, 3, generator=gen, dtype=torch.float64)
    g = -torch.rand(6, 1, generator=gen, dtype=torch.float64)
    beta = torch.rand(6, 1, generator=gen, dtype=torch.float64)
    pool = torch.randn(8, 1, 3, 4, generator=gen)
    before = pool.clone()
    cu = torch.tensor([0, 2, 2, 5, 3, 9])          # spans [0,2) [2,2) [2,5) [5,3) [3,9)
    ri = torch.tensor([0, 1, 2, 3, 4])
    wi = torch.tensor([5, 6, 7, -1, 4])
    res = oracle.gdn_decode_varlen(q, k, v, g, beta, pool, cu, ri, wi)
    assert res["n_bad"] == 2
    assert torch.equal(pool[6], before[1])                       # empty span: copy
    assert torch.equal(pool[4], before[4])                       # bad span: run as empty, in place
    assert np.isnan(res["out"][5]).all()                         # token 5 lies in no valid span
    assert not np.isnan(res["out"][:5]).any()
    one = oracle.gdn_decode(q[None, 2:5], k[None, 2:5], v[None, 2:5], g[None, 2:5], beta[None, 2:5],
                            before.clone(), torch.tensor([2]), torch.tensor([-1]))
    assert np.array_equal(res["out"][2:5], one["out"][0])


# --------------------------------------------------------------------------- chunked (matrix) form

def _chunked_delta_rule(S0, q, k, v, a, beta, C):
    """The delta rule over T tokens in chunks of C, written as matrix products
    (numpy, fp64): per chunk, with P[t][s] = a_{s+1}..a_t and E_t = a_0..a_t,
    (I + tril_-1(beta_t P[t][s] k_t.k_s)) d = beta (v - E K S0),
    O = E Q S0 + (P o tril(Q K^T)) d,  S = E_last S0 + K^T (P[last][:] d).
    S0 is K x V; q, k [T, K]; v [T, V]; a (decay factors), beta [T]."""
    S = S0.copy()
    outs = []
    for c0 in range(0, len(a), C):
        qc, kc, vc, ac, bc = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C], a[c0:c0 + C], beta[c0:c0 + C]
        n = len(ac)
        P = np.zeros((n, n))
        for t in range(n):
            for s in range(t + 1):
                P[t, s] = np.prod(ac[s + 1:t + 1])
        E = np.cumprod(ac)
        A = np.tril(bc[:, None] * P * (kc @ kc.T), -1)
        R = bc[:, None] * (vc - E[:, None] * (kc @ S))
        d = np.linalg.solve(np.eye(n) + A, R)
        outs.append(E[:, None] * (qc @ S) + (P * (qc @ kc.T)) @ d)
        S = E[-1] * S + kc.T @ (P[-1][:, None] * d)
    return np.concatenate(outs), S


@pytest.mark.parametrize("C", [1, 4, 5, 16])
def test_delta_rule_matches_chunked_matrix_form(C):
    """The oracle's token-by-token delta rule equals the chunked matrix form
    (numpy solve and matmuls, any chunk size) on 11 tokens: outputs and final
    state to fp64 rounding.  With C = 1 the form reduces to the recurrence; with
    C > 1 it pins the decay / read-out / update order across a chunk."""
    gen = torch.Generator().manual_seed(81)
    T, K, V = 11, 6, 5
    q = torch.randn(1, T, 1, K, generator=gen, dtype=torch.float64)
    k = F.normalize(torch.randn(1, T, 1, K, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(1, T, 1, V, generator=gen, dtype=torch.float64)
    g = -torch.rand(1, T, 1, generator=gen, dtype=torch.float64)
    beta = torch.rand(1, T, 1, generator=gen, dtype=torch.float64)
    pool = torch.randn(2, 1, V, K, generator=gen, dtype=torch.float64).float()
    res = oracle.gdn_decode(q, k, v, g, beta, pool.clone(), torch.tensor([1]), torch.tensor([-1]))
    S0 = pool[1, 0].double().numpy().T                       # K x V
    o, S = _chunked_delta_rule(S0, q[0, :, 0].numpy(), k[0, :, 0].numpy(), v[0, :, 0].numpy(),
                               np.exp(g[0, :, 0].numpy()), beta[0, :, 0].numpy(), C)
    np.testing.assert_allclose(res["out"][0, :, 0], o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(res["final_state"][0, 0], S.T, rtol=1e-11, atol=1e-12)


def test_la_matches_chunked_matrix_form():
    """Lightning Attention is the chunked form with d = v (beta = 1 and no
    read-out correction): P and E from the constant rate lambda."""
    gen = torch.Generator().manual_seed(82)
    T, K, V, H = 9, 4, 3, 1
    q = torch.randn(1, T, H, K, generator=gen, dtype=torch.float64)
    k = torch.randn(1, T, H, K, generator=gen, dtype=torch.float64)
    v = torch.randn(1, T, H, V, generator=gen, dtype=torch.float64)
    lam = torch.tensor([0.8])
    pool = torch.randn(2 * H, V, K, generator=gen, dtype=torch.float64).float()
    res = oracle.la_decode(q, k, v, lam, pool.clone(), torch.tensor([1]), torch.tensor([-1]))
    S = pool[1].double().numpy().T
    a = np.full(T, float(lam[0]))
    outs = []
    C = 4
    for c0 in range(0, T, C):
        qc, kc, vc, ac = q[0, c0:c0 + C, 0].numpy(), k[0, c0:c0 + C, 0].numpy(), v[0, c0:c0 + C, 0].numpy(), a[c0:c0 + C]
        n = len(ac)
        P = np.array([[np.prod(ac[s + 1:t + 1]) if s <= t else 0.0 for s in range(n)] for t in range(n)])
        E = np.cumprod(ac)
        outs.append(E[:, None] * (qc @ S) + (P * (qc @ kc.T)) @ vc)
        S = E[-1] * S + kc.T @ (P[-1][:, None] * vc)
    np.testing.assert_allclose(res["out"][0, :, 0], np.concatenate(outs), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(res["final_state"][0, 0], S.T, rtol=1e-11, atol=1e-12)


def test_kda_matches_per_channel_chunked_form():
    """KDA (decay per key channel) equals its chunked form: with per-channel
    decay products P[t][s][k] = a_{s+1}[k]..a_t[k] and E_t[k] = a_0[k]..a_t[k],
    A[t][s] = beta_t sum_k k_t[k] P[t][s][k] k_s[k] (s < t),
    (I + A) d = beta (v - (E o K) S0),  o_t = (E_t o q_t) S0 + sum_{s<=t} (q_t . (P[t][s] o k_s)) d_s,
    S = diag(E_last) S0 + sum_s (P[last][s] o k_s) d_s^T  (numpy, fp64, chunk 4 over 10 tokens)."""
    gen = torch.Generator().manual_seed(83)
    T, K, V, C = 10, 5, 4, 4
    q = torch.randn(1, T, 1, K, generator=gen, dtype=torch.float64)
    k = F.normalize(torch.randn(1, T, 1, K, generator=gen, dtype=torch.float64), dim=-1)
    v = torch.randn(1, T, 1, V, generator=gen, dtype=torch.float64)
    g = -torch.rand(1, T, 1, K, generator=gen, dtype=torch.float64)
    beta = torch.rand(1, T, 1, generator=gen, dtype=torch.float64)
    pool = torch.randn(2, 1, V, K, generator=gen, dtype=torch.float64).float()
    res = oracle.kda_decode(q, k, v, g, beta, pool.clone(), torch.tensor([1]), torch.tensor([-1]))
    S = pool[1, 0].double().numpy().T                        # K x V
    qn, kn, vn = q[0, :, 0].numpy(), k[0, :, 0].numpy(), v[0, :, 0].numpy()
    an, bn = np.exp(g[0, :, 0].numpy()), beta[0, :, 0].numpy()
    outs = []
    for c0 in range(0, T, C):
        qc, kc, vc, ac, bc = qn[c0:c0 + C], kn[c0:c0 + C], vn[c0:c0 + C], an[c0:c0 + C], bn[c0:c0 + C]
        n = len(bc)
        P = np.zeros((n, n, K))
        for t in range(n):
            for s in range(t + 1):
                P[t, s] = np.prod(ac[s + 1:t + 1], axis=0) if t > s else np.ones(K)
        E = np.cumprod(ac, axis=0)                            # [n, K]
        A = np.zeros((n, n))
        Mq = np.zeros((n, n))
        for t in range(n):
            for s in range(t + 1):
                if s < t:
                    A[t, s] = bc[t] * np.sum(kc[t] * P[t, s] * kc[s])
                Mq[t, s] = np.sum(qc[t] * P[t, s] * kc[s])
        R = bc[:, None] * (vc - (E * kc) @ S)
        d = np.linalg.solve(np.eye(n) + A, R)
        outs.append((E * qc) @ S + Mq @ d)
        S = E[-1][:, None] * S + (P[-1] * kc).T @ d
    np.testing.assert_allclose(res["out"][0, :, 0], np.concatenate(outs), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(res["final_state"][0, 0], S.T, rtol=1e-11, atol=1e-12)
