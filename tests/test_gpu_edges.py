"""GPU parity on the method's degenerate inputs and at the boundary's maximum
sizes, against the fp64 oracle (whole workloads, every output and state).

Degenerate cases of the gated delta rule / Lightning-Attention recurrence:
beta = 0 (the state only decays), g = 0 (no decay), g = -inf (the state is
forgotten before the token is written), very negative g (exp underflows), beta
= 1, all-zero k rows under the in-kernel l2 norm (normalised to zero, so no
update), all-zero q (zero output) and all-zero v.  Maximum sizes: the largest
batch and v-head count the C ABI accepts (65535) and a value dimension far
past the shared-memory staging limit.
"""
import pytest
import torch

import _parity as P
import workloads as W

pytestmark = pytest.mark.gpu
F32 = torch.float32


def _degenerate_gates(w, gen):
    """Overwrite w's activated gates in place: each (b, t, hv) gets one of
    beta = 0, beta = 1, g = 0, g = -inf, g = -80 or its drawn value (for KDA
    the whole decay row of that (b, t, hv))."""
    pick = torch.randint(0, 6, tuple(w.beta.shape), generator=gen)
    w.beta[pick == 0] = 0.0
    w.beta[pick == 1] = 1.0
    for code, val in ((2, 0.0), (3, float("-inf")), (4, -80.0)):
        w.g[pick == code] = val


@pytest.mark.parametrize("form,state_dtype,T", [("gdn", F32, 1), ("gdn", F32, 3), ("kda", F32, 2),
                                                ("gdn", torch.bfloat16, 1)])
def test_degenerate_gates(form, state_dtype, T, cuda_device):
    w = W.make_custom(form, B=12, T=T, H=2, HV=4, K=128, V=96, seed=31, state_dtype=state_dtype,
                      cache_intermediate=T > 1)
    _degenerate_gates(w, torch.Generator().manual_seed(5))
    P.full_check(w, cuda_device)


@pytest.mark.parametrize("form", ["gdn", "kda", "la"])
def test_zero_vectors(form, cuda_device):
    """Zero k rows (l2-normalised in kernel for GDN/KDA: k_hat = 0), zero q rows
    and zero v rows on some tokens."""
    raw = form != "la"
    w = W.make_custom(form, B=6, T=3, H=2, HV=2, K=64, V=80, seed=32, raw_gates=raw, in_dtype=F32,
                      out_dtype=F32, cache_intermediate=True)
    gen = torch.Generator().manual_seed(6)
    for name in ("k", "q", "v"):
        t = getattr(w, name)
        m = torch.rand(t.shape[:3], generator=gen) < 0.3
        t[m] = 0.0
    P.full_check(w, cuda_device)


def test_max_batch(cuda_device):
    """B = 65535 (the ABI maximum) with a small state: many tiles per CTA."""
    w = W.make_custom("gdn", B=65535, T=1, H=1, HV=1, K=16, V=16, P=65536, seed=33, in_dtype=F32,
                      out_dtype=F32)
    P.full_check(w, cuda_device)


def test_max_value_heads(cuda_device):
    """HV = 65535 v-heads sharing one q/k head (a GQA group of 65535)."""
    w = W.make_custom("gdn", B=1, T=2, H=1, HV=65535, K=16, V=16, P=2, seed=34)
    P.full_check(w, cuda_device)


@pytest.mark.parametrize("state_kv", [False, True])
def test_long_value_dimension(state_kv, cuda_device):
    """V of 65540 / 65543 (far past the staged-v limit): v is read from global
    memory inside the token loop and the last tile is partial."""
    # a [k][v] row must be a whole number of 16-byte chunks: V a multiple of 4 there
    w = W.make_custom("gdn", B=2, T=2, H=1, HV=1, K=16, V=65540 if state_kv else 65543, seed=35,
                      state_kv=state_kv, separate_write=True)
    P.full_check(w, cuda_device)
