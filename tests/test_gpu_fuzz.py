"""Seeded random parity sweeps: small decode problems with every option drawn at
random (form, K, V, T, B, GQA group, input / output / state / cache dtypes,
state layout, gate flags, separate and skipped writes, strided, flat and packed
pools), each checked in full against the oracle (outputs, cached states,
written slots, and every other pool byte untouched).  The draw is seeded, so a
failure names a reproducible case.
"""
import random

import pytest
import torch

import _parity as P
import workloads as W

pytestmark = pytest.mark.gpu
F32, BF16 = torch.float32, torch.bfloat16
N_CASES = 200


def draw_case(seed):
    rnd = random.Random(seed)
    form = rnd.choice(["gdn", "gdn", "kda", "la"])
    K = rnd.choice([16, 32, 64, 128])
    T = rnd.choice([1, 1, 2, 3, 4, 5, 8, 9])
    B = rnd.randint(1, 9)
    H = rnd.randint(1, 3)
    HV = H * rnd.choice([1, 1, 2, 3]) if form != "la" else H
    state_dtype = rnd.choice([F32, F32, BF16])
    inter_dtype = rnd.choice([None, F32, BF16])
    state_kv = form != "la" and rnd.random() < 0.3
    V = rnd.randint(1, 200)
    if state_kv:                       # a [k][v] row is a whole number of 16-byte chunks
        step = 8 if BF16 in (state_dtype, inter_dtype) else 4
        V = max(step, V - V % step)
    kw = dict(B=B, T=T, H=H, HV=HV, K=K, V=V, seed=1000 + seed, state_dtype=state_dtype,
              in_dtype=rnd.choice([F32, BF16]), out_dtype=rnd.choice([F32, BF16]),
              cache_intermediate=rnd.random() < 0.4, inter_dtype=inter_dtype,
              index_dtype=rnd.choice([torch.int32, torch.int64]))
    if form != "la":
        kw.update(raw_gates=rnd.random() < 0.5, state_kv=state_kv)
    if rnd.random() < 0.4:
        kw.update(separate_write=True, skip_frac=rnd.choice([0.0, 0.25, 0.5]))
    elif rnd.random() < 0.3:
        kw.update(skip_frac=0.34)
    layout = rnd.random()
    if form == "la" and layout < 0.5:
        kw.update(flat_pool=True)
    elif layout < 0.25:
        kw.update(stride_mult=rnd.choice([2, 3]))
    if H == HV and rnd.random() < 0.3:
        kw.update(packed=True)
    return form, kw


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed, cuda_device):
    form, kw = draw_case(seed)
    w = W.make_custom(form, **kw)
    P.full_check(w, cuda_device)


def draw_varlen_case(seed):
    """Random variable-length spans: 1-12 sequences of 0-40 tokens, the same
    option space as the fixed-T draw (bar the [k][v] layout and packed views)."""
    rnd = random.Random(10_000 + seed)
    form = rnd.choice(["gdn", "gdn", "kda", "la"])
    K = rnd.choice([16, 32, 64, 128])
    H = rnd.randint(1, 3)
    HV = H * rnd.choice([1, 1, 2, 3]) if form != "la" else H
    lengths = [rnd.choice([0, 1, 1, 2, 3, 5, 8, 9, 12, 13, 17, 25, 40]) for _ in range(rnd.randint(1, 12))]
    kw = dict(H=H, HV=HV, K=K, V=rnd.randint(1, 200), seed=2000 + seed,
              state_dtype=rnd.choice([F32, F32, BF16]), in_dtype=rnd.choice([F32, BF16]),
              out_dtype=rnd.choice([F32, BF16]), cache_intermediate=rnd.random() < 0.4,
              inter_dtype=rnd.choice([None, F32, BF16]), index_dtype=rnd.choice([torch.int32, torch.int64]))
    if form != "la":
        kw.update(raw_gates=rnd.random() < 0.5)
    if rnd.random() < 0.4:
        kw.update(separate_write=True, skip_frac=rnd.choice([0.0, 0.25, 0.5]))
    if form == "la":
        kw.update(flat_pool=rnd.random() < 0.5)
    elif rnd.random() < 0.25:
        kw.update(stride_mult=rnd.choice([2, 3]))
    return form, lengths, kw


@pytest.mark.parametrize("seed", range(60))
def test_random_varlen_case(seed, cuda_device):
    form, lengths, kw = draw_varlen_case(seed)
    w = W.make_varlen(form, lengths, **kw)
    P.varlen_check(w, cuda_device)
