"""Helpers shared by the GPU parity tests: run a workload through the C ABI and
through the fp64 oracle, and compare.

Tolerances (written here once, used by every GPU test):
  * bf16 outputs: |gpu - oracle| <= 2e-3 where |oracle| < 1.  At |oracle| >= 1
    bf16 itself cannot hold o within 2e-3 (half an ulp there is >= 3.9e-3),
    so the bound is half a bf16 ulp of the oracle value plus 1e-4 relative.
  * fp32 state (pool writeback, intermediate cache) and fp32 outputs:
    |gpu - oracle| <= 1e-4 |oracle| + 1e-6, elementwise.
  * bf16 state: the same plus one bf16 ulp (2^-8 relative) for the final
    rounding of the fp32 result.
  * every pool byte outside the written (slot, head) states: bit-identical.
"""
from __future__ import annotations

import numpy as np
import torch

import linear_attention_recurrent_gb300 as lar
import oracle

STATE_RTOL, STATE_ATOL = 1e-4, 1e-6
BF16_STATE_RTOL = 2.0 ** -8 + 1e-4
OUT_BF16_ATOL = 2e-3


def bf16_out_tol(ref: np.ndarray) -> np.ndarray:
    a = np.abs(ref)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(a, 1e-30))) - 8.0)
    return np.where(a < 1.0, OUT_BF16_ATOL, half_ulp + 1e-4 * a)


def assert_out_close(gpu: torch.Tensor, ref: np.ndarray, what="out"):
    g = gpu.detach().float().cpu().double().numpy()
    if g.shape != ref.shape and g.size == ref.size:   # rank-3 (T = 1) outputs
        ref = ref.reshape(g.shape)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    tol = bf16_out_tol(ref) if gpu.dtype == torch.bfloat16 else STATE_RTOL * np.abs(ref) + STATE_ATOL
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def assert_state_close(gpu: torch.Tensor, ref: np.ndarray, what="state"):
    g = gpu.detach().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    rtol = BF16_STATE_RTOL if gpu.dtype == torch.bfloat16 else STATE_RTOL
    bad = err > rtol * np.abs(ref) + STATE_ATOL
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"max err {err.max():.3e}")
    return float(err.max())


def storage(w):
    """The tensor that owns the pool's bytes (the backing buffer of a strided view)."""
    return w.backing if w.backing is not None else w.pool


def written_mask(w, write_idx=None) -> torch.Tensor:
    """Boolean mask over dim 0 of storage(w): the rows the decode may write."""
    wi = (write_idx if write_idx is not None else
          (w.write_idx if w.write_idx is not None else w.read_idx)).cpu().long()
    st = storage(w)
    mask = torch.zeros(st.shape[0], dtype=torch.bool)
    valid = wi[(wi >= 0) & (wi < w.P)]
    if st.dim() == 3:                       # flat [P*HV, V, K]
        for s in valid.tolist():
            mask[s * w.HV:(s + 1) * w.HV] = True
    else:
        mult = w.pool.stride(0) // w.backing.stride(0) if w.backing is not None else 1
        mask[valid * mult] = True
    return mask


def slot_state(pool: torch.Tensor, w, slot: int) -> torch.Tensor:
    """[HV, V, K] state of one slot of a (possibly flat) pool view."""
    if pool.dim() == 3:
        return pool[slot * w.HV:(slot + 1) * w.HV]
    return pool[slot]


def to_dev(t, dev):
    return None if t is None else t.to(dev)


def qkv_dev(w, dev):
    """w's q, k, v on the device.  Packed workloads stay packed there: the
    fused buffer is copied once and q, k, v are its head-dim slices, which is
    asserted on the device tensors themselves."""
    q, k, v = w.qkv_to(dev)
    if w.fused is not None:
        assert_packed_views(w, q, k, v)
    return q, k, v


def assert_packed_views(w, q, k, v):
    """q, k, v (device tensors) are head-dim slices of one fused buffer: the
    host views' strides and their element offsets K and 2K inside each row."""
    es = q.element_size()
    assert q.is_cuda and not q.is_contiguous()
    assert q.stride() == w.q.stride() == k.stride() and v.stride() == w.v.stride()
    assert q.stride()[-2] == 2 * w.K + w.V, q.stride()
    assert k.data_ptr() == q.data_ptr() + w.K * es
    assert v.data_ptr() == q.data_ptr() + 2 * w.K * es


def run_gpu(w, dev, *, pool=None, read_idx=None, write_idx="same", inter=True, dev_err=None,
            q=None, k=None, v=None):
    """Run w's decode on the GPU.  `pool` (a device view) is updated in place.
    Returns (out, inter)."""
    pool = pool if pool is not None else w.pool.to(dev)
    ri = to_dev(read_idx if read_idx is not None else w.read_idx, dev)
    wi = to_dev(w.write_idx if write_idx == "same" else write_idx, dev)
    if q is None and k is None and v is None:
        q, k, v = qkv_dev(w, dev)
    it = None
    if inter and w.cache_intermediate:
        shape = (w.B, w.T, w.HV, w.K, w.V) if w.state_kv else (w.B, w.T, w.HV, w.V, w.K)
        it = torch.full(shape, float("nan"), device=dev, dtype=w.inter_dtype)
    if w.form == "la":
        out = lar.la_decode(q, k, v, to_dev(w.decay, dev), pool, ri, wi, inter=it,
                            scale=w.scale, dev_err=dev_err, out_dtype=w.out_dtype)
    else:
        fn = lar.gdn_decode if w.form == "gdn" else lar.kda_decode
        out = fn(q, k, v, to_dev(w.g, dev), to_dev(w.beta, dev), pool, ri, wi, inter=it,
                 A_log=to_dev(w.A_log, dev), dt_bias=to_dev(w.dt_bias, dev), scale=w.scale,
                 qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw,
                 state_kv=w.state_kv, dev_err=dev_err, out_dtype=w.out_dtype)
    return out, it


def run_oracle(w, host_pool, *, read_idx=None, write_idx="same", batch=None):
    """Oracle on w (optionally on a subset `batch` of entries).  `host_pool`
    is a float32 CPU view updated in place."""
    sel = (lambda t: t) if batch is None else (lambda t: None if t is None else t[batch])
    ri = read_idx if read_idx is not None else w.read_idx
    wi = w.write_idx if write_idx == "same" else write_idx
    if w.form == "la":
        return oracle.la_decode(sel(w.q), sel(w.k), sel(w.v), w.decay, host_pool, sel(ri), sel(wi),
                                scale=w.scale, cache_intermediate=w.cache_intermediate)
    fn = oracle.gdn_decode if w.form == "gdn" else oracle.kda_decode
    return fn(sel(w.q), sel(w.k), sel(w.v), sel(w.g), sel(w.beta), host_pool, sel(ri), sel(wi),
              A_log=w.A_log, dt_bias=w.dt_bias, qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw,
              beta_raw=w.beta_raw, scale=w.scale, cache_intermediate=w.cache_intermediate,
              layout="kv" if w.state_kv else "vk")


def full_check(w, dev):
    """Whole-workload parity: out, intermediate states, written slots against
    the oracle; every other storage byte bit-identical.  Returns max errors."""
    st_host = storage(w)
    dev_storage = st_host.to(dev)
    before = dev_storage.clone()
    if w.backing is not None:
        mult = w.pool.stride(0) // w.backing.stride(0)
        pool_dev = dev_storage[::mult]
        host_view = st_host.clone()[::mult]
    else:
        pool_dev = dev_storage
        host_view = st_host.clone()
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, inter = run_gpu(w, dev, pool=pool_dev, dev_err=dev_err)
    torch.cuda.synchronize()
    ref = run_oracle(w, host_view)
    errs = {"out": assert_out_close(out, ref["out"])}
    # the oracle reports states as [v][k]; a [k][v] pool is compared through its transpose
    tr = (lambda x: x.transpose(-1, -2)) if w.state_kv else (lambda x: x)
    if inter is not None:
        errs["inter"] = assert_state_close(tr(inter), ref["inter"], "inter")
    mask = written_mask(w)
    assert torch.equal(dev_storage[~mask.to(dev)], before[~mask.to(dev)]), "untouched pool bytes changed"
    wi = (w.write_idx if w.write_idx is not None else w.read_idx).tolist()
    for b, s in enumerate(wi):
        if 0 <= s < w.P:
            errs["state"] = max(errs.get("state", 0.0),
                                assert_state_close(tr(slot_state(pool_dev, w, s)), ref["final_state"][b],
                                                   f"slot {s} (entry {b})"))
    assert int(dev_err.item()) == 0
    return errs


# --------------------------------------------------------------------------- variable-length spans

def run_gpu_varlen(w, dev, *, pool, cu_seqlens=None, dev_err=None, out_fill=float("nan")):
    """Run a make_varlen workload through *_decode_varlen.  out (and the state
    cache) start filled with `out_fill`, so untouched rows can be checked."""
    cu = to_dev(w.cu_seqlens if cu_seqlens is None else cu_seqlens, dev)
    ri, wi = to_dev(w.read_idx, dev), to_dev(w.write_idx, dev)
    out = torch.full(tuple(w.v.shape), out_fill, dtype=w.out_dtype, device=dev)
    it = None
    if w.cache_intermediate:
        it = torch.full((w.v.shape[0], w.HV, w.V, w.K), out_fill, device=dev, dtype=w.inter_dtype)
    q, k, v = qkv_dev(w, dev)
    if w.form == "la":
        lar.la_decode_varlen(q, k, v, to_dev(w.decay, dev), pool, cu, ri, wi, out=out, inter=it,
                             scale=w.scale, dev_err=dev_err)
    else:
        fn = lar.gdn_decode_varlen if w.form == "gdn" else lar.kda_decode_varlen
        fn(q, k, v, to_dev(w.g, dev), to_dev(w.beta, dev), pool, cu, ri, wi, out=out, inter=it,
           A_log=to_dev(w.A_log, dev), dt_bias=to_dev(w.dt_bias, dev), scale=w.scale,
           qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw, dev_err=dev_err)
    return out, it


def run_oracle_varlen(w, host_pool, cu_seqlens=None):
    cu = w.cu_seqlens if cu_seqlens is None else cu_seqlens
    if w.form == "la":
        return oracle.la_decode_varlen(w.q, w.k, w.v, w.decay, host_pool, cu, w.read_idx, w.write_idx,
                                       scale=w.scale, cache_intermediate=w.cache_intermediate)
    fn = oracle.gdn_decode_varlen if w.form == "gdn" else oracle.kda_decode_varlen
    return fn(w.q, w.k, w.v, w.g, w.beta, host_pool, cu, w.read_idx, w.write_idx, A_log=w.A_log,
              dt_bias=w.dt_bias, qk_l2norm=w.qk_l2norm, gate_raw=w.gate_raw, beta_raw=w.beta_raw,
              scale=w.scale, cache_intermediate=w.cache_intermediate)


def varlen_check(w, dev, *, cu_seqlens=None, expect_err=0):
    """Variable-length parity: the outputs and cached states of every token in
    a valid span against the oracle, rows of tokens outside every span left as
    allocated (NaN), written slots against the oracle's final states, every
    other pool byte bit-identical, and the device error word as expected."""
    st_host = storage(w)
    dev_storage = st_host.to(dev)
    before = dev_storage.clone()
    if w.backing is not None:
        mult = w.pool.stride(0) // w.backing.stride(0)
        pool_dev, host_view = dev_storage[::mult], st_host.clone()[::mult]
    else:
        pool_dev, host_view = dev_storage, st_host.clone()
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, inter = run_gpu_varlen(w, dev, pool=pool_dev, cu_seqlens=cu_seqlens, dev_err=dev_err)
    torch.cuda.synchronize()
    ref = run_oracle_varlen(w, host_view, cu_seqlens)
    covered = ~np.isnan(ref["out"]).all(axis=(1, 2))
    cov_t = torch.from_numpy(covered)
    errs = {}
    if covered.any():
        errs["out"] = assert_out_close(out[cov_t.to(dev)], ref["out"][covered])
        if inter is not None:
            errs["inter"] = assert_state_close(inter[cov_t.to(dev)], ref["inter"][covered], "inter")
    if (~covered).any():
        assert torch.isnan(out[(~cov_t).to(dev)].float()).all(), "output rows outside every span written"
        if inter is not None:
            assert torch.isnan(inter[(~cov_t).to(dev)].float()).all(), "cache rows outside every span written"
    mask = written_mask(w)
    assert torch.equal(dev_storage[~mask.to(dev)], before[~mask.to(dev)]), "untouched pool bytes changed"
    for n, s in enumerate(w.write_idx.tolist()):
        if 0 <= s < w.P:
            errs["state"] = max(errs.get("state", 0.0),
                                assert_state_close(slot_state(pool_dev, w, s), ref["final_state"][n],
                                                   f"slot {s} (sequence {n})"))
    assert int(dev_err.item()) == expect_err, int(dev_err.item())
    return errs
