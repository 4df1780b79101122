"""Plain fp64 CPU oracle for the recurrent linear-attention decode step.

TEST INFRASTRUCTURE ONLY: the library never imports this package.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use
it.  It shares no code with the CUDA path; the arithmetic lives in
``oracle.c`` (plain loops, fp64), which this module compiles with gcc on first
use and calls through ctypes.

Every input other than the pool is widened exactly to a contiguous fp64 array
(bf16 -> fp32 -> fp64 loses nothing).  The pool is a float32 CPU tensor (or
numpy array) or a bfloat16 CPU tensor, possibly a strided view of a larger
backing buffer, and is updated IN PLACE through its own strides (bf16 written
back rounded to nearest even straight from fp64), exactly as the writeback rule of
the flashinfer "fp32 sibling of #3268" page asks.

Functions return a dict with
  ``out``          fp64 [B,T,HV,V] (unrounded),
  ``final_state``  fp64 [B,HV,V,K] (the state after the last token, storage order),
  ``inter``        fp64 [B,T,HV,V,K] or None,
  ``n_bad``        number of slot indices >= the pool size that were seen.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
# tests that plant mistakes in a copy of oracle.c point this at the mutated build
_OVERRIDE = os.environ.get("LAR_ORACLE_LIB")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain -O2, no fast-math, no -march)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _OVERRIDE:
                lib = ctypes.CDLL(_OVERRIDE)
            else:
                build()
                lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            vp = ctypes.c_void_p
            for name in ("oracle_gdn_decode", "oracle_kda_decode"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_long
                fn.argtypes = [i64] * 6 + [dp] * 7 + [ctypes.c_int] * 3 + [
                    ctypes.c_double, vp, ctypes.c_int, i64, ip, ip, ip, dp, dp, dp]
            for name in ("oracle_gdn_decode_tokens", "oracle_kda_decode_tokens"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_long
                fn.argtypes = [i64] * 6 + [dp] * 7 + [ctypes.c_int] * 3 + [
                    ctypes.c_double, vp, ctypes.c_int, i64, ip, ip, ip, ip, dp, dp, dp]
            lib.oracle_la_decode.restype = ctypes.c_long
            lib.oracle_la_decode.argtypes = [i64] * 5 + [dp] * 4 + [
                ctypes.c_double, vp, ctypes.c_int, i64, ip, ip, ip, dp, dp, dp]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            _lib = lib
    return _lib


def _f64(x):
    """Exact widening of a torch tensor / numpy array to a contiguous fp64 array."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: bf16/fp16/fp32 -> fp64 is exact
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _pool_view(pool):
    """numpy view sharing memory with `pool` (writes land in it): float32, or
    the raw 16-bit patterns of a bfloat16 pool.  Returns (array, address,
    element strides, is_bf16)."""
    bf16 = False
    if hasattr(pool, "detach"):
        if pool.device.type != "cpu":
            raise TypeError("oracle pool must be a CPU tensor")
        if str(pool.dtype) == "torch.bfloat16":
            bf16 = True
            import torch
            arr = pool.detach().view(torch.int16).numpy()
        elif str(pool.dtype) == "torch.float32":
            arr = pool.detach().numpy()
        else:
            raise TypeError("oracle pool must be float32 or bfloat16")
    else:
        arr = pool
        if arr.dtype != np.float32:
            raise TypeError("oracle pool arrays must be float32")
    es = arr.dtype.itemsize
    if any(s % es for s in arr.strides):
        raise ValueError("pool strides must be whole elements")
    strides = np.array([s // es for s in arr.strides], dtype=np.int64)
    # address of the view's first element (numpy handles the offset)
    return arr, arr.__array_interface__["data"][0], strides, bf16


def round_bf16(x: float) -> int:
    """Bit pattern of the bfloat16 nearest to x (ties to even), as the oracle stores it."""
    return int(_load().oracle_round_bf16(float(x)))


def _as_btxk(x, name):
    """[B,H,K] means T = 1; [B,T,H,K] as is."""
    if x.ndim == 3:
        return x[:, None]
    if x.ndim != 4:
        raise ValueError(f"{name} must be [B,T,H,K] or [B,H,K]")
    return x


def _as_btx(x, name, ndim_full):
    if x.ndim == ndim_full - 1:
        return x[:, None]
    if x.ndim != ndim_full:
        raise ValueError(f"{name} has rank {x.ndim}")
    return x


def _delta(per_channel, q, k, v, g, beta, pool, read_idx, write_idx, A_log, dt_bias,
           qk_l2norm, gate_raw, beta_raw, scale, cache_intermediate, tokens=None, layout="vk"):
    lib = _load()
    q = _as_btxk(_f64(q), "q")
    k = _as_btxk(_f64(k), "k")
    v = _as_btxk(_f64(v), "v")
    g = _as_btx(_f64(g), "g", 4 if per_channel else 3)
    beta = _as_btx(_f64(beta), "beta", 3)
    q, k, v, g, beta = (np.ascontiguousarray(a) for a in (q, k, v, g, beta))
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if k.shape != q.shape or v.shape[:2] != (B, T):
        raise ValueError("q/k/v shapes disagree")
    arr, pptr, st, pbf = _pool_view(pool)
    if arr.ndim == 3:  # flat [P*HV, V, K]: one slot spans HV consecutive rows
        if arr.shape[0] % HV:
            raise ValueError("flat pool rows must be a multiple of HV")
        P = arr.shape[0] // HV
        st = np.array([st[0] * HV, st[0], st[1], st[2]], dtype=np.int64)
    elif arr.ndim == 4:
        P = arr.shape[0]
    else:
        raise ValueError("pool must be [P,HV,V,K] or [P*HV,V,K]")
    if layout == "kv":
        # the pool holds S itself ([.., k, v]): the element of S[k][v] is reached
        # with the row stride on k and the inner stride on v
        st = np.array([st[0], st[1], st[3], st[2]], dtype=np.int64)
    elif layout != "vk":
        raise ValueError("layout must be 'vk' or 'kv'")
    ri = _i64(read_idx)
    wi = _i64(write_idx)
    A = _f64(A_log)
    D = _f64(dt_bias)
    out = np.zeros((B, T, HV, V))
    fin = np.zeros((B, HV, V, K))
    inter = np.zeros((B, T, HV, V, K)) if cache_intermediate else None
    dp = ctypes.c_double
    if tokens is None:
        fn = lib.oracle_kda_decode if per_channel else lib.oracle_gdn_decode
        bad = fn(B, T, H, HV, K, V, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(g, dp),
                 _ptr(beta, dp), _ptr(A, dp), _ptr(D, dp), int(qk_l2norm), int(gate_raw),
                 int(beta_raw), float(scale), pptr, int(pbf), P, _ptr(st, ctypes.c_int64),
                 _ptr(ri, ctypes.c_int64), _ptr(wi, ctypes.c_int64), _ptr(out, dp),
                 _ptr(fin, dp), _ptr(inter, dp))
    else:
        na, sidx = _i64(tokens[0]), _i64(tokens[1])
        if sidx.shape != (B, T):
            raise ValueError("state_idx must be [B, T]")
        fn = lib.oracle_kda_decode_tokens if per_channel else lib.oracle_gdn_decode_tokens
        bad = fn(B, T, H, HV, K, V, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp), _ptr(g, dp),
                 _ptr(beta, dp), _ptr(A, dp), _ptr(D, dp), int(qk_l2norm), int(gate_raw),
                 int(beta_raw), float(scale), pptr, int(pbf), P, _ptr(st, ctypes.c_int64),
                 _ptr(ri, ctypes.c_int64), _ptr(na, ctypes.c_int64),
                 _ptr(np.ascontiguousarray(sidx), ctypes.c_int64), _ptr(out, dp), _ptr(fin, dp),
                 _ptr(inter, dp))
    if bad < 0:
        raise ValueError("oracle rejected its arguments")
    return {"out": out, "final_state": fin, "inter": inter, "n_bad": int(bad)}


def gdn_decode(q, k, v, g, beta, pool, read_idx, write_idx=None, *, A_log=None,
               dt_bias=None, qk_l2norm=False, gate_raw=False, beta_raw=False, scale=1.0,
               cache_intermediate=False, layout="vk"):
    """GDN: scalar log-decay g[b,t,hv]; see oracle.c for the recurrence.
    layout "vk": pool[p, hv, v, k] = S[k][v] (default); "kv": pool[p, hv, k, v] = S[k][v].
    Returned states are in the [v][k] order either way."""
    return _delta(False, q, k, v, g, beta, pool, read_idx, write_idx, A_log, dt_bias,
                  qk_l2norm, gate_raw, beta_raw, scale, cache_intermediate, layout=layout)


def kda_decode(q, k, v, g, beta, pool, read_idx, write_idx=None, *, A_log=None,
               dt_bias=None, qk_l2norm=False, gate_raw=False, beta_raw=False, scale=1.0,
               cache_intermediate=False, layout="vk"):
    """KDA: per-key-channel log-decay g[b,t,hv,k]; see oracle.c (layout as gdn_decode)."""
    return _delta(True, q, k, v, g, beta, pool, read_idx, write_idx, A_log, dt_bias,
                  qk_l2norm, gate_raw, beta_raw, scale, cache_intermediate, layout=layout)


def gdn_decode_tokens(q, k, v, g, beta, pool, state_idx, *, read_idx=None, num_accepted=None,
                      A_log=None, dt_bias=None, qk_l2norm=False, gate_raw=False, beta_raw=False,
                      scale=1.0, cache_intermediate=False):
    """GDN with per-token pool slots: the state after token t is written to slot
    state_idx[b, t]; the seed comes from state_idx[b, num_accepted[b] - 1] when
    num_accepted is given, else from read_idx[b]."""
    return _delta(False, q, k, v, g, beta, pool, read_idx, None, A_log, dt_bias, qk_l2norm,
                  gate_raw, beta_raw, scale, cache_intermediate, tokens=(num_accepted, state_idx))


def kda_decode_tokens(q, k, v, g, beta, pool, state_idx, *, read_idx=None, num_accepted=None,
                      A_log=None, dt_bias=None, qk_l2norm=False, gate_raw=False, beta_raw=False,
                      scale=1.0, cache_intermediate=False):
    """KDA with per-token pool slots (see gdn_decode_tokens)."""
    return _delta(True, q, k, v, g, beta, pool, read_idx, None, A_log, dt_bias, qk_l2norm,
                  gate_raw, beta_raw, scale, cache_intermediate, tokens=(num_accepted, state_idx))


def _varlen(run, per_token, cu_seqlens, pool, read_idx, write_idx, cache_intermediate, HV, V, K, ntok):
    """Variable-length spans: sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1
    and is run as a batch of one with T = its length (T = 0 copies the read
    state to the write slot).  `per_token` are the token-major inputs, sliced
    per sequence and given a batch axis.  A span that is reversed or runs past
    the token arrays is run as empty and counted in n_bad.  Outputs of tokens
    outside every span stay NaN."""
    cu = _i64(cu_seqlens)
    ri = _i64(read_idx)
    wi = None if write_idx is None else _i64(write_idx)
    N = cu.shape[0] - 1
    out = np.full((ntok, HV, V), np.nan)
    fin = np.zeros((N, HV, V, K))
    inter = np.full((ntok, HV, V, K), np.nan) if cache_intermediate else None
    bad = 0
    for n in range(N):
        lo, hi = int(cu[n]), int(cu[n + 1])
        if not 0 <= lo <= hi <= ntok:
            lo = hi = 0
            bad += 1
        part = [None if x is None else x[lo:hi][None] for x in per_token]
        res = run(*part, pool, ri[n:n + 1], None if wi is None else wi[n:n + 1])
        out[lo:hi] = res["out"][0]
        fin[n] = res["final_state"][0]
        if inter is not None:
            inter[lo:hi] = res["inter"][0]
        bad += res["n_bad"]
    return {"out": out, "final_state": fin, "inter": inter, "n_bad": bad}


def gdn_decode_varlen(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx=None, *, A_log=None,
                      dt_bias=None, qk_l2norm=False, gate_raw=False, beta_raw=False, scale=1.0,
                      cache_intermediate=False):
    """GDN over token-major variable-length spans: q, k [Ntok,H,K], v [Ntok,HV,V],
    g, beta [Ntok,HV]; out [Ntok,HV,V], final_state [N,HV,V,K], inter [Ntok,HV,V,K]."""
    run = lambda q_, k_, v_, g_, b_, pool_, r_, w_: gdn_decode(
        q_, k_, v_, g_, b_, pool_, r_, w_, A_log=A_log, dt_bias=dt_bias, qk_l2norm=qk_l2norm,
        gate_raw=gate_raw, beta_raw=beta_raw, scale=scale, cache_intermediate=cache_intermediate)
    return _varlen(run, (_f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)), cu_seqlens, pool, read_idx,
                   write_idx, cache_intermediate, v.shape[1], v.shape[2], q.shape[2], q.shape[0])


def kda_decode_varlen(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx=None, *, A_log=None,
                      dt_bias=None, qk_l2norm=False, gate_raw=False, beta_raw=False, scale=1.0,
                      cache_intermediate=False):
    """KDA over token-major variable-length spans (g [Ntok,HV,K]); see gdn_decode_varlen."""
    run = lambda q_, k_, v_, g_, b_, pool_, r_, w_: kda_decode(
        q_, k_, v_, g_, b_, pool_, r_, w_, A_log=A_log, dt_bias=dt_bias, qk_l2norm=qk_l2norm,
        gate_raw=gate_raw, beta_raw=beta_raw, scale=scale, cache_intermediate=cache_intermediate)
    return _varlen(run, (_f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)), cu_seqlens, pool, read_idx,
                   write_idx, cache_intermediate, v.shape[1], v.shape[2], q.shape[2], q.shape[0])


def la_decode_varlen(q, k, v, decay, pool, cu_seqlens, read_idx, write_idx=None, *, scale=1.0,
                     cache_intermediate=False):
    """Lightning Attention over token-major variable-length spans; see gdn_decode_varlen."""
    run = lambda q_, k_, v_, pool_, r_, w_: la_decode(q_, k_, v_, decay, pool_, r_, w_, scale=scale,
                                                      cache_intermediate=cache_intermediate)
    return _varlen(run, (_f64(q), _f64(k), _f64(v)), cu_seqlens, pool, read_idx, write_idx,
                   cache_intermediate, v.shape[1], v.shape[2], q.shape[2], q.shape[0])


def la_decode(q, k, v, decay, pool, read_idx, write_idx=None, *, scale=1.0,
              cache_intermediate=False):
    """Lightning Attention: S <- lambda_h S + k (x) v, o = S^T q; pool [P*H,V,K] or [P,H,V,K]."""
    lib = _load()
    q = np.ascontiguousarray(_as_btxk(_f64(q), "q"))
    k = np.ascontiguousarray(_as_btxk(_f64(k), "k"))
    v = np.ascontiguousarray(_as_btxk(_f64(v), "v"))
    lam = _f64(decay)
    B, T, H, K = q.shape
    V = v.shape[3]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or lam.shape != (H,):
        raise ValueError("q/k/v/decay shapes disagree")
    arr, pptr, st, pbf = _pool_view(pool)
    if arr.ndim == 4:  # [P,H,V,K] is only valid as a flat [P*H,V,K] view
        if st[0] != st[1] * H:
            raise ValueError("4D LA pool must have slot stride == H * head stride")
        rows = arr.shape[0] * H
        st = np.array([st[1], st[2], st[3]], dtype=np.int64)
    elif arr.ndim == 3:
        rows = arr.shape[0]
    else:
        raise ValueError("LA pool must be [P*H,V,K]")
    ri = _i64(read_idx)
    wi = _i64(write_idx)
    out = np.zeros((B, T, H, V))
    fin = np.zeros((B, H, V, K))
    inter = np.zeros((B, T, H, V, K)) if cache_intermediate else None
    dp = ctypes.c_double
    bad = lib.oracle_la_decode(B, T, H, K, V, _ptr(q, dp), _ptr(k, dp), _ptr(v, dp),
                               _ptr(lam, dp), float(scale), pptr, int(pbf), rows,
                               _ptr(st, ctypes.c_int64), _ptr(ri, ctypes.c_int64),
                               _ptr(wi, ctypes.c_int64), _ptr(out, dp), _ptr(fin, dp),
                               _ptr(inter, dp))
    if bad < 0:
        raise ValueError("oracle rejected its arguments")
    return {"out": out, "final_state": fin, "inter": inter, "n_bad": int(bad)}
