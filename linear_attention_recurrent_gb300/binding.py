"""ctypes binding over liblar.so: the same three calls as include/lar.h, taking
torch tensors.  Marshalling only -- every step of the decode runs in the CUDA
kernels behind the C ABI; there is no Python or CPU fallback.  A missing
library, a CPU tensor or a non-OK status raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

_LIB_PATH = _build.LIB

LAR_F32, LAR_BF16, LAR_I32, LAR_I64 = 0, 1, 2, 3
LAR_QK_L2NORM, LAR_GATE_RAW, LAR_BETA_RAW, LAR_STATE_KV = 1, 2, 4, 8
LAR_DEVERR_READ_SLOT, LAR_DEVERR_WRITE_SLOT, LAR_DEVERR_ACCEPTED, LAR_DEVERR_SEQLEN = 1, 2, 4, 8
LAR_DEVERR_TIMEOUT = 16

STATUS = {0: "LAR_OK", 1: "LAR_ERR_NULL", 2: "LAR_ERR_DTYPE", 3: "LAR_ERR_RANK",
          4: "LAR_ERR_SHAPE", 5: "LAR_ERR_STRIDE", 6: "LAR_ERR_ALIGN", 7: "LAR_ERR_ARG",
          8: "LAR_ERR_ALIAS", 9: "LAR_ERR_LAUNCH"}

_DT = {torch.float32: LAR_F32, torch.bfloat16: LAR_BF16, torch.int32: LAR_I32,
       torch.int64: LAR_I64}


class LarTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5), ("stride", ctypes.c_int64 * 5)]


class LarError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({msg})")
        self.status = status


_lib = None


def library_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load liblar.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(LarTensor)
        tail = [ctypes.c_float, ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
        for name in ("gdn_decode", "kda_decode"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [P] * 12 + tail
        for name in ("gdn_decode_tokens", "kda_decode_tokens"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [P] * 12 + tail
        lib.la_decode.restype = ctypes.c_int
        lib.la_decode.argtypes = [P] * 9 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        for name in ("gdn_decode_varlen", "kda_decode_varlen"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [P] * 13 + tail
        lib.la_decode_varlen.restype = ctypes.c_int
        lib.la_decode_varlen.argtypes = [P] * 10 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        for name in ("gdn_prefill", "kda_prefill"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [P] * 12 + tail
        lib.la_prefill.restype = ctypes.c_int
        lib.la_prefill.argtypes = [P] * 9 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
        lib.lar_status_string.restype = ctypes.c_char_p
        lib.lar_status_string.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def describe(t: torch.Tensor | None):
    """lar_tensor descriptor of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("liblar works on CUDA tensors only")
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    if t.dim() < 1 or t.dim() > 5:
        raise ValueError(f"unsupported rank {t.dim()}")
    d = LarTensor()
    d.data = t.data_ptr()
    d.dtype = _DT[t.dtype]
    d.ndim = t.dim()
    for i, (s, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = s
        d.stride[i] = st
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _device_of(tensors, dev_err=None, stream=None) -> torch.device:
    """The one CUDA device every tensor of a call (and dev_err, and a torch
    stream when given) lives on; mixed devices are rejected before anything is
    launched (a kernel reading another GPU's memory without peer access would
    fault)."""
    ts = [t for t in tensors if t is not None] + ([dev_err] if dev_err is not None else [])
    devs = {t.device for t in ts}
    if len(devs) != 1:
        raise ValueError(f"the tensors of one call must share one CUDA device, got {sorted(map(str, devs))}")
    dev = devs.pop()
    if dev.type != "cuda":
        raise ValueError("liblar works on CUDA tensors only")
    if dev_err is not None and (dev_err.dtype != torch.int32 or dev_err.numel() < 1):
        raise ValueError("dev_err must be a CUDA int32 tensor of at least one element")
    sdev = getattr(stream, "device", None)
    if sdev is not None and torch.device(sdev) != dev:
        raise ValueError(f"stream is on {sdev}, the tensors on {dev}")
    return dev


def _stream(stream, dev=None):
    if stream is None:
        return torch.cuda.current_stream(dev).cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn, status):
    if status != 0:
        raise LarError(fn, status, load().lar_status_string(status).decode())


def _flags(qk_l2norm, gate_raw, beta_raw, state_kv=False):
    return (LAR_QK_L2NORM if qk_l2norm else 0) | (LAR_GATE_RAW if gate_raw else 0) | \
        (LAR_BETA_RAW if beta_raw else 0) | (LAR_STATE_KV if state_kv else 0)


def gdn_decode(q, k, v, g, beta, pool, read_idx, write_idx=None, *, out=None, inter=None,
               A_log=None, dt_bias=None, scale=1.0, qk_l2norm=False, gate_raw=False,
               beta_raw=False, state_kv=False, dev_err=None, out_dtype=None, stream=None):
    """Gated delta rule decode (scalar decay).  Updates `pool` in place; returns `out`.
    state_kv: the pool (and inter) hold S as [k][v], v fastest."""
    return _delta("gdn_decode", q, k, v, g, beta, pool, read_idx, write_idx, out, inter, A_log,
                  dt_bias, scale, _flags(qk_l2norm, gate_raw, beta_raw, state_kv), dev_err,
                  out_dtype, stream)


def kda_decode(q, k, v, g, beta, pool, read_idx, write_idx=None, *, out=None, inter=None,
               A_log=None, dt_bias=None, scale=1.0, qk_l2norm=False, gate_raw=False,
               beta_raw=False, state_kv=False, dev_err=None, out_dtype=None, stream=None):
    """Gated delta rule decode (per-key-channel decay).  Updates `pool` in place."""
    return _delta("kda_decode", q, k, v, g, beta, pool, read_idx, write_idx, out, inter, A_log,
                  dt_bias, scale, _flags(qk_l2norm, gate_raw, beta_raw, state_kv), dev_err,
                  out_dtype, stream)


def _delta(name, q, k, v, g, beta, pool, read_idx, write_idx, out, inter, A_log, dt_bias, scale,
           flags, dev_err, out_dtype, stream):
    lib = load()
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    ts = (q, k, v, g, beta, A_log, dt_bias, pool, read_idx, write_idx, out, inter)
    dev = _device_of(ts, dev_err, stream)
    ds = [describe(t) for t in ts]
    err = dev_err.data_ptr() if dev_err is not None else None
    with torch.cuda.device(dev):
        st = getattr(lib, name)(*[_ref(d) for d in ds], float(scale), flags, err, _stream(stream, dev))
    _check(name, st)
    return out


def gdn_decode_tokens(q, k, v, g, beta, pool, state_idx, *, read_idx=None, num_accepted=None,
                      out=None, A_log=None, dt_bias=None, scale=1.0, qk_l2norm=False,
                      gate_raw=False, beta_raw=False, dev_err=None, out_dtype=None, stream=None):
    """GDN with per-token pool slots: the state after token t goes to slot
    state_idx[b, t]; the seed is slot state_idx[b, num_accepted[b] - 1] (or
    read_idx[b] when num_accepted is None)."""
    return _tokens("gdn_decode_tokens", q, k, v, g, beta, pool, state_idx, read_idx, num_accepted,
                   out, A_log, dt_bias, scale, _flags(qk_l2norm, gate_raw, beta_raw), dev_err,
                   out_dtype, stream)


def kda_decode_tokens(q, k, v, g, beta, pool, state_idx, *, read_idx=None, num_accepted=None,
                      out=None, A_log=None, dt_bias=None, scale=1.0, qk_l2norm=False,
                      gate_raw=False, beta_raw=False, dev_err=None, out_dtype=None, stream=None):
    """KDA with per-token pool slots (see gdn_decode_tokens)."""
    return _tokens("kda_decode_tokens", q, k, v, g, beta, pool, state_idx, read_idx, num_accepted,
                   out, A_log, dt_bias, scale, _flags(qk_l2norm, gate_raw, beta_raw), dev_err,
                   out_dtype, stream)


def _tokens(name, q, k, v, g, beta, pool, state_idx, read_idx, num_accepted, out, A_log, dt_bias,
            scale, flags, dev_err, out_dtype, stream):
    lib = load()
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    ts = (q, k, v, g, beta, A_log, dt_bias, pool, read_idx, num_accepted, state_idx, out)
    dev = _device_of(ts, dev_err, stream)
    ds = [describe(t) for t in ts]
    err = dev_err.data_ptr() if dev_err is not None else None
    with torch.cuda.device(dev):
        st = getattr(lib, name)(*[_ref(d) for d in ds], float(scale), flags, err, _stream(stream, dev))
    _check(name, st)
    return out


def la_decode(q, k, v, decay, pool, read_idx, write_idx=None, *, out=None, inter=None, scale=1.0,
              dev_err=None, out_dtype=None, stream=None):
    """Lightning-Attention decode.  Updates `pool` in place; returns `out`."""
    lib = load()
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    ts = (q, k, v, decay, pool, read_idx, write_idx, out, inter)
    dev = _device_of(ts, dev_err, stream)
    ds = [describe(t) for t in ts]
    err = dev_err.data_ptr() if dev_err is not None else None
    with torch.cuda.device(dev):
        st = lib.la_decode(*[_ref(d) for d in ds], float(scale), err, _stream(stream, dev))
    _check("la_decode", st)
    return out


def gdn_decode_varlen(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx=None, *, out=None,
                      inter=None, A_log=None, dt_bias=None, scale=1.0, qk_l2norm=False, gate_raw=False,
                      beta_raw=False, dev_err=None, out_dtype=None, stream=None):
    """GDN over variable-length spans: q, k [Ntok, H, K], v [Ntok, HV, V], g and
    beta [Ntok, HV]; sequence n owns tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.
    Returns out [Ntok, HV, V] (tokens outside every span are left as allocated)."""
    return _varlen("gdn_decode_varlen", q, k, v, (g, beta, A_log, dt_bias), pool, cu_seqlens, read_idx,
                   write_idx, out, inter, scale, _flags(qk_l2norm, gate_raw, beta_raw), dev_err, out_dtype,
                   stream)


def kda_decode_varlen(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx=None, *, out=None,
                      inter=None, A_log=None, dt_bias=None, scale=1.0, qk_l2norm=False, gate_raw=False,
                      beta_raw=False, dev_err=None, out_dtype=None, stream=None):
    """KDA over variable-length spans (g [Ntok, HV, K]); see gdn_decode_varlen."""
    return _varlen("kda_decode_varlen", q, k, v, (g, beta, A_log, dt_bias), pool, cu_seqlens, read_idx,
                   write_idx, out, inter, scale, _flags(qk_l2norm, gate_raw, beta_raw), dev_err, out_dtype,
                   stream)


def la_decode_varlen(q, k, v, decay, pool, cu_seqlens, read_idx, write_idx=None, *, out=None, inter=None,
                     scale=1.0, dev_err=None, out_dtype=None, stream=None):
    """Lightning Attention over variable-length spans; see gdn_decode_varlen."""
    return _varlen("la_decode_varlen", q, k, v, (decay,), pool, cu_seqlens, read_idx, write_idx, out, inter,
                   scale, None, dev_err, out_dtype, stream)


def gdn_prefill(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx=None, *, out=None, A_log=None,
                dt_bias=None, scale=1.0, qk_l2norm=False, gate_raw=False, beta_raw=False, dev_err=None,
                out_dtype=None, stream=None):
    """Chunked GDN prefill over variable-length spans (K = V = 128): the
    arguments and results of gdn_decode_varlen, without a state cache."""
    return _varlen("gdn_prefill", q, k, v, (g, beta, A_log, dt_bias), pool, cu_seqlens, read_idx, write_idx, out,
                   _NO_CACHE, scale, _flags(qk_l2norm, gate_raw, beta_raw), dev_err, out_dtype, stream)


def kda_prefill(q, k, v, g, beta, pool, cu_seqlens, read_idx, write_idx=None, *, out=None, A_log=None,
                dt_bias=None, scale=1.0, qk_l2norm=False, gate_raw=False, beta_raw=False, dev_err=None,
                out_dtype=None, stream=None):
    """Chunked KDA prefill over variable-length spans (K = V = 128): the
    arguments and results of kda_decode_varlen (g [Ntok, HV, K]), without a
    state cache."""
    return _varlen("kda_prefill", q, k, v, (g, beta, A_log, dt_bias), pool, cu_seqlens, read_idx, write_idx, out,
                   _NO_CACHE, scale, _flags(qk_l2norm, gate_raw, beta_raw), dev_err, out_dtype, stream)


def la_prefill(q, k, v, decay, pool, cu_seqlens, read_idx, write_idx=None, *, out=None, scale=1.0,
               dev_err=None, out_dtype=None, stream=None):
    """Chunked Lightning-Attention prefill over variable-length spans (K = V = 128)."""
    return _varlen("la_prefill", q, k, v, (decay,), pool, cu_seqlens, read_idx, write_idx, out, _NO_CACHE,
                   scale, None, dev_err, out_dtype, stream)


_NO_CACHE = object()   # the prefill calls take no state-cache argument


def _varlen(name, q, k, v, gates, pool, cu_seqlens, read_idx, write_idx, out, inter, scale, flags, dev_err,
            out_dtype, stream):
    lib = load()
    if out is None:
        out = torch.empty(v.shape, dtype=out_dtype or v.dtype, device=v.device)
    tail_t = () if inter is _NO_CACHE else (inter,)
    ts = (q, k, v) + tuple(gates) + (pool, cu_seqlens, read_idx, write_idx, out) + tail_t
    dev = _device_of(ts, dev_err, stream)
    ds = [describe(t) for t in ts]
    err = dev_err.data_ptr() if dev_err is not None else None
    tail = [float(scale)] + ([] if flags is None else [flags]) + [err, _stream(stream, dev)]
    with torch.cuda.device(dev):
        st = getattr(lib, name)(*[_ref(d) for d in ds], *tail)
    _check(name, st)
    return out


class PreparedCall:
    """A decode call whose descriptors are built once, for tight launch loops.
    The tensors it was built from must stay alive and keep their storage.
    Passing ``state_idx`` (and ``num_accepted`` or ``read_idx``) selects the
    per-token-slot call (gdn_decode_tokens / kda_decode_tokens); passing
    ``cu_seqlens`` selects the variable-length call (*_decode_varlen), and with
    ``prefill=True`` the chunked prefill call (gdn_prefill / la_prefill)."""

    def __init__(self, form, *, scale=1.0, qk_l2norm=False, gate_raw=False, beta_raw=False,
                 state_kv=False, dev_err=None, stream=None, prefill=False, **tensors):
        lib = load()
        tokens = tensors.get("state_idx") is not None
        varlen = tensors.get("cu_seqlens") is not None
        if prefill and (not varlen or tensors.get("inter") is not None):
            raise ValueError("the prefill call takes cu_seqlens and no state cache")
        if prefill:
            self._name = f"{form}_prefill"
        else:
            self._name = f"{form}_decode_varlen" if varlen else (f"{form}_decode_tokens" if tokens else f"{form}_decode")
        self._fn = getattr(lib, self._name)
        self._keep = (tensors, dev_err)
        self._dev = _device_of(tensors.values(), dev_err, stream)
        err = dev_err.data_ptr() if dev_err is not None else None
        st = _stream(stream, self._dev)
        if form == "la":
            names = ("q", "k", "v", "decay", "pool") + (("cu_seqlens",) if varlen else ()) + \
                ("read_idx", "write_idx", "out") + (() if prefill else ("inter",))
            self._descs = [describe(tensors.get(n)) for n in names]
            self._args = [_ref(d) for d in self._descs] + [float(scale), err, st]
        elif varlen:
            names = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool", "cu_seqlens", "read_idx",
                     "write_idx", "out") + (() if prefill else ("inter",))
            self._descs = [describe(tensors.get(n)) for n in names]
            # a state_kv flag is passed on, for the library to reject
            self._args = [_ref(d) for d in self._descs] + [
                float(scale), _flags(qk_l2norm, gate_raw, beta_raw, state_kv), err, st]
        else:
            if tokens:
                names = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool", "read_idx",
                         "num_accepted", "state_idx", "out")
            else:
                names = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool", "read_idx",
                         "write_idx", "out", "inter")
            self._descs = [describe(tensors.get(n)) for n in names]
            self._args = [_ref(d) for d in self._descs] + [
                float(scale), _flags(qk_l2norm, gate_raw, beta_raw, state_kv), err, st]

    def __call__(self):
        if torch.cuda.current_device() == self._dev.index:
            st = self._fn(*self._args)
        else:
            with torch.cuda.device(self._dev):
                st = self._fn(*self._args)
        if st != 0:
            _check(self._name, st)


class StepGraph:
    """One serving step captured once as a CUDA graph and replayed with one
    launch: the copies of the step's inputs to the device (``copies_in``, pairs
    ``(device_dst, src)``), a ``PreparedCall`` built on ``stream``, and the
    copies of its results back (``copies_out``, pairs ``(dst, device_src)``).
    Replays reuse the captured storage: the caller refills the source buffers
    (pinned host memory for asynchronous copies) between replays and keeps every
    tensor alive.  ``stream`` must not be the default stream (a capture needs
    its own).  ``warmup`` eager runs of the step come first, so that the call's
    one-time setup (the library's attribute and occupancy caches) happens
    outside the capture."""

    def __init__(self, call: PreparedCall, *, copies_in=(), copies_out=(), stream: torch.cuda.Stream,
                 warmup: int = 1):
        if stream is None or stream == torch.cuda.default_stream(stream.device):
            raise ValueError("StepGraph needs a non-default stream")
        self._call, self._in, self._out, self._stream = call, list(copies_in), list(copies_out), stream
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                self._body()
        stream.synchronize()
        self._graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self._graph, stream=stream, capture_error_mode="thread_local"):
            self._body()

    def _body(self):
        for dst, src in self._in:
            dst.copy_(src, non_blocking=True)
        self._call()
        for dst, src in self._out:
            dst.copy_(src, non_blocking=True)

    def replay(self):
        """Launch the step on its stream (asynchronous: synchronize the stream
        before reading host-side results)."""
        with torch.cuda.stream(self._stream):
            self._graph.replay()
