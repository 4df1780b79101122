"""The C ABI without a GPU: liblar.so loads, exports every function include/lar.h
declares, and rejects invalid arguments on the host with the documented status
before anything is launched.  Descriptors here carry fake (never dereferenced)
addresses; every call below fails validation, so no CUDA call is made."""
import ctypes
import os
import re

import pytest

from linear_attention_recurrent_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lar.h")

OK, NULL, DTYPE, RANK, SHAPE, STRIDE, ALIGN, ARG, ALIAS = range(9)
F32, BF16, I32, I64 = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, re.M)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("gdn_decode", "kda_decode", "la_decode", "lar_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(10):
        assert lib.lar_status_string(s)
    assert lib.lar_status_string(0) == b"ok"


_next_addr = [0x10000000]


def fake(shape, dtype=F32, strides=None, addr=None):
    d = binding.LarTensor()
    es = {F32: 4, BF16: 2, I32: 4, I64: 8}[dtype]
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    n = 1 + sum((s - 1) * st for s, st in zip(shape, strides))
    if addr is None:
        addr = _next_addr[0]
        _next_addr[0] += ((n * es + 4095) // 4096 + 1) * 4096
    d.data = addr
    d.dtype = dtype
    d.ndim = len(shape)
    for i, (s, st) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = st
    return d


def gdn_args(B=2, T=1, H=2, HV=4, K=128, V=64, P=8, kda=False):
    a = dict(q=fake([B, T, H, K], BF16), k=fake([B, T, H, K], BF16), v=fake([B, T, HV, V], BF16),
             g=fake([B, T, HV, K] if kda else [B, T, HV]), beta=fake([B, T, HV]),
             A_log=None, dt_bias=None, pool=fake([P, HV, V, K]), read_idx=fake([B], I32),
             write_idx=fake([B], I32), out=fake([B, T, HV, V], BF16), inter=None)
    return a


ORDER = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool", "read_idx", "write_idx", "out",
         "inter")


def call(lib, a, flags=0, kda=False):
    fn = lib.kda_decode if kda else lib.gdn_decode
    refs = [ctypes.byref(a[n]) if a[n] is not None else None for n in ORDER]
    return fn(*refs, 1.0, flags, None, None)


def test_empty_batch_is_a_no_op(lib):
    assert call(lib, gdn_args(B=0)) == OK


@pytest.mark.parametrize("mutate,flags,expect", [
    (lambda a: a.update(q=None), 0, NULL),
    (lambda a: a.update(pool=None), 0, NULL),
    (lambda a: a.update(g=None), 0, NULL),
    (lambda a: setattr(a["q"], "ndim", 6), 0, RANK),
    (lambda a: a.update(q=fake([2, 1, 2, 100], BF16), k=fake([2, 1, 2, 100], BF16)), 0, SHAPE),
    (lambda a: a.update(v=fake([2, 1, 3, 64], BF16), out=fake([2, 1, 3, 64], BF16)), 0, SHAPE),
    (lambda a: a.update(pool=fake([8, 4, 64, 128], I32)), 0, DTYPE),
    # a bf16 pool whose rows start 8 bytes apart cannot move in 16-byte chunks
    (lambda a: a.update(pool=fake([8, 4, 64, 128], BF16, strides=[4 * 64 * 132, 64 * 132, 132, 1])), 0, ALIGN),
    (lambda a: a.update(inter=fake([2, 1, 4, 64, 128], I32)), 0, DTYPE),
    (lambda a: a.update(q=fake([2, 1, 2, 128], I32)), 0, DTYPE),
    (lambda a: a.update(pool=fake([8, 4, 64, 128], strides=[64 * 256 * 4, 64 * 256, 256, 2])), 0, STRIDE),
    (lambda a: a.update(pool=fake([8, 4, 64, 128], addr=0x7000004)), 0, ALIGN),
    (lambda a: a.update(pool=fake([8, 4, 64, 128], strides=[4 * 64 * 130, 64 * 130, 130, 1])), 0, ALIGN),
    (lambda a: a.update(A_log=fake([4])), 0, ARG),                  # gate params without the flag
    (lambda a: a.update(dt_bias=fake([4])), 0, ARG),
    (lambda a: None, 2, NULL),                                        # LAR_GATE_RAW without A_log
    (lambda a: a.update(A_log=fake([3])), 2, SHAPE),
    (lambda a: None, 16, ARG),                                        # unknown flag bit
    (lambda a: a.update(read_idx=fake([3], I32)), 0, SHAPE),
    (lambda a: a.update(read_idx=fake([2], F32)), 0, DTYPE),
    (lambda a: a.update(write_idx=fake([2, 1], I32)), 0, RANK),
    (lambda a: a.update(inter=fake([2, 1, 4, 64, 64])), 0, SHAPE),
    (lambda a: a.update(inter=fake([2, 1, 4, 64, 128], strides=[1, 1, 1, 1, 2])), 0, STRIDE),
    (lambda a: a.update(out=fake([2, 1, 4, 64], F32, addr=a["pool"].data)), 0, ALIAS),
    (lambda a: a.update(out=fake([2, 1, 4, 64], BF16, addr=a["v"].data)), 0, ALIAS),
])
def test_gdn_rejects_on_host(lib, mutate, flags, expect):
    a = gdn_args()
    mutate(a)
    assert call(lib, a, flags) == expect


def test_multi_token_limit(lib):
    assert call(lib, gdn_args(T=17)) == SHAPE


def test_kda_gate_shape(lib):
    a = gdn_args(kda=True)
    a["g"] = fake([2, 1, 4])                                          # GDN-shaped gate
    assert call(lib, a, kda=True) == SHAPE
    a = gdn_args(kda=True)
    a["A_log"], a["dt_bias"] = fake([4]), fake([4])                   # dt_bias must be [HV*K]
    assert call(lib, a, flags=2, kda=True) == SHAPE


def la_call(lib, B=2, H=4, K=128, V=128, P=5, pool=None, decay=None):
    q, k, v = fake([B, H, K], BF16), fake([B, H, K], BF16), fake([B, H, V], BF16)
    pool = pool or fake([P * H, V, K])
    decay = decay or fake([H])
    ri, out = fake([B], I64), fake([B, H, V], BF16)
    refs = [ctypes.byref(x) for x in (q, k, v, decay, pool, ri)] + [None, ctypes.byref(out), None]
    return lib.la_decode(*refs, 1.0, None, None)


def test_la_rejects_on_host(lib):
    assert la_call(lib, pool=fake([4 * 5 + 1, 128, 128])) == SHAPE   # rows not a multiple of H
    assert la_call(lib, decay=fake([3])) == SHAPE
    assert la_call(lib, decay=fake([4], BF16)) == DTYPE
    # 4D pool whose slot stride is not H * head stride cannot be the flat layout
    assert la_call(lib, pool=fake([5, 4, 128, 128], strides=[8 * 128 * 128, 128 * 128, 128, 1])) == STRIDE
    assert la_call(lib, B=0) == OK


def tok_call(lib, a, state_idx, read_idx="default", num_accepted=None):
    ri = a["read_idx"] if read_idx == "default" else read_idx
    args = [a[n] for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool")] + [ri, num_accepted,
                                                                                         state_idx, a["out"]]
    refs = [ctypes.byref(x) if x is not None else None for x in args]
    return lib.gdn_decode_tokens(*refs, 1.0, 0, None, None)


def test_token_slots_rejects_on_host(lib):
    a = gdn_args(B=2, T=3)
    good = fake([2, 3], I32)
    assert tok_call(lib, a, None) == NULL
    assert tok_call(lib, a, fake([6], I32)) == RANK                   # flat table: rejected, not guessed
    assert tok_call(lib, a, fake([2, 4], I32)) == SHAPE
    assert tok_call(lib, a, fake([2, 3], F32)) == DTYPE
    assert tok_call(lib, a, good, read_idx=None) == ARG               # no seed source
    assert tok_call(lib, a, good, num_accepted=fake([2], I32)) == ARG  # two seed sources
    assert tok_call(lib, a, good, read_idx=None, num_accepted=fake([3], I32)) == SHAPE
    assert tok_call(lib, gdn_args(B=0, T=3), fake([0, 3], I32)) == OK


def test_kv_layout_validation(lib):
    KV = 8
    a = gdn_args(B=2, T=1, H=2, HV=4, K=128, V=64)
    a["pool"] = fake([8, 4, 64, 128])                                 # [P,HV,V,K] is not [P,HV,K,V]
    assert call(lib, a, KV) == SHAPE
    a = gdn_args(B=2, T=1, H=2, HV=4, K=128, V=66)
    a["pool"] = fake([8, 4, 128, 66])                                 # 66 fp32 rows: not 16-byte chunks
    assert call(lib, a, KV) == SHAPE
    a = gdn_args(B=2, T=1, H=2, HV=4, K=128, V=64)
    a["pool"] = fake([8, 4, 128, 64], strides=[4 * 128 * 64, 128 * 64, 1, 128])   # v not contiguous
    assert call(lib, a, KV) == STRIDE
    # per-token slots are served for the [v][k] layout only
    a = gdn_args(B=2, T=3)
    a["pool"] = fake([8, 4, 128, 64])
    refs = [ctypes.byref(x) if x is not None else None for x in
            [a[n] for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool")] + [a["read_idx"], None,
                                                                                       fake([2, 3], I32), a["out"]]]
    assert lib.gdn_decode_tokens(*refs, 1.0, KV, None, None) == ARG


def varlen_args(NT=10, N=3, H=2, HV=4, K=128, V=64, P=8, kda=False):
    return dict(q=fake([NT, H, K], BF16), k=fake([NT, H, K], BF16), v=fake([NT, HV, V], BF16),
                g=fake([NT, HV, K] if kda else [NT, HV]), beta=fake([NT, HV]), A_log=None, dt_bias=None,
                pool=fake([P, HV, V, K]), cu_seqlens=fake([N + 1], I32), read_idx=fake([N], I32),
                write_idx=fake([N], I32), out=fake([NT, HV, V], BF16), inter=None)


VARLEN_ORDER = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool", "cu_seqlens", "read_idx",
                "write_idx", "out", "inter")


def varlen_call(lib, a, flags=0, kda=False):
    fn = lib.kda_decode_varlen if kda else lib.gdn_decode_varlen
    refs = [ctypes.byref(a[n]) if a[n] is not None else None for n in VARLEN_ORDER]
    return fn(*refs, 1.0, flags, None, None)


def test_varlen_no_sequences_is_a_no_op(lib):
    assert varlen_call(lib, varlen_args(N=0)) == OK


@pytest.mark.parametrize("mutate,flags,expect", [
    (lambda a: a.update(cu_seqlens=None), 0, NULL),
    (lambda a: a.update(q=fake([2, 10, 2, 128], BF16)), 0, RANK),          # batched shapes are not varlen
    (lambda a: a.update(cu_seqlens=fake([4], F32)), 0, DTYPE),
    (lambda a: a.update(cu_seqlens=fake([4, 1], I32)), 0, RANK),
    (lambda a: a.update(read_idx=fake([4], I32)), 0, SHAPE),              # N + 1 offsets, N slots
    (lambda a: a.update(out=fake([9, 4, 64], BF16)), 0, SHAPE),
    (lambda a: a.update(g=fake([10, 4, 128])), 0, RANK),                  # KDA-shaped gate on GDN
    (lambda a: a.update(beta=fake([10, 3])), 0, SHAPE),
    (lambda a: a.update(inter=fake([10, 4, 64, 128, 1])), 0, RANK),
    (lambda a: a.update(inter=fake([3, 4, 64, 128])), 0, SHAPE),          # per token, not per sequence
    (lambda a: a.update(out=fake([10, 4, 64], F32, addr=a["pool"].data)), 0, ALIAS),
    (lambda a: None, 8, ARG),                                             # no K x V layout here
    (lambda a: None, 2, NULL),                                            # raw gates without A_log
])
def test_varlen_rejects_on_host(lib, mutate, flags, expect):
    a = varlen_args()
    mutate(a)
    assert varlen_call(lib, a, flags) == expect


def test_varlen_kda_and_la_shapes(lib):
    a = varlen_args(kda=True)
    a["g"] = fake([10, 4])
    assert varlen_call(lib, a, kda=True) == RANK
    q, k, v = fake([10, 4, 128], BF16), fake([10, 4, 128], BF16), fake([10, 4, 128], BF16)
    pool, decay, cu, ri, out = fake([5 * 4, 128, 128]), fake([4]), fake([3], I64), fake([2], I64), fake([10, 4, 128], BF16)
    la = lambda decay: lib.la_decode_varlen(*[ctypes.byref(x) for x in (q, k, v, decay, pool, cu, ri)], None,
                                            ctypes.byref(out), None, 1.0, None, None)
    assert la(fake([3])) == SHAPE
    assert la(fake([4], BF16)) == DTYPE
    cu0, ri0 = fake([1], I64), fake([0], I64)
    assert lib.la_decode_varlen(*[ctypes.byref(x) for x in (q, k, v, decay, pool, cu0, ri0)], None,
                                ctypes.byref(out), None, 1.0, None, None) == OK


PREFILL_ORDER = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool", "cu_seqlens", "read_idx",
                 "write_idx", "out")


def prefill_call(lib, a, flags=0):
    refs = [ctypes.byref(a[n]) if a[n] is not None else None for n in PREFILL_ORDER]
    return lib.gdn_prefill(*refs, 1.0, flags, None, None)


def test_kda_prefill_rejects_on_host(lib):
    def kda(a, flags=0):
        refs = [ctypes.byref(a[n]) if a[n] is not None else None for n in PREFILL_ORDER]
        return lib.kda_prefill(*refs, 1.0, flags, None, None)
    assert kda(varlen_args(N=0, V=128, kda=True)) == OK
    assert kda(varlen_args(K=64, V=64, kda=True)) == SHAPE           # built for K = V = 128
    assert kda(varlen_args(V=128)) == RANK                            # GDN-shaped gate [Ntok, HV]
    a = varlen_args(V=128, kda=True)
    a["A_log"], a["dt_bias"] = fake([4]), fake([4])                  # dt_bias must be [HV*K]
    assert kda(a, flags=2) == SHAPE
    assert kda(varlen_args(V=128, kda=True), flags=8) == ARG         # no K x V layout


def test_prefill_rejects_on_host(lib):
    assert prefill_call(lib, varlen_args(N=0, V=128)) == OK                # no sequences: nothing to do
    assert prefill_call(lib, varlen_args(K=64, V=64)) == SHAPE             # built for K = V = 128
    assert prefill_call(lib, varlen_args(K=128, V=64)) == SHAPE
    assert prefill_call(lib, varlen_args(V=128), flags=8) == ARG           # no K x V layout
    a = varlen_args(V=128)
    a["cu_seqlens"] = None
    assert prefill_call(lib, a) == NULL
    q, k, v = fake([10, 4, 128], BF16), fake([10, 4, 128], BF16), fake([10, 4, 128], BF16)
    pool, cu, ri, out = fake([5 * 4, 128, 128]), fake([3], I64), fake([2], I64), fake([10, 4, 128], BF16)
    la = lambda decay: lib.la_prefill(*[ctypes.byref(x) for x in (q, k, v, decay, pool, cu, ri)], None,
                                      ctypes.byref(out), 1.0, None, None)
    assert la(fake([3])) == SHAPE
    assert la(fake([4], BF16)) == DTYPE


def _err_word(addr):
    return ctypes.cast(ctypes.c_void_p(addr), ctypes.POINTER(ctypes.c_int32))


def test_dev_err_alignment_and_aliasing(lib):
    """The device error word is a 4-byte output: misaligned -> ALIGN; inside
    the pool, the output, the cache or an input -> ALIAS (decode, per-token
    slots, varlen, prefill and LA calls alike)."""
    def gdn(a, err):
        refs = [ctypes.byref(a[n]) if a[n] is not None else None for n in ORDER]
        return lib.gdn_decode(*refs, 1.0, 0, err, None)

    a = gdn_args()
    assert gdn(a, _err_word(0x7FF00002)) == ALIGN
    assert gdn(a, _err_word(a["pool"].data + 4096)) == ALIAS
    assert gdn(a, _err_word(a["out"].data)) == ALIAS
    assert gdn(a, _err_word(a["read_idx"].data + 4)) == ALIAS          # an input: the kernel reads it
    a["inter"] = fake([2, 1, 4, 64, 128])
    assert gdn(a, _err_word(a["inter"].data + 64)) == ALIAS
    # a word of its own passes these checks (the call then fails on an unrelated bad argument,
    # so nothing is launched)
    a = gdn_args()
    a["read_idx"] = fake([3], I32)
    assert gdn(a, _err_word(0x7FF00000)) == SHAPE

    a = gdn_args(B=2, T=3)
    refs = [ctypes.byref(x) if x is not None else None for x in
            [a[n] for n in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "pool")] + [a["read_idx"], None,
                                                                                       fake([2, 3], I32), a["out"]]]
    assert lib.gdn_decode_tokens(*refs, 1.0, 0, _err_word(a["pool"].data), None) == ALIAS
    assert lib.gdn_decode_tokens(*refs, 1.0, 0, _err_word(0x7FF00001), None) == ALIGN

    v = varlen_args(V=128)
    vrefs = [ctypes.byref(v[n]) if v[n] is not None else None for n in VARLEN_ORDER]
    assert lib.gdn_decode_varlen(*vrefs, 1.0, 0, _err_word(v["cu_seqlens"].data), None) == ALIAS
    assert lib.gdn_decode_varlen(*vrefs, 1.0, 0, _err_word(0x7FF00003), None) == ALIGN
    prefs = [ctypes.byref(v[n]) if v[n] is not None else None for n in PREFILL_ORDER]
    assert lib.gdn_prefill(*prefs, 1.0, 0, _err_word(v["out"].data + 8), None) == ALIAS

    q, k, vv = fake([2, 4, 128], BF16), fake([2, 4, 128], BF16), fake([2, 4, 128], BF16)
    pool, decay, ri, out = fake([5 * 4, 128, 128]), fake([4]), fake([2], I64), fake([2, 4, 128], BF16)
    refs = [ctypes.byref(x) for x in (q, k, vv, decay, pool, ri)] + [None, ctypes.byref(out), None]
    assert lib.la_decode(*refs, 1.0, _err_word(decay.data), None) == ALIAS
    assert lib.la_decode(*refs, 1.0, _err_word(0x7FF00002), None) == ALIGN


def test_binding_rejects_cpu_and_mixed_devices():
    """The Python binding places a call on the one device all of its tensors
    share; CPU tensors and mixed devices are refused before the C ABI is
    reached (checked here with CPU and meta tensors, which need no GPU)."""
    import torch
    cpu = torch.zeros(4)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        binding._device_of([cpu, cpu])
    with pytest.raises(ValueError, match="one CUDA device"):
        binding._device_of([cpu, torch.empty(4, device="meta")])
    with pytest.raises(ValueError, match="one CUDA device"):
        binding._device_of([cpu], dev_err=torch.empty(1, dtype=torch.int32, device="meta"))
