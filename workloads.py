"""Seeded synthetic inputs for the recurrent decode step.

This module is the one piece shared by the oracle side (tests) and the CUDA
side (tests, ``bench.py``, ``smoke()``).  It draws inputs and nothing else: it
performs none of the decode arithmetic, and imports neither the oracle nor the
library.  Where a workload recipe defines an input as a transformed draw
(``q, k`` l2-normalised in fp32 before the bf16 cast, ``g = -softplus(N(0,1))``,
``beta = sigmoid(N(0,1))``, ``lambda_h = exp(-2^(-8(h+1)/H))``), torch's own
functions shape the distribution; the decode kernels receive the result as
plain data with their in-kernel gate / l2norm switches off.

Recipes (seed s; CPU ``torch.Generator``; draw order q, k, v, g or a, beta,
A_log, dt_bias, read_idx, write_idx, then the pool):

=================  ===========================================================
gdn_tiny           B=2 T=1 H=HV=2 K=V=16, fp32 everywhere, pool [4,2,16,16],
                   read = write = [3, 1], seed 0
gdn_b64            B=64 T=1 H=16 HV=32 K=V=128, bf16 q/k/v/out, fp32 g/beta,
                   pool [256,32,128,128]; read = write = randperm(256)[:64]; seed 2
gdn_mtp_strided    B=16 T=4 H=16 HV=32, pool = backing[::2] of [256,32,128,128];
                   read = randperm(128)[:16]; write = 16 distinct unread slots,
                   4 of them set to -1; all T states cached; seed 3
kda_b256           B=256 T=1 H=HV=24, raw bf16 q/k (l2norm in kernel), raw bf16
                   gate a [B,T,HV,K], A_log ~ U(log 1, log 16) [HV], dt_bias ~
                   N(0, 0.1) [HV*K], raw beta logits; pool [320,24,128,128];
                   read = write = randperm(320)[:256]; seed 4
gdn_b64_bf16       gdn_b64 with a bfloat16 state pool (drawn in fp32, rounded once)
gdn_b64_kv         gdn_b64 with the state held untransposed, pool [256,32,128(k),128(v)]
gdn_spec_b64       B=64 T=4 H=16 HV=32, per-token pool slots: one row of 4 distinct
                   slots per sequence (of 320), seed = slot of the last accepted
                   token, accepted counts uniform in 1..4; seed 6
la_b512_packed     B=512 T=1 H=64, q/k/v head-dim slices of one fused bf16
                   [B,H,384] buffer (q, k ~ N(0,1)/sqrt(128), v ~ N(0,1)),
                   lambda_h = exp(-2^(-8(h+1)/64)), flat pool [640*64,128,128];
                   read = write = randperm(640)[:512]; seed 5
gdn_b64_kv_bf16    gdn_b64_kv with a bfloat16 state pool
kda_b256_bf16      kda_b256 with a bfloat16 state pool
la_b512_bf16       la_b512_packed with a bfloat16 state pool
gdn_varlen_b64     N=64 variable-length spans (draw order: 48 lengths U{1..4}, 16
                   lengths U{16..128}, a permutation of the 64), token-major bf16
                   q/k/v [Ntok,..] drawn as gdn_b64 draws them, fp32 g/beta
                   [Ntok,HV], H=16 HV=32 K=V=128, pool [256,32,128,128];
                   read = write = randperm(256)[:64]; seed 7
gdn_prefill_n16    N=16 spans, lengths U{256..1024} (drawn first), otherwise drawn as
                   gdn_varlen_b64; pool [64,32,128,128], read = write =
                   randperm(64)[:16]; run through the chunked prefill call; seed 8
kda_prefill_n16    N=16 spans, lengths U{256..1024} (drawn first), H=HV=24
                   K=V=128, token-major raw bf16 q/k/a drawn as kda_b256 draws
                   them (l2 norm, gate chain and sigmoid in kernel); pool
                   [64,24,128,128], read = write = randperm(64)[:16]; run
                   through the chunked prefill call; seed 9
=================  ===========================================================

Pool entries are N(0, 0.1^2) (standard deviation 0.1).  Full-size pools are
large (up to 2.7 GB), so ``pool_device="cuda"`` draws them on the device with
a CUDA ``torch.Generator`` seeded with s; the oracle then reads a host copy of
those drawn values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch
import torch.nn.functional as F

BF16 = torch.bfloat16
F32 = torch.float32

CONFIGS = ("gdn_tiny", "gdn_b64", "gdn_mtp_strided", "kda_b256", "la_b512_packed",
           "gdn_b64_bf16", "gdn_spec_b64", "gdn_b64_kv", "gdn_b64_kv_bf16", "kda_b256_bf16",
           "la_b512_bf16", "gdn_varlen_b64", "gdn_prefill_n16", "kda_prefill_n16")
SEEDS = {"gdn_tiny": 0, "gdn_b64": 2, "gdn_mtp_strided": 3, "kda_b256": 4,
         "la_b512_packed": 5, "gdn_b64_bf16": 2, "gdn_spec_b64": 6, "gdn_b64_kv": 2,
         "gdn_b64_kv_bf16": 2, "kda_b256_bf16": 4, "la_b512_bf16": 5, "gdn_varlen_b64": 7,
         "gdn_prefill_n16": 8, "kda_prefill_n16": 9}


@dataclass
class Workload:
    name: str
    form: str                      # "gdn" | "kda" | "la"
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    P: int                         # pool slots
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    pool: torch.Tensor             # the view the decode step reads and writes
    read_idx: torch.Tensor
    write_idx: torch.Tensor | None
    out_dtype: torch.dtype
    g: torch.Tensor | None = None
    beta: torch.Tensor | None = None
    A_log: torch.Tensor | None = None
    dt_bias: torch.Tensor | None = None
    decay: torch.Tensor | None = None
    backing: torch.Tensor | None = None    # set when `pool` is a strided view
    fused: torch.Tensor | None = None      # set when q/k/v are slices of one buffer
    qk_l2norm: bool = False
    gate_raw: bool = False
    beta_raw: bool = False
    scale: float = 1.0
    cache_intermediate: bool = False
    inter_dtype: torch.dtype = F32
    state_kv: bool = False                     # pool / cache hold S as [k][v] (v fastest)
    cu_seqlens: torch.Tensor | None = None     # [N+1] token offsets (variable-length mode)
    state_idx: torch.Tensor | None = None      # per-token write slots [B, T] (token-slot mode)
    num_accepted: torch.Tensor | None = None   # seed selection [B] (token-slot mode)
    meta: dict = field(default_factory=dict)

    def algorithmic_bytes(self) -> int:
        """Bytes a perfect implementation moves per call (each input read once,
        each output written once): state read for entries with a valid read
        slot, state write for entries with a valid write slot, every cached
        intermediate state, plus q/k/v/gate/out/index bytes."""
        unit = self.K * self.V * self.pool.element_size()
        heads = self.HV
        if self.state_idx is not None:
            tab = self.state_idx.to("cpu")
            if self.num_accepted is not None:
                a = self.num_accepted.to("cpu").long()
                ok = (a >= 1) & (a <= self.T)
                seed = torch.where(ok, tab.gather(1, (a.clamp(1, self.T) - 1)[:, None])[:, 0],
                                   torch.full_like(a, -1))
            else:
                seed = self.read_idx.to("cpu")
            n_read = int(((seed >= 0) & (seed < self.P)).sum())
            n_write = int(((tab >= 0) & (tab < self.P)).sum())
        else:
            r = self.read_idx.to("cpu")
            w = (self.write_idx if self.write_idx is not None else self.read_idx).to("cpu")
            n_read = int(((r >= 0) & (r < self.P)).sum())
            n_write = int(((w >= 0) & (w < self.P)).sum())
        total = (n_read + n_write) * heads * unit
        if self.cache_intermediate:
            total += self.tokens() * heads * self.K * self.V * torch.finfo(self.inter_dtype).bits // 8
        small = [self.q, self.k, self.v, self.g, self.beta, self.A_log, self.dt_bias,
                 self.decay, self.state_idx, self.num_accepted]
        if self.state_idx is None:
            small += [self.read_idx, self.write_idx]
        elif self.num_accepted is None:
            small += [self.read_idx]
        if self.cu_seqlens is not None:
            small += [self.cu_seqlens]
        total += sum(t.numel() * t.element_size() for t in small if t is not None)
        total += self.tokens() * heads * self.V * torch.finfo(self.out_dtype).bits // 8
        return int(total)

    def alu_ops(self) -> int:
        """fp32 lane operations of the state update per call: per token and state
        element a decay multiply, the S^T k and S^T q multiply-adds and the
        rank-1 update (GDN, KDA: 4); LA has no S^T k (3)."""
        per = 3 if self.form == "la" else 4
        return self.tokens() * self.HV * self.K * self.V * per

    def tokens(self) -> int:
        """Tokens the call decodes (in variable-length mode: the tokens inside
        the spans, the only ones that produce an output)."""
        if self.cu_seqlens is not None:
            cu = self.cu_seqlens.to("cpu").long()
            return int((cu[1:] - cu[:-1]).clamp(min=0).sum())
        return self.B * self.T

    def qkv_to(self, device):
        """(q, k, v) on `device`.  When they are views of one fused buffer, that
        buffer is copied once (same shape and strides) and q, k, v become the
        same views of the copy (same shapes, strides and offsets), so a call on
        the device sees the packed layout.  (`Tensor.to` of a non-dense view
        would hand back a dense copy.)"""
        if self.fused is None:
            return self.q.to(device), self.k.to(device), self.v.to(device)
        f = self.fused
        fd = torch.empty_strided(f.shape, f.stride(), dtype=f.dtype, device=device)
        fd.copy_(f)

        def view(t):
            assert t.untyped_storage().data_ptr() == f.untyped_storage().data_ptr()
            return fd.as_strided(t.shape, t.stride(), fd.storage_offset() + t.storage_offset() - f.storage_offset())

        return view(self.q), view(self.k), view(self.v)


def _normal(gen, shape, std=1.0):
    return torch.randn(shape, generator=gen, dtype=F32) * std


def _l2n(x):
    return F.normalize(x, p=2.0, dim=-1)


def _draw_pool(gen, shape, seed, device, dtype=F32):
    """N(0, 0.1^2) state, drawn in fp32 and (for a bf16 pool) rounded once."""
    if torch.device(device).type == "cpu":
        return _normal(gen, shape, 0.1).to(dtype)
    dg = torch.Generator(device=device)
    dg.manual_seed(seed)
    pool = torch.empty(shape, dtype=F32, device=device)
    pool.normal_(0.0, 0.1, generator=dg)
    return pool.to(dtype)


def make_meta(name: str) -> dict:
    """Workload flags known without drawing it (which call runs it)."""
    if name not in CONFIGS:
        raise KeyError(name)
    # split: a variable-length call without a state cache at K = V = 128 runs its
    # long spans in the chunked kernel and the rest in the token-by-token kernel
    return {"prefill": name in ("gdn_prefill_n16", "kda_prefill_n16"), "split": name == "gdn_varlen_b64"}


def make(name: str, *, seed: int | None = None, pool_device="cpu",
         index_dtype=torch.int32) -> Workload:
    """Draw the named workload (see the module docstring for the recipes)."""
    s = SEEDS[name] if seed is None else seed
    gen = torch.Generator().manual_seed(s)
    if name == "gdn_tiny":
        B, T, H, HV, K, V, P = 2, 1, 2, 2, 16, 16, 4
        q = _l2n(_normal(gen, (B, T, H, K)))
        k = _l2n(_normal(gen, (B, T, H, K)))
        v = _normal(gen, (B, T, HV, V))
        g = -F.softplus(_normal(gen, (B, T, HV)))
        beta = torch.sigmoid(_normal(gen, (B, T, HV)))
        ri = torch.tensor([3, 1], dtype=index_dtype)
        pool = _draw_pool(gen, (P, HV, V, K), s, pool_device)
        return Workload(name, "gdn", B, T, H, HV, K, V, P, q, k, v, pool, ri, ri.clone(),
                        F32, g=g, beta=beta)
    if name in ("gdn_b64", "gdn_b64_bf16", "gdn_b64_kv", "gdn_b64_kv_bf16"):
        B, T, H, HV, K, V, P = 64, 1, 16, 32, 128, 128, 256
        q = _l2n(_normal(gen, (B, T, H, K))).to(BF16)
        k = _l2n(_normal(gen, (B, T, H, K))).to(BF16)
        v = _normal(gen, (B, T, HV, V)).to(BF16)
        g = -F.softplus(_normal(gen, (B, T, HV)))
        beta = torch.sigmoid(_normal(gen, (B, T, HV)))
        ri = torch.randperm(P, generator=gen)[:B].to(index_dtype)
        kv = name.startswith("gdn_b64_kv")
        pool = _draw_pool(gen, (P, HV, K, V) if kv else (P, HV, V, K), s, pool_device,
                          BF16 if name.endswith("_bf16") else F32)
        return Workload(name, "gdn", B, T, H, HV, K, V, P, q, k, v, pool, ri, ri.clone(),
                        BF16, g=g, beta=beta, state_kv=kv)
    if name == "gdn_mtp_strided":
        B, T, H, HV, K, V, M = 16, 4, 16, 32, 128, 128, 2
        P = 128
        q = _l2n(_normal(gen, (B, T, H, K))).to(BF16)
        k = _l2n(_normal(gen, (B, T, H, K))).to(BF16)
        v = _normal(gen, (B, T, HV, V)).to(BF16)
        g = -F.softplus(_normal(gen, (B, T, HV)))
        beta = torch.sigmoid(_normal(gen, (B, T, HV)))
        ri, wi = _read_write_disjoint(gen, P, B, skip_frac=0.25)
        backing = _draw_pool(gen, (P * M, HV, V, K), s, pool_device)
        pool = backing[::M]
        return Workload(name, "gdn", B, T, H, HV, K, V, P, q, k, v, pool,
                        ri.to(index_dtype), wi.to(index_dtype), BF16, g=g, beta=beta,
                        backing=backing, cache_intermediate=True, meta={"stride_mult": M})
    if name == "gdn_spec_b64":
        # speculative verify: one row of T slots per sequence, reused every step;
        # the seed is the state after the last accepted draft token
        B, T, H, HV, K, V, P = 64, 4, 16, 32, 128, 128, 320
        q = _l2n(_normal(gen, (B, T, H, K))).to(BF16)
        k = _l2n(_normal(gen, (B, T, H, K))).to(BF16)
        v = _normal(gen, (B, T, HV, V)).to(BF16)
        g = -F.softplus(_normal(gen, (B, T, HV)))
        beta = torch.sigmoid(_normal(gen, (B, T, HV)))
        table = torch.randperm(P, generator=gen)[:B * T].view(B, T).to(index_dtype)
        accepted = torch.randint(1, T + 1, (B,), generator=gen).to(index_dtype)
        pool = _draw_pool(gen, (P, HV, V, K), s, pool_device)
        return Workload(name, "gdn", B, T, H, HV, K, V, P, q, k, v, pool, table[:, 0].clone(), None,
                        BF16, g=g, beta=beta, state_idx=table, num_accepted=accepted)
    if name in ("kda_b256", "kda_b256_bf16"):
        B, T, H, HV, K, V, P = 256, 1, 24, 24, 128, 128, 320
        q = _normal(gen, (B, T, H, K)).to(BF16)
        k = _normal(gen, (B, T, H, K)).to(BF16)
        v = _normal(gen, (B, T, HV, V)).to(BF16)
        a = _normal(gen, (B, T, HV, K)).to(BF16)
        b_raw = _normal(gen, (B, T, HV))
        A_log = torch.empty(HV).uniform_(math.log(1.0), math.log(16.0), generator=gen)
        dt_bias = _normal(gen, (HV * K,), 0.1)
        ri = torch.randperm(P, generator=gen)[:B].to(index_dtype)
        pool = _draw_pool(gen, (P, HV, V, K), s, pool_device, BF16 if name.endswith("_bf16") else F32)
        return Workload(name, "kda", B, T, H, HV, K, V, P, q, k, v, pool, ri, ri.clone(),
                        BF16, g=a, beta=b_raw, A_log=A_log, dt_bias=dt_bias,
                        qk_l2norm=True, gate_raw=True, beta_raw=True)
    if name in ("la_b512_packed", "la_b512_bf16"):
        B, H, K, V, P = 512, 64, 128, 128, 640
        fused = torch.cat([_normal(gen, (B, H, K), 1.0 / math.sqrt(K)),
                           _normal(gen, (B, H, K), 1.0 / math.sqrt(K)),
                           _normal(gen, (B, H, V))], dim=-1).to(BF16)
        q, k, v = fused[..., :K], fused[..., K:2 * K], fused[..., 2 * K:]
        decay = la_decay_rates(H)
        ri = torch.randperm(P, generator=gen)[:B].to(index_dtype)
        pool = _draw_pool(gen, (P * H, V, K), s, pool_device, BF16 if name.endswith("_bf16") else F32)
        return Workload(name, "la", B, 1, H, H, K, V, P, q, k, v, pool, ri, ri.clone(),
                        BF16, decay=decay, fused=fused)
    if name == "gdn_varlen_b64":
        # variable-length spans: 48 short decode / verify spans and 16 prefill
        # chunks, in random order, token-major
        N, H, HV, K, V, P = 64, 16, 32, 128, 128, 256
        short = torch.randint(1, 5, (48,), generator=gen)
        long_ = torch.randint(16, 129, (16,), generator=gen)
        lengths = torch.cat([short, long_])[torch.randperm(N, generator=gen)]
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
        NT = int(cu[-1])
        q = _l2n(_normal(gen, (NT, H, K))).to(BF16)
        k = _l2n(_normal(gen, (NT, H, K))).to(BF16)
        v = _normal(gen, (NT, HV, V)).to(BF16)
        g = -F.softplus(_normal(gen, (NT, HV)))
        beta = torch.sigmoid(_normal(gen, (NT, HV)))
        ri = torch.randperm(P, generator=gen)[:N].to(index_dtype)
        pool = _draw_pool(gen, (P, HV, V, K), s, pool_device)
        return Workload(name, "gdn", N, 0, H, HV, K, V, P, q, k, v, pool, ri, ri.clone(),
                        BF16, g=g, beta=beta, cu_seqlens=cu)
    if name == "gdn_prefill_n16":
        # long spans for the chunked prefill call: 16 sequences of 256-1024 tokens
        N, H, HV, K, V, P = 16, 16, 32, 128, 128, 64
        lengths = torch.randint(256, 1025, (N,), generator=gen)
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
        NT = int(cu[-1])
        q = _l2n(_normal(gen, (NT, H, K))).to(BF16)
        k = _l2n(_normal(gen, (NT, H, K))).to(BF16)
        v = _normal(gen, (NT, HV, V)).to(BF16)
        g = -F.softplus(_normal(gen, (NT, HV)))
        beta = torch.sigmoid(_normal(gen, (NT, HV)))
        ri = torch.randperm(P, generator=gen)[:N].to(index_dtype)
        pool = _draw_pool(gen, (P, HV, V, K), s, pool_device)
        return Workload(name, "gdn", N, 0, H, HV, K, V, P, q, k, v, pool, ri, ri.clone(),
                        BF16, g=g, beta=beta, cu_seqlens=cu, meta={"prefill": True})
    if name == "kda_prefill_n16":
        # long spans for the chunked KDA call: 16 sequences of 256-1024 tokens
        N, H, HV, K, V, P = 16, 24, 24, 128, 128, 64
        lengths = torch.randint(256, 1025, (N,), generator=gen)
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
        NT = int(cu[-1])
        q = _normal(gen, (NT, H, K)).to(BF16)
        k = _normal(gen, (NT, H, K)).to(BF16)
        v = _normal(gen, (NT, HV, V)).to(BF16)
        a = _normal(gen, (NT, HV, K)).to(BF16)
        b_raw = _normal(gen, (NT, HV))
        A_log = torch.empty(HV).uniform_(math.log(1.0), math.log(16.0), generator=gen)
        dt_bias = _normal(gen, (HV * K,), 0.1)
        ri = torch.randperm(P, generator=gen)[:N].to(index_dtype)
        pool = _draw_pool(gen, (P, HV, V, K), s, pool_device)
        return Workload(name, "kda", N, 0, H, HV, K, V, P, q, k, v, pool, ri, ri.clone(),
                        BF16, g=a, beta=b_raw, A_log=A_log, dt_bias=dt_bias, cu_seqlens=cu,
                        qk_l2norm=True, gate_raw=True, beta_raw=True, meta={"prefill": True})
    raise KeyError(name)


def la_decay_rates(H: int) -> torch.Tensor:
    """lambda_h = exp(-2^(-8(h+1)/H)), h = 0..H-1, as fp32 (the LA workload's rates)."""
    h = torch.arange(H, dtype=torch.float64)
    return torch.exp(-torch.pow(2.0, -8.0 * (h + 1) / H)).to(F32)


def _read_write_disjoint(gen, P, B, skip_frac=0.0):
    """Distinct read slots, and distinct write slots drawn from the slots no entry
    reads; round(skip_frac * B) write entries are then set to -1."""
    perm = torch.randperm(P, generator=gen)
    ri = perm[:B].clone()
    unread = perm[B:]
    wi = unread[torch.randperm(unread.numel(), generator=gen)[:B]].clone()
    n_skip = int(round(skip_frac * B))
    if n_skip:
        wi[torch.randperm(B, generator=gen)[:n_skip]] = -1
    return ri, wi


def make_custom(form: str, *, B: int, T: int, H: int, HV: int | None = None, K: int = 128,
                V: int = 128, P: int | None = None, seed: int = 0, in_dtype=BF16,
                out_dtype=BF16, separate_write: bool = False, skip_frac: float = 0.0,
                stride_mult: int = 1, cache_intermediate: bool = False,
                raw_gates: bool = False, packed: bool = False, flat_pool: bool = False,
                index_dtype=torch.int32, pool_device="cpu", state_dtype=F32,
                inter_dtype=None, state_kv: bool = False) -> Workload:
    """A workload of any size in the same distributions as the named recipes.

    ``raw_gates``: q/k raw N(0,1) with in-kernel l2norm, raw gate input and beta
    logits with A_log/dt_bias (the KDA recipe); otherwise activated g/beta and
    pre-normalised q/k (the GDN recipe).  LA always uses the LA recipe.
    ``separate_write``: write slots distinct from every read slot.
    ``stride_mult`` > 1: the pool is backing[::stride_mult].
    ``packed``: q/k/v are slices of one fused [B,T,H,2K+V] buffer (needs H == HV).
    ``state_dtype``: fp32 or bf16 pool; ``inter_dtype``: the state cache's type
    (default: the pool's).  ``state_kv``: the pool holds S as [P, HV, K, V].
    """
    HV = H if HV is None else HV
    P = max(2 * B, 4) if P is None else P
    gen = torch.Generator().manual_seed(seed)
    fused = None
    if form == "la":
        HV = H
        if packed:
            fused = torch.cat([_normal(gen, (B, T, H, K), 1.0 / math.sqrt(K)),
                               _normal(gen, (B, T, H, K), 1.0 / math.sqrt(K)),
                               _normal(gen, (B, T, H, V))], dim=-1).to(in_dtype)
            q, k, v = fused[..., :K], fused[..., K:2 * K], fused[..., 2 * K:]
        else:
            q = _normal(gen, (B, T, H, K), 1.0 / math.sqrt(K)).to(in_dtype)
            k = _normal(gen, (B, T, H, K), 1.0 / math.sqrt(K)).to(in_dtype)
            v = _normal(gen, (B, T, H, V)).to(in_dtype)
        g = beta = A_log = dt_bias = None
        decay = la_decay_rates(H)
    else:
        if packed:
            if H != HV:
                raise ValueError("packed q/k/v needs H == HV")
            raw = torch.cat([_normal(gen, (B, T, H, K)), _normal(gen, (B, T, H, K)),
                             _normal(gen, (B, T, H, V))], dim=-1)
            if not raw_gates:
                raw = torch.cat([_l2n(raw[..., :K]), _l2n(raw[..., K:2 * K]),
                                 raw[..., 2 * K:]], dim=-1)
            fused = raw.to(in_dtype)
            q, k, v = fused[..., :K], fused[..., K:2 * K], fused[..., 2 * K:]
        else:
            qf, kf = _normal(gen, (B, T, H, K)), _normal(gen, (B, T, H, K))
            if not raw_gates:
                qf, kf = _l2n(qf), _l2n(kf)
            q, k = qf.to(in_dtype), kf.to(in_dtype)
            v = _normal(gen, (B, T, HV, V)).to(in_dtype)
        gshape = (B, T, HV, K) if form == "kda" else (B, T, HV)
        if raw_gates:
            g = _normal(gen, gshape).to(in_dtype)
            beta = _normal(gen, (B, T, HV))
            A_log = torch.empty(HV).uniform_(math.log(1.0), math.log(16.0), generator=gen)
            dt_bias = _normal(gen, (HV * K,) if form == "kda" else (HV,), 0.1)
        else:
            g = -F.softplus(_normal(gen, gshape))
            beta = torch.sigmoid(_normal(gen, (B, T, HV)))
            A_log = dt_bias = None
        decay = None
    if separate_write:
        ri, wi = _read_write_disjoint(gen, P, B, skip_frac)
    else:
        ri = torch.randperm(P, generator=gen)[:B]
        wi = ri.clone()
        n_skip = int(round(skip_frac * B))
        if n_skip:
            wi[torch.randperm(B, generator=gen)[:n_skip]] = -1
    backing = None
    if form == "la" and flat_pool:
        pool = _draw_pool(gen, (P * H, V, K), seed, pool_device, state_dtype)
    elif stride_mult > 1:
        rows = (K, V) if state_kv else (V, K)
        backing = _draw_pool(gen, (P * stride_mult, HV) + rows, seed, pool_device, state_dtype)
        pool = backing[::stride_mult]
    elif state_kv:
        pool = _draw_pool(gen, (P, HV, K, V), seed, pool_device, state_dtype)
    else:
        pool = _draw_pool(gen, (P, HV, V, K), seed, pool_device, state_dtype)
    return Workload(f"custom_{form}", form, B, T, H, HV, K, V, P, q, k, v, pool,
                    ri.to(index_dtype), wi.to(index_dtype), out_dtype, g=g, beta=beta,
                    A_log=A_log, dt_bias=dt_bias, decay=decay, backing=backing,
                    fused=fused, qk_l2norm=raw_gates and form != "la",
                    gate_raw=raw_gates and form != "la",
                    beta_raw=raw_gates and form != "la",
                    cache_intermediate=cache_intermediate,
                    inter_dtype=state_dtype if inter_dtype is None else inter_dtype,
                    state_kv=state_kv)


def make_varlen(form: str, lengths, *, H: int, HV: int | None = None, K: int = 128, V: int = 128,
                P: int | None = None, seed: int = 0, pool_device="cpu", **kw) -> Workload:
    """Variable-length spans: sequence n owns ``lengths[n]`` consecutive tokens
    of token-major inputs (q, k [Ntok,H,K], v [Ntok,HV,V], g and beta
    [Ntok,HV] or [Ntok,HV,K]), ``cu_seqlens`` = [0, cumsum(lengths)].  The
    tokens are drawn as ``make_custom`` draws one sequence of Ntok tokens; the
    N read / write slots are then drawn from a second generator seeded with
    seed + 1 (``separate_write`` and ``skip_frac`` as in ``make_custom``).
    Other keywords go to ``make_custom`` (dtypes, gates, pool layout, cache)."""
    lengths = [int(x) for x in lengths]
    N, ntok = len(lengths), sum(lengths)
    HV = H if HV is None else HV
    P = max(2 * N, 4) if P is None else P
    separate_write = kw.pop("separate_write", False)
    skip_frac = kw.pop("skip_frac", 0.0)
    index_dtype = kw.pop("index_dtype", torch.int32)
    w = make_custom(form, B=1, T=ntok, H=H, HV=HV, K=K, V=V, P=P, seed=seed,
                    pool_device=pool_device, **kw)
    gen = torch.Generator().manual_seed(seed + 1)
    if separate_write:
        ri, wi = _read_write_disjoint(gen, P, N, skip_frac)
    else:
        ri = torch.randperm(P, generator=gen)[:N]
        wi = ri.clone()
        n_skip = int(round(skip_frac * N))
        if n_skip:
            wi[torch.randperm(N, generator=gen)[:n_skip]] = -1
    tok = lambda x: None if x is None else x[0]
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    w.name, w.B, w.T = f"varlen_{form}", N, 0
    w.q, w.k, w.v, w.g, w.beta = tok(w.q), tok(w.k), tok(w.v), tok(w.g), tok(w.beta)
    w.fused = tok(w.fused)
    w.read_idx, w.write_idx = ri.to(index_dtype), wi.to(index_dtype)
    w.cu_seqlens = cu
    return w


def disjoint_index_sets(P: int, B: int, n: int, seed: int, index_dtype=torch.int32):
    """n index sets of B distinct slots each, pairwise disjoint (n * B <= P)."""
    if n * B > P:
        raise ValueError("not enough slots for disjoint sets")
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(seed))
    return [perm[i * B:(i + 1) * B].to(index_dtype) for i in range(n)]
