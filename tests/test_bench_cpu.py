"""bench.py host logic on the CPU: the reference (oracle) arm's JSON line, and
the multi-process path (world size 2, gloo): max-over-ranks timing, rank 0
alone printing, the other ranks exiting cleanly."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REQUIRED = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "config", "cpu_baseline", "e2e"}


def _run(cmd, env=None, timeout=600):
    e = dict(os.environ)
    e.update(env or {})
    e["CUDA_VISIBLE_DEVICES"] = ""
    return subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=timeout, env=e)


def test_reference_arm_single_process():
    r = _run([sys.executable, "bench.py", "--impl", "reference", "--config", "gdn_tiny",
              "--steps", "5", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert REQUIRED <= set(d) and d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_reference_arm_two_ranks_gloo():
    port = _free_port()
    r = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
              "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
              "reference", "--gpus", "2", "--config", "gdn_tiny", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1                      # rank 0 alone prints
    assert json.loads(lines[0])["n_gpus"] == 2


def _max_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    q.put((rank, bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_max_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_roofline_bound_and_sample_bytes():
    """The roofline names the larger ideal time (HBM for fixed-T decode, the
    FMA pipe for long variable-length spans), and the reference arm's sample
    bytes of all entries equal the whole step's algorithmic bytes."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    dec = W.make_custom("gdn", B=64, T=1, H=16, HV=32, K=128, V=128, P=128, seed=1)
    r = bench.roofline(dec, "x", 0.045, 6000.0, 6791.4, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - 6000.0 / 6791.4) < 1e-4
    vl = W.make_varlen("gdn", [256] * 16, H=16, HV=32, K=128, V=128, P=64, seed=1)
    assert vl.alu_ops() == 16 * 256 * 32 * 128 * 128 * 4
    r = bench.roofline(vl, "x", 1.0, 100.0, 6791.4, "measured")
    assert r["bound"] == "alu" and r["unit"] == "T lane-op/s"
    assert abs(r["achieved"] - vl.alu_ops() / 1e-3 / 1e12) < 1e-3
    assert bench.sample_bytes(vl, vl.B) == vl.algorithmic_bytes()
    mixed = W.make("gdn_varlen_b64")
    assert abs(bench.sample_bytes(mixed, mixed.B) - mixed.algorithmic_bytes()) < 1
    assert bench.sample_bytes(mixed, 8) < mixed.algorithmic_bytes()


def test_oracle_step_on_variable_length_spans():
    """The CPU baseline's per-entry oracle step on variable-length spans writes
    what one whole-workload oracle call writes."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import workloads as W
    w = W.make_varlen("gdn", [3, 0, 5, 1], H=1, HV=2, K=16, V=8, seed=4, separate_write=True)
    ref_pool, step_pool = w.pool.clone(), w.pool.clone()
    oracle.gdn_decode_varlen(w.q, w.k, w.v, w.g, w.beta, ref_pool, w.cu_seqlens, w.read_idx, w.write_idx)
    bench._oracle_step(w, step_pool, torch.arange(w.B))
    assert torch.equal(ref_pool, step_pool)


def test_kernel_hash_ignores_comments_and_separates_kernels():
    """ncu traffic figures are keyed by a hash of the kernel's code: comments
    and whitespace do not count, string literals do, and the decode and
    prefill kernels are hashed from their own sources."""
    sys.path.insert(0, ROOT)
    import bench
    a = 'int f() { return 1; } // one\n/* two */ const char* s = "// kept";\n'
    b = 'int f()  {  return 1; }\nconst char* s = "// kept"; // other\n'
    c = 'int f() { return 2; }\nconst char* s = "// kept";\n'
    assert bench._code_only(a) == bench._code_only(b) != bench._code_only(c)
    assert '"// kept"' in bench._code_only(a)
    assert bench.kernel_source_hash("gdn_b64") == bench.kernel_source_hash("kda_b256")
    assert bench.kernel_source_hash("gdn_b64") != bench.kernel_source_hash("gdn_prefill_n16")
    # a split variable-length call runs both kernels: its hash covers both sets of sources
    split = bench.kernel_source_hash("gdn_varlen_b64")
    assert split not in (bench.kernel_source_hash("gdn_b64"), bench.kernel_source_hash("gdn_prefill_n16"))


def test_launches_per_call():
    """gpu_launches counts both kernels of a split variable-length call, and one
    when no span can reach the chunked kernel's 16 tokens (it is not launched)."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    assert bench.launches_per_step(W.make("gdn_b64")) == 1
    assert bench.launches_per_step(W.make("gdn_prefill_n16")) == 1
    assert bench.launches_per_step(W.make("gdn_varlen_b64")) == 2
    assert bench.launches_per_step(W.make_varlen("gdn", [1] * 15, H=1, HV=2)) == 1
    assert bench.launches_per_step(W.make_varlen("gdn", [1] * 16, H=1, HV=2)) == 2
    assert bench.launches_per_step(W.make_varlen("gdn", [20], H=1, HV=2, K=64, V=64)) == 1
    assert bench.launches_per_step(W.make_varlen("gdn", [20], H=1, HV=2, cache_intermediate=True)) == 1
