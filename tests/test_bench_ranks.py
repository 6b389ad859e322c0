"""The bench's multi-rank host logic on CPU: two gloo ranks agree on the
slowest rank's time, and the whole-job rate counts every rank's units over
it.  Each rank gets its own prompts but the same model, and the reference arm
prints on rank 0 only."""
import os
import socket
import sys
from types import SimpleNamespace

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import configs as C  # noqa: E402
from workloads import generate as G  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(ms[rank], world, "cpu")
        q.put((rank, slowest, bench.whole_job_rate(128, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port, ms = _free_port(), [12.5, 30.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in got:
        assert slowest == 30.0
        assert rate == 2 * 128 / 0.030


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.0, 1, "cpu") == 7.0
    assert bench.whole_job_rate(100, 1, 50.0) == 2000.0


def test_ranks_share_the_model_not_the_prompts():
    w = C.get("mid_bf16")
    w0, w1 = bench.rank_workload(w, 0), bench.rank_workload(w, 1)
    assert w0 == w
    assert not np.array_equal(G.prompt_tokens(w0), G.prompt_tokens(w1))
    # everything but the seed (the shapes, the model's scale, the schedule)
    # is the base workload's; the bench draws the weights from the base
    assert w1.seed != w.seed and bench.replace(w1, seed=w.seed) == w


def test_reference_arm_prints_on_rank_zero_only(capsys):
    args = SimpleNamespace(gpus=2, steps=1, warmup=0)
    bench.reference_arm(args, C.get("tiny_fp32"), 1)
    assert capsys.readouterr().out == ""


def test_profile_hash_ignores_comments_only():
    a = "int f(int x) {  // the sum\n  return x + 1; /* one\n more */ }\n"
    b = "int f(int x) {\n  return x + 1;\n}\n"
    c = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(b) != bench._code_only(c)


def test_profile_summaries_are_of_the_current_sources():
    """Every traffic line under profiles/ names a measured kernel and the hash
    of that kernel's current sources, so the bench reports each captured
    traffic figure and no figure of an older revision of a kernel."""
    import re
    pat = re.compile(r"traffic: kernel=(\S+) workload=(\S+) bytes_per_launch=(\d+) src_sha256=([0-9a-f]+)")
    pdir = os.path.join(ROOT, "profiles")
    seen = 0
    for name in sorted(os.listdir(pdir)):
        with open(os.path.join(pdir, name)) as f:
            for m in pat.finditer(f.read()):
                kernel, workload, nbytes, sha = m.groups()
                assert bench._src_key(kernel) is not None, (name, kernel)
                assert sha == bench.kernel_src_sha(kernel), (name, kernel)
                assert bench.profiled_traffic(kernel, workload) == int(nbytes), (name, kernel, workload)
                assert C.get(workload) is not None
                seen += 1
    assert seen >= 10


def test_cpu_baseline_sample_repeats_to_the_minimum_work():
    """The oracle sample runs once for the reference arm's steps, and repeats
    until the requested oracle work has run for the CPU baseline; the tiny
    workload's generation is timed whole, not extrapolated."""
    w = C.get("tiny_fp32")
    m = G.model(w)
    g1, d1 = bench.oracle_sample(w, m)
    assert g1 > 0 and "whole generation" in d1 and "repetitions" not in d1
    g2, d2 = bench.oracle_sample(w, m, 0.2)
    assert g2 > 0 and "repetitions" in d2
    n = int(d2.split("the median of ")[1].split(" ")[0])
    assert n >= 2
