"""CPU checks of bench.py's host logic: the replica timing path across two
gloo ranks (barrier + max over ranks), and the reference arm (the fp64
oracle timed on host cores) printing one JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), MOE_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + r, w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, m))


def test_replica_timing_takes_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]


def test_work_model_counts_touched_experts():
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.WORKLOADS["dsv3"]
    offsets = [0] * 10 + [wl.N * wl.K] * (wl.E + 1 - 10)     # only expert 9 has rows
    wm = bench.work_model(wl, offsets)
    assert wm["touched_experts"] == 1 and wm["empty_experts"] == wl.E - 1
    assert wm["ffn_flop"] == 6 * wl.N * wl.K * wl.D * wl.Dff
    assert wm["ffn_bytes"] == 3 * wl.D * wl.Dff * 2 + 4 * wl.N * wl.K * wl.D + 4 * wl.N * wl.K * wl.Dff


def test_work_model_layer_bytes_one_token():
    """The one-launch layer's algorithmic bytes (its roofline denominator) at
    the Qwen3 one-token shape, eight distinct experts with one row each,
    listed tensor by tensor: what the layer must read once and write once."""
    sys.path.insert(0, ROOT)
    import bench
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.WORKLOADS["qwen3_N1"]
    N, D, E, K, Dff, A = wl.N, wl.D, wl.E, wl.K, wl.Dff, wl.N * wl.K
    assert (N, D, E, K, Dff) == (1, 2048, 128, 8, 768) and wl.act == synth.ACT_SWIGLU
    offsets = [min(e, A) for e in range(E + 1)]              # experts 0..7 get one row each
    reads_common = {"x": N * D * 2, "W_gate": E * D * 2}
    writes_common = {"ids + weights": N * K * (4 + 4), "expert_offsets": (E + 1) * 4,
                     "perm_src + inv_perm": A * (4 + 4), "h": A * Dff * 2, "y_perm": A * D * 2, "out": N * D * 2}
    bf16 = dict(reads_common, **writes_common, experts=8 * 3 * D * Dff * 2, x_perm=A * D * 2)
    assert bench.work_model(wl, offsets)["layer_bytes"] == sum(bf16.values()) == 76_108_420
    e4m3 = dict(reads_common, **writes_common,
                experts=8 * (3 * D * Dff + (Dff + Dff + D) * 4),     # codes + W1, W3, W2 row scales
                token_codes=N * D, token_scales=N * 4, permuted_codes=A * D, h_codes=A * Dff, h_scales=A * 4)
    assert bench.work_model(wl, offsets, e4m3=True)["layer_bytes"] == sum(e4m3.values()) == 38_466_216


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
