"""Host-side logic of bench.py: argument defaults, max-over-ranks timing with
two gloo ranks on the CPU, and the reference arm's JSON line (no GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    q.put((rank, bench.max_over_ranks(10.0 + rank * 5.0, world)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 15.0, 1: 15.0}


def test_defaults_and_single_rank():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.config == "C2" and a.warmup >= 3 and a.impl == "ours"
    assert bench.max_over_ranks(3.5, 1) == 3.5
    peak, src = bench.hbm_peak()
    assert peak > 1000 and src in ("of measured", "of fallback")


def test_reference_arm_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                          "--warmup", "1", "--config", "C1"], capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2"],
                         capture_output=True, text=True, env=env, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == ""


def test_shortlist_oracle_round_small():
    """The CPU legs of the shortlist workload go through the mapped oracle,
    whole and cut to a prefix of each column (the map cut with it)."""
    import synth
    r = synth.make_c5s(cols=4, V_local=4096, k=8)
    assert r.target is None and r.id_map.shape == (4096,)
    assert bench.oracle_round(r, 2) == r.logit_bytes()
    assert bench.oracle_round(r, 2, cols=([0, 3], []), n=1000) == 2 * 1000 * 2
    c = bench.workload_config(bench.parse_args(["--config", "C5s"]), r, None)
    assert c["workload"].startswith("C5s: shortlist") and c["lanes"] == 0


def test_part_modes():
    """--part: the fused round by default; the split round and each call
    alone are labelled in the config."""
    import synth
    assert bench.parse_args([]).part == "round"
    r = synth.make_c1(V=1000)
    assert "part" not in bench.workload_config(bench.parse_args([]), r, None)
    for part, word in (("split", "two launches"), ("topk", "spec_topk alone"), ("verify", "spec_verify_v alone")):
        c = bench.workload_config(bench.parse_args(["--part", part]), r, None)
        assert word in c["part"]


def test_cpu_baseline_fields():
    """The oracle leg: all cores, plus one core for small rounds."""
    import synth
    r = synth.make_c1(V=5000)
    c = bench.cpu_baseline(r, budget_s=0.05)
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["columns_per_s"] > 0
    assert c["one_core"]["value"] > 0 and c["one_core"]["us_per_round"] > 0
    assert "one_core" not in bench.cpu_baseline(r, budget_s=0.01, one_core_max_bytes=0)


def test_config_carries_input_hashes():
    """Every input buffer's content hash is in the config: equal for equal
    seeds, different for another seed."""
    import synth
    a, b, c = synth.make_c1(V=3000), synth.make_c1(V=3000), synth.make_c1(seed=2, V=3000)
    args = bench.parse_args(["--config", "C1"])
    ha = bench.workload_config(args, a, None)["input_sha256_16"]
    assert set(ha) == {"draft_logits", "target_logits", "drafts"}
    assert ha == bench.workload_config(args, b, None)["input_sha256_16"]
    assert ha["draft_logits"] != bench.workload_config(args, c, None)["input_sha256_16"]["draft_logits"]
    s = synth.make_c5s(cols=2, V_local=1024)
    assert "id_map" in bench.input_hashes(s) and "target_logits" not in bench.input_hashes(s)
