"""bench.py host logic on the CPU: the N>1 aggregation over gloo ranks and the
reference arm (the oracle timed on the host)."""
import json
import os
import socket
import subprocess
import sys
import time

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # replicas: each rank ran its own batch; value = all tokens / slowest rank
    tokens, seconds = bench.aggregate(1000 * (rank + 1), 0.5 + rank, world)
    out.put((rank, tokens, seconds))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for _, tokens, seconds in got:
        assert tokens == 3000 and seconds == 1.5


def test_aggregate_single_rank_is_identity():
    import bench
    assert bench.aggregate(42, 0.25, 1) == (42, 0.25)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny_fp32", "--steps", "1", "--warmup", "0",
                        "--cpu-seconds", "1"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "config", "cpu_baseline", "e2e"):
        assert key in d
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_is_bounded_for_many_steps():
    # the driver may pass any --steps/--warmup: the oracle's time stays within
    # the --ref-seconds budget, and the line says how many tokens were timed
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny_fp32", "--steps", "2000", "--warmup", "20",
                        "--ref-seconds", "1"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert time.time() - t0 < 120
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert d["steps"] == 2000 and d["value"] > 0
    assert "over 2000 timed steps" in d["cpu_baseline"]["sample"]
    assert d["ms_per_step"] * 2000 / 1e3 < 5.0  # oracle time summed over the timed steps


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny_fp32", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_roofline_decode_arithmetic():
    """The decode line's roofline: achieved = gate/up weight bytes of the
    activated experts / the gate/up stage time, frac = achieved / peak; the
    whole-FFN and whole-layer figures use all three projections."""
    import bench
    from mixture_experts_gb300 import inputs
    s = inputs.CONFIGS["mixtral_decode"]
    pk = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0}
    avg = [0.01, 0.01, 0.300, 0.150, 0.01]  # ms per stage
    r = bench.roofline(s, "decode", s.T * s.k, 8, avg, 0.5, pk, "measured", "no_such_config")
    per_expert = 2 * s.f * s.d * 2
    assert r["bound"] == "hbm" and r["algorithmic_bytes_per_launch"] == 8 * per_expert
    assert r["achieved"] == pytest.approx(8 * per_expert / 0.300e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0)
    all_bytes = 8 * 3 * s.f * s.d * 2
    assert r["expert_ffn_total"]["bytes"] == all_bytes
    assert r["layer"]["achieved_gbs"] == pytest.approx(all_bytes / 0.5e-3 / 1e9)
    assert r["traffic"] is None  # no committed capture under that name


def test_roofline_prefill_arithmetic():
    """The prefill line's roofline: gate/up FLOP (2 x rows x d x 2f) over the
    gate/up stage time against the sustained and the burst bf16 peaks, the
    down GEMM and the whole layer (2 x rows x 3 x d x f FLOP) beside it."""
    import bench
    from mixture_experts_gb300 import inputs
    s = inputs.CONFIGS["mixtral_prefill"]
    pk = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    rows = s.T * s.k
    avg = [0.02, 0.03, 1.300, 0.650, 0.03]
    r = bench.roofline(s, "prefill", rows, 8, avg, 2.0, pk, "measured", "no_such_config")
    fl = 2.0 * rows * s.d * 2 * s.f
    assert r["bound"] == "tensor" and r["algorithmic_flops_per_launch"] == fl
    assert r["achieved"] == pytest.approx(fl / 1.300e-3 / 1e12)
    assert r["frac_burst"] == pytest.approx(r["achieved"] / 2000.0)
    assert r["frac"] == r["frac_sustained"] == pytest.approx(r["achieved"] / 1800.0)
    assert r["down_gemm"]["achieved"] == pytest.approx(2.0 * rows * s.f * s.d / 0.650e-3 / 1e12)
    assert r["layer"]["flops"] == 2.0 * rows * 3 * s.d * s.f
    # bf16 activations: the prefill forward writes y_perm in bf16
    assert r["overhead_bytes"]["y_perm"] == 2 * rows * s.d * 2


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    """A committed DRAM-traffic figure is reported only while the hash of the
    kernel's sources matches the one recorded with it."""
    import bench
    real = bench.sources_sha("dec")  # the hash of the sources in this tree
    rec = {"mixtral_decode": {"kernel": "k_dec_gateup", "bytes_per_launch": 123,
                              "source_sha": real, "how": "test"},
           "mixtral_prefill": {"kernel": "k_tc_gemm_pair<0>", "bytes_per_launch": 456,
                               "source_sha": "0" * 16, "how": "test"}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the kernel files stay where they are; only the record is the test's
    monkeypatch.setattr(bench, "sources_sha", lambda kind: real if kind == "dec" else "f" * 16)
    assert bench.traffic_record("mixtral_decode", "dec") == 123
    assert bench.traffic_record("mixtral_prefill", "tc") is None  # sources changed
    assert bench.traffic_record("skewed", "tc") is None  # never captured


@pytest.mark.parametrize("wdt,per_weight", [("bf16", 2.0), ("f32", 4.0),
                                            ("i4g128", 0.5 + 2.0 / 128),
                                            ("mxfp8", 1.0 + 1.0 / 32),
                                            ("mxfp4", 0.5 + 1.0 / 32)])
def test_expert_bytes_per_format(wdt, per_weight):
    """One expert's bytes in the handle: 3·f·d weights at the format's width
    plus its scales (int4: a bf16 per 128; MX: an E8M0 byte per 32)."""
    import bench
    from mixture_experts_gb300 import inputs
    s = inputs.MoEShape("x", T=32, d=4096, E=8, k=2, f=14336, wdt=wdt,
                        act="f32" if wdt == "f32" else "bf16")
    assert bench.expert_bytes(s) == 3 * 14336 * 4096 * per_weight
