"""Benchmark of one sparse MoE layer forward on GB300.

Headline workload: the Mixtral-8x7B-shaped layer at a decode batch (T=32,
d=4096, E=8, k=2, d_ff=14336, bf16), whose expert FFN streams the 2.8 GB of
activated expert weights once per forward. At N=1 a default run also measures
the other workloads (prefill, int4, skewed, fp32) and reports each under the
line's "configs" key with its own roofline, stage split, clocks and oracle
sample. Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample

A "step" is one whole forward (router, dispatch, expert FFN, combine) over the
workload's T tokens with inputs resident in HBM. Multi-GPU runs are replicas
(every rank holds the layer and processes its own T tokens; no collective on
the data path), so scaling is weak and value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; achieved HBM GB/s or TC TFLOPS vs chip peak"
STAGES = ["router", "dispatch", "expert_gateup", "expert_down", "combine"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--config", default="mixtral_decode")
    p.add_argument("--impl", default="coli", choices=["coli", "reference"])
    p.add_argument("--ref-seconds", type=float, default=60.0,
                   help="--impl reference: oracle time budget for the whole run, whatever "
                        "--steps and --warmup are")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="budget of the oracle CPU-baseline sample")
    p.add_argument("--sub-cpu-seconds", type=float, default=6.0,
                   help="budget of the oracle sample of each non-headline workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--headline-only", action="store_true",
                   help="measure only --config (default: also every other workload, at N=1)")
    p.add_argument("--experts", type=int, default=0,
                   help="profiling aid: keep the per-expert shapes but use this many experts "
                        "(and T scaled to keep the rows per expert)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_desc(s):
    return (f"{s.name}: T={s.T}, d={s.d}, E={s.E}, k={s.k}, d_ff={s.f}, act={s.act}, "
            f"experts={s.wdt}" + (", Zipf router bias" if s.bias == "zipf" else "")
            + (f", experts in host memory with {s.slots} HBM slots" if s.slots else ""))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def aggregate(local_tokens: int, local_seconds: float, world: int):
    """(total tokens over ranks, max seconds over ranks); needs an initialised
    process group when world > 1."""
    if world == 1:
        return local_tokens, local_seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    n = torch.tensor([float(local_tokens)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return int(n.item()), float(t.item())


# ---------------------------------------------------------------- CPU oracle leg
def host_desc() -> str:
    """CPU model and core count of this host, for the baseline line."""
    model = None
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and ":" in ln:
                    model = ln.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    parts = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1"}
    if model in parts:
        model = f"{parts[model]}, CPU part {model}"
    return f"1 of {os.cpu_count()} cores ({model or 'unknown CPU'})"


def oracle_sample(s, layer, budget_s: float):
    """Time the oracle (as it stands, one thread pinned to one core) on a
    bounded sample of this workload's tokens; returns (tokens/s, tokens timed,
    seconds)."""
    import numpy as np
    import oracle
    oracle.build()
    saved = None
    if hasattr(os, "sched_setaffinity"):
        saved = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {min(saved)})
    try:
        t0 = time.perf_counter()
        oracle.moe_forward(layer, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f, tokens=[0])
        one = max(time.perf_counter() - t0, 1e-6)
        n = int(max(1, min(s.T, budget_s / one)))
        tokens = np.arange(n, dtype=np.int32) % s.T
        t0 = time.perf_counter()
        oracle.moe_forward(layer, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f, tokens=tokens)
        dt = time.perf_counter() - t0
    finally:
        if saved is not None:
            os.sched_setaffinity(0, saved)
    return n / dt, n, dt


def run_reference(args):
    """The reference arm: the oracle (the plain CPU statement of the layer) as
    it stands, one thread pinned to one core. One token's cost is measured
    once; the tokens that fit in --ref-seconds are spread over the timed steps
    (at most the workload's T per step, so a step may hold none when there are
    more steps than tokens), and the warm-up steps only page the oracle in.
    The run therefore ends in about --ref-seconds whatever --steps is; value =
    tokens timed / time spent on them."""
    import numpy as np
    import oracle
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from mixture_experts_gb300 import inputs
    s = inputs.CONFIGS[args.config]
    layer = inputs.make_layer(s, seed=0)
    oracle.build()
    saved = None
    if hasattr(os, "sched_setaffinity"):
        saved = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {min(saved)})

    def timed(n):
        if n <= 0:
            return 0.0
        tokens = np.arange(n, dtype=np.int32) % s.T
        t0 = time.perf_counter()
        oracle.moe_forward(layer, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f, tokens=tokens)
        return time.perf_counter() - t0

    try:
        t_one = max(timed(1), 1e-6)  # also the warm-up: pages the oracle and the layer in
        for _ in range(max(0, args.warmup - 1)):
            timed(0)
        steps = max(1, args.steps)
        budget_tokens = max(1, min(int(args.ref_seconds / t_one), steps * s.T))
        per_step, n_total = [], 0
        for i in range(steps):
            n = (i + 1) * budget_tokens // steps - i * budget_tokens // steps
            per_step.append(timed(n))
            n_total += n
    finally:
        if saved is not None:
            os.sched_setaffinity(0, saved)
    t_total = sum(per_step)
    value = n_total / t_total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_total / len(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": workload_desc(s)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n_total} tokens over {len(per_step)} timed steps (of "
                                   f"the {s.T} tokens of a step), whole layer per token, "
                                   f"one thread on one core",
                         "host": host_desc()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="coli_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, pw = [], [], []
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                pass
            for i, n in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------- traffic record
KERNEL_SOURCES = {
    "dec": ("k_ffn_dec.cu", "common.cuh"),
    "tc": ("k_ffn_tc.cu", "tcgen05.cuh", "common.cuh"),
}


def sources_sha(kind: str) -> str:
    """Hash of the dominant kernel's source files (the .cu and its headers)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "mixture_experts_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(config: str, kind: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, if the kernel's sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh).get(config)
    if not rec:
        return None
    return rec["bytes_per_launch"] if rec.get("source_sha") == sources_sha(kind) else None


# ---------------------------------------------------------------- GPU leg
QNAME = {"i4g128": "int4", "mxfp8": "E4M3", "mxfp4": "E2M1"}  # quantised expert formats


def roofline(s, path, n_rows, active, avg, ms_fwd, pk, pk_src, config_name):
    """Dominant kernel's roofline (gate/up projection: the decode weight
    stream or the prefill grouped GEMM) plus whole-layer figures."""
    gu_ms = avg[2]
    ffn_ms = avg[2] + avg[3]
    if path == "decode":
        if s.wdt == "i4g128":
            per_expert = 2 * s.f * s.d // 2 + 2 * s.f * (s.d // 128) * 2
            all_bytes = active * (3 * s.f * s.d // 2 + 3 * s.f * (s.d // 128) * 2)
        elif s.wdt in ("mxfp8", "mxfp4"):
            per = 1 if s.wdt == "mxfp8" else 2    # elements per byte
            per_expert = 2 * s.f * s.d // per + 2 * s.f * (s.d // 32)
            all_bytes = active * (3 * s.f * s.d // per + 3 * s.f * (s.d // 32))
        else:
            wsz = 4 if s.wdt == "f32" else 2
            per_expert = 2 * s.f * s.d * wsz
            all_bytes = active * 3 * s.f * s.d * wsz
        alg = per_expert * active
        achieved = alg / (gu_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": traffic_record(config_name, "dec"),
                "kernel": ("k_mx_gateup (MX expert gate/up projection + SwiGLU)"
                           if s.wdt in ("mxfp8", "mxfp4") else
                           "k_dec_gateup (expert gate/up projection + SwiGLU)"),
                "algorithmic_bytes_per_launch": alg,
                "unit_work": f"{per_expert} B of gate/up weights per activated expert x "
                             f"{active} activated experts",
                "peak_source": f"{pk_src} hbm_gbs"}
        roof["expert_ffn_total"] = {
            "bytes": all_bytes, "achieved_gbs": all_bytes / (ffn_ms / 1e3) / 1e9,
            "frac": all_bytes / (ffn_ms / 1e3) / 1e9 / pk["hbm_gbs"]}
        # the layer's figure: activated-expert weight bytes over the whole forward
        roof["layer"] = {"achieved_gbs": all_bytes / (ms_fwd / 1e3) / 1e9,
                         "frac": all_bytes / (ms_fwd / 1e3) / 1e9 / pk["hbm_gbs"]}
    else:
        flops = 2.0 * n_rows * s.d * 2 * s.f
        achieved = flops / (gu_ms / 1e3) / 1e12
        burst = pk["bf16_tflops"]
        sust = pk.get("bf16_tflops_sustained", burst)
        roof = {"bound": "tensor", "achieved": achieved, "peak": sust, "unit": "TFLOP/s",
                "frac": achieved / sust, "frac_burst": achieved / burst,
                "frac_sustained": achieved / sust,
                "traffic": traffic_record(config_name, "tc"),
                "kernel": (f"k_tcq_gemm<{QNAME[s.wdt]}> (gate/up grouped GEMM, weights "
                           "dequantised into tensor memory, + SwiGLU)" if s.wdt in QNAME else
                           "k_tc_gemm_pair (gate/up grouped GEMM on CTA pairs + SwiGLU)"),
                "algorithmic_flops_per_launch": flops,
                "unit_work": f"2 x {n_rows} rows x d={s.d} x 2f={2 * s.f} FLOP",
                "peak_source": f"{pk_src} bf16_tflops_sustained (burst {burst})"}
        dn_flops = 2.0 * n_rows * s.f * s.d
        dn = dn_flops / (avg[3] / 1e3) / 1e12
        roof["down_gemm"] = {"achieved": dn, "frac_burst": dn / burst, "frac_sustained": dn / sust}
        layer_flops = 2.0 * n_rows * 3 * s.d * s.f
        lay = layer_flops / (ms_fwd / 1e3) / 1e12
        roof["layer"] = {"flops": layer_flops, "achieved_tflops": lay, "frac_burst": lay / burst,
                         "frac_sustained": lay / sust}
    # intermediates are not algorithmic bytes: x_perm (written by dispatch,
    # read by gate/up), H (written and read), y_perm (fp32, written by down,
    # read by combine), listed separately per forward; the decode path with
    # bf16/int4 experts reads token rows of x directly and writes no x_perm
    asz = 4 if s.act == "f32" else 2
    xperm = 0 if (path == "decode" and s.wdt != "f32") else 2 * n_rows * s.d * asz
    if path == "decode" and s.wdt in ("mxfp8", "mxfp4"):
        xperm = 2 * s.T * s.d * 2  # the fp16 copy of the token rows
    # the prefill path writes y_perm in bf16 for bf16 activations
    ysz = 2 if (path == "prefill" and s.act == "bf16") else 4
    roof["overhead_bytes"] = {
        "x_perm": xperm, "H": 2 * n_rows * s.f * (4 if s.wdt == "f32" else 2),
        "y_perm": 2 * n_rows * s.d * ysz}
    return roof


def expert_bytes(s) -> int:
    """Bytes of one expert's three projections in the handle (weights plus
    their scales): bf16 / f32 elements, int4 nibbles with a bf16 scale per 128,
    MX codes with an E8M0 byte per 32."""
    n = 3 * s.f * s.d  # weights of gate, up and down
    if s.wdt == "i4g128":
        return n // 2 + (n // 128) * 2
    if s.wdt == "mxfp8":
        return n + n // 32
    if s.wdt == "mxfp4":
        return n // 2 + n // 32
    return n * (4 if s.wdt == "f32" else 2)


def tier_record(s, layer, counts, avg, pk, torch):
    """Residency tier: bytes each forward reads from HBM slots and from host
    memory over NVLink-C2C, the FFN's effective host-read rate (host bytes /
    (FFN time - HBM bytes at the HBM peak)), and a pinned host -> device copy
    of 1 GiB timed in the same process as the reference rate."""
    slots, _ = layer.residency()
    per = expert_bytes(s)
    active = [e for e in range(s.E) if counts[e] > 0]
    hbm = sum(per for e in active if slots[e] >= 0)
    host = sum(per for e in active if slots[e] < 0)
    ffn_s = (avg[2] + avg[3]) / 1e3
    c2c = host / max(ffn_s - hbm / (pk["hbm_gbs"] * 1e9), 1e-9) / 1e9
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8).pin_memory()
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        dst.copy_(src, non_blocking=True)
    b.record()
    b.synchronize()
    h2d = 3 * n / (a.elapsed_time(b) / 1e3) / 1e9
    del src, dst
    return {"expert_slots": s.slots, "max_promotions": s.promotions,
            "active_resident": sum(1 for e in active if slots[e] >= 0),
            "active_streamed": sum(1 for e in active if slots[e] < 0),
            "bytes_from_hbm": hbm, "bytes_from_host": host,
            "ffn_host_read_gbs": c2c, "pinned_h2d_copy_gbs": h2d,
            "frac_of_h2d_copy": c2c / h2d}


def measure(s, steps, warmup, world, rank, local, cpu_seconds, with_e2e=True,
            config_name=None):
    """Times `steps` forwards of workload `s` (inputs resident in HBM) and
    returns the per-workload record: value, stage split, roofline, clocks,
    end-to-end figure through the host-buffer API and the oracle sample."""
    import torch
    import mixture_experts_gb300 as moe
    from mixture_experts_gb300 import inputs

    host = inputs.make_layer(s, seed=0)
    if rank > 0:  # replicas: same weights, this rank's own tokens
        host["x"] = inputs.random_rows(s.T, s.d, s.act_code, seed=1000 + rank)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in host.items()}
    layer = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev,
                         expert_slots=s.slots, max_promotions=s.promotions)
    x = dev["x"]
    dev = None  # the handle holds its own copy of the weights
    torch.cuda.empty_cache()
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    path = {moe.PATH_DECODE: "decode", moe.PATH_PREFILL: "prefill"}[layer.path_for(s.T)]

    weight_bytes = sum(v.numel() * v.element_size() for k, v in host.items()
                       if k.startswith(("w_gate", "w_up", "w_down", "s_")) and v is not None)
    flush = weight_bytes < 2 * L2_BYTES
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda") if flush else None

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, warmup)):
        layer(x, y)
    barrier()

    def busy(seconds: float) -> int:
        """Untimed forwards of the same workload for about `seconds`."""
        n, t_end = 0, time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(8):
                layer(x, y)
            torch.cuda.synchronize()
            n += 8
        return n

    # clocks are sampled under load only: the sampler starts while untimed
    # forwards run, and a timed region shorter than the sampling needs is
    # followed by more of them (stated in the record's clocks.window)
    clocks = ClockSampler(local)
    clocks.start()
    pre = busy(0.5)
    barrier()

    def timed_pass() -> float:
        """K forwards between CUDA events on the launching stream (L2 flushed
        before each one when the inputs fit in L2); returns milliseconds."""
        barrier()
        if flush:
            per = []
            for _ in range(steps):
                scrub.zero_()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                layer(x, y)
                b.record(stream)
                b.synchronize()
                per.append(a.elapsed_time(b))
            ms = sum(per)
        else:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(steps):
                layer(x, y)
            b.record(stream)
            barrier()
            ms = a.elapsed_time(b)
        barrier()
        return ms

    # ---- timed region: K forwards, no instrumentation inside
    elapsed_ms = timed_pass()
    # ---- the same K forwards again with per-stage CUDA events, for the split
    moe.coli_moe_set_timing(layer.h, True)
    moe.coli_moe_stage_times(layer.h)  # reset sums
    timed_pass()
    stage_ms, n_fwd, n_launch = moe.coli_moe_stage_times(layer.h)
    moe.coli_moe_set_timing(layer.h, False)
    post = busy(0.5 - elapsed_ms / 1e3) if elapsed_ms < 500.0 else 0
    clk = clocks.stop()
    clk["window"] = (f"{pre} untimed forwards while the sampler started, the timed region, "
                     "the same forwards again with per-stage events"
                     + (f", then {post} more untimed forwards (the timed region lasted "
                        f"{elapsed_ms:.1f} ms)" if post else ""))
    tokens, seconds = aggregate(s.T * steps, elapsed_ms / 1e3, world)
    value = tokens / seconds

    pk, pk_src = peaks()
    dbg = layer.debug(s.T)
    counts = dbg["counts"].cpu().numpy()
    active = int((counts > 0).sum())
    n_rows = int(counts.sum())
    avg = [m / max(1, n_fwd) for m in stage_ms]
    roof = roofline(s, path, n_rows, active, avg, elapsed_ms / steps, pk, pk_src,
                    config_name or s.name)

    if s.slots:
        roof["tier"] = tier_record(s, layer, counts, avg, pk, torch)
    rec = {"workload": workload_desc(s), "path": path, "value": value, "unit": "tokens/s",
           "steps": steps, "warmup": max(3, warmup), "ms_per_step": elapsed_ms / steps,
           "l2": ("L2 flushed between steps" if flush else
                  f"inputs larger than L2: {weight_bytes / 1e9:.2f} GB of expert weights "
                  f"streamed per step"),
           "active_experts": active, "roofline": roof,
           "stage_ms": dict(zip(STAGES, [round(m, 5) for m in avg])),
           "gpu_launches": int(n_launch * steps / max(1, n_fwd)), "clocks": clk}

    if with_e2e:
        # end to end through the public API with host buffers (pinned)
        xh = host["x"].pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        for _ in range(3):
            layer.forward_host(xh, yh)
        e2e_steps = max(10, min(steps, 500))
        barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            layer.forward_host(xh, yh)
        e2e_s = time.perf_counter() - t0
        e_tokens, e_seconds = aggregate(s.T * e2e_steps, e2e_s, world)
        io_bytes = s.T * s.d * (4 if s.act == "f32" else 2)
        rec["e2e"] = {"value": e_tokens / e_seconds, "unit": "tokens/s",
                      "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes}
    layer.close()
    del x, y, scrub
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and cpu_seconds > 0:
        tps, n, dt = oracle_sample(s, host, cpu_seconds)
        rec["cpu_baseline"] = {
            "value": tps, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} of the {s.T} tokens of one step, whole layer per token "
                      f"({dt:.1f} s, one thread)",
            "host": host_desc()}
    else:
        rec["cpu_baseline"] = None
    return rec


# the other workloads measured beside the headline one in a default run:
# the remaining configurations, then the quantised-expert and residency layers
EXTRA = ["mixtral_prefill", "fine_int4", "skewed", "tiny_fp32", "mixtral_prefill_int4",
         "mixtral_prefill_mxfp8", "mixtral_decode_mxfp8", "fine_mxfp4", "mixtral_decode_tier"]


def sub_steps(s, K: int) -> int:
    """Timed forwards for a non-headline workload: at least K, and enough
    for about 0.3 s of timed work (capped), from a rough cost model."""
    flops = 2.0 * s.T * s.k * 3 * s.d * s.f
    bpw = {"i4g128": 0.53, "mxfp8": 1.03, "mxfp4": 0.53}.get(s.wdt, 2.0)  # bytes per weight
    if s.slots:
        bpw *= 8.0  # most experts read over C2C
    est_ms = max(0.02, flops / 1.2e15 * 1e3,
                 3 * s.d * s.f * min(s.E, s.T * s.k) * bpw / 5.0e12 * 1e3)
    return int(max(K, min(400, 300.0 / est_ms)))


def run_coli(args):
    import torch
    import mixture_experts_gb300 as moe
    from mixture_experts_gb300 import inputs

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    moe.build()
    s = inputs.CONFIGS[args.config]
    if args.experts:
        s = s.with_(name=f"{s.name}[E={args.experts}]", E=args.experts,
                    T=max(1, s.T * args.experts // s.E), k=min(s.k, args.experts))
    cpu_s = 0 if (args.no_cpu_baseline or world > 1) else args.cpu_seconds
    head = measure(s, args.steps, args.warmup, world, rank, local, cpu_s,
                   config_name=args.config)

    others = {}
    if world == 1 and not args.headline_only and not args.experts:
        for name in EXTRA:
            if name == args.config:
                continue
            so = inputs.CONFIGS[name]
            rec = measure(so, sub_steps(so, args.steps), args.warmup, world, rank, local,
                          0 if args.no_cpu_baseline else args.sub_cpu_seconds, with_e2e=False,
                          config_name=name)
            rec.pop("e2e", None)
            others[name] = rec

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if s.act == "bf16" else "f32",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
            "config": {"workload": head["workload"], "path": head["path"],
                       "parallelism": f"replicas x{world}", "l2": head["l2"],
                       "active_experts": head["active_experts"]},
            "roofline": head["roofline"],
            "stage_ms": head["stage_ms"],
            "cpu_baseline": head["cpu_baseline"],
            "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "clocks": head["clocks"],
        }
        if others:
            line["configs"] = others
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return line


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_coli(args)


if __name__ == "__main__":
    main()
