"""CUDA path vs the oracle, element by element, through the C ABI (GPU)."""
import os

import numpy as np
import pytest
import torch

import mixture_experts_gb300 as moe
import oracle
from mixture_experts_gb300 import inputs
from parity import (TOL, check_layer, check_routing, cuda_layer, host_dict, make_handle,
                    oracle_routing, rel_err, y_to_f64)

pytestmark = pytest.mark.gpu

S = inputs.MoEShape
SMALL = {
    "tiny_fp32": inputs.CONFIGS["tiny_fp32"],
    "decode_bf16": S("decode_bf16", T=24, d=512, E=8, k=2, f=384),
    "prefill_bf16": S("prefill_bf16", T=600, d=512, E=8, k=2, f=768),
    "int4": S("int4", T=40, d=1024, E=16, k=4, f=256, wdt="i4g128"),
    "int4_big_groups": S("int4_big_groups", T=70, d=256, E=2, k=1, f=256, wdt="i4g128"),
    "skew_small": S("skew_small", T=2048, d=256, E=64, k=4, f=128, bias="zipf"),
    "e256_sparse": S("e256_sparse", T=50, d=256, E=256, k=8, f=128),
    "e1_k1": S("e1_k1", T=5, d=128, E=1, k=1, f=64),
    "k_eq_e": S("k_eq_e", T=9, d=128, E=4, k=4, f=64),
    "hot_expert": S("hot_expert", T=50, d=256, E=8, k=2, f=128, bias="hot0"),
    "one_token": S("one_token", T=1, d=256, E=8, k=2, f=128),
    "fp32_e64": S("fp32_e64", T=33, d=192, E=64, k=3, f=64, act="f32", wdt="f32"),
    # int4 experts with hundreds of rows each: the tcgen05 grouped GEMM with
    # the weights dequantised in shared memory
    "int4_prefill": S("int4_prefill", T=600, d=512, E=4, k=2, f=384, wdt="i4g128"),
    # block-scaled experts (decode path, fp16 MMAs): one and two token tiles
    # per pass, several passes per expert
    "mxfp8": S("mxfp8", T=40, d=512, E=8, k=2, f=256, wdt="mxfp8"),
    "mxfp4": S("mxfp4", T=60, d=384, E=6, k=3, f=384, wdt="mxfp4"),
    "mxfp8_bias": S("mxfp8_bias", T=90, d=256, E=16, k=4, f=128, wdt="mxfp8", bias="zipf"),
    # MX experts with hundreds of rows each: the tensor-core GEMM with the
    # weights dequantised into tensor memory (ragged K: 384 = one and a half
    # E2M1 slots; f = 640: odd weight-tile count)
    "mxfp8_prefill": S("mxfp8_prefill", T=700, d=384, E=5, k=2, f=640, wdt="mxfp8"),
    "mxfp4_prefill": S("mxfp4_prefill", T=800, d=384, E=6, k=3, f=640, wdt="mxfp4"),
}


@pytest.fixture(scope="module", autouse=True)
def built():
    moe.build()
    assert torch.cuda.is_available()


def run_layer(s, lay, path=moe.PATH_AUTO):
    dev = cuda_layer(lay)
    layer = make_handle(s, dev, path=path)
    y = layer(dev["x"])
    dbg = layer.debug(s.T)
    torch.cuda.synchronize()
    assert layer.status() == moe.COLI_OK
    return layer, y, host_dict(dbg)


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_small(name):
    s = SMALL[name]
    lay = inputs.make_layer(s, seed=11)
    _, y, dbg = run_layer(s, lay)
    check_layer(s, lay, y, dbg)


@pytest.mark.parametrize("name", ["decode_bf16", "prefill_bf16", "skew_small", "int4_prefill",
                                  "mxfp8_prefill", "mxfp4_prefill"])
def test_paths_agree(name):
    """Decode (weight streaming) and prefill (tcgen05 grouped GEMM) paths give
    the same routing and outputs within rounding on the same inputs."""
    s = SMALL[name]
    lay = inputs.make_layer(s, seed=12)
    _, y_dec, dbg_dec = run_layer(s, lay, path=moe.PATH_DECODE)
    layer_pre, y_pre, dbg_pre = run_layer(s, lay, path=moe.PATH_PREFILL)
    assert layer_pre.path_for(s.T) == moe.PATH_PREFILL
    for key in ("topk_idx", "counts", "offsets", "row_token", "assign_row"):
        assert np.array_equal(dbg_dec[key], dbg_pre[key]), key
    check_layer(s, lay, y_dec, dbg_dec)
    check_layer(s, lay, y_pre, dbg_pre)
    assert rel_err(y_to_f64(y_pre), y_to_f64(y_dec)) <= TOL[s.wdt]


def test_deterministic_and_host_api():
    s = SMALL["int4"]
    lay = inputs.make_layer(s, seed=13)
    dev = cuda_layer(lay)
    layer = make_handle(s, dev)
    y1 = layer(dev["x"]).clone()
    y2 = layer(dev["x"]).clone()
    assert torch.equal(y1, y2)
    xh = lay["x"].pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    layer.forward_host(xh, yh)
    assert torch.equal(yh, y1.cpu())


FULL = ["tiny_fp32", "mixtral_decode", "mixtral_prefill", "fine_int4", "skewed"]


@pytest.mark.parametrize("name", FULL)
def test_full_config(name):
    """The five configurations at full size, in the launch configuration the
    benchmark times: routing and dispatch of every token, and the output of
    every token (near-ties excepted) against the oracle, whose token list is
    split over the host's cores (bit-identical to one thread)."""
    s = inputs.CONFIGS[name]
    lay = inputs.make_layer(s, seed=0)
    layer, y, dbg = run_layer(s, lay)
    err, near = check_layer(s, lay, y, dbg, threads=os.cpu_count() or 1)
    print(f"{name}: path={layer.path_for(s.T)} rel_err={err:.3e} near_ties={near} "
          f"tokens_checked={s.T - near}")


@pytest.mark.parametrize("name", ["mixtral_decode_mxfp8", "fine_mxfp4"])
def test_full_mx_layers(name):
    """The decode layers with MX experts at full size: every token."""
    s = inputs.CONFIGS[name]
    lay = inputs.make_layer(s, seed=0)
    layer, y, dbg = run_layer(s, lay)
    assert layer.path_for(s.T) == moe.PATH_DECODE
    err, near = check_layer(s, lay, y, dbg, threads=os.cpu_count() or 1)
    print(f"{name}: rel_err={err:.3e} near_ties={near} tokens_checked={s.T - near}")


def test_full_mxfp8_prefill_layer_sampled():
    """The Mixtral-shaped layer with MXFP8 experts at the prefill batch:
    routing and dispatch of every token, outputs of 512 seeded tokens."""
    s = inputs.CONFIGS["mixtral_prefill_mxfp8"]
    lay = inputs.make_layer(s, seed=0)
    layer, y, dbg = run_layer(s, lay)
    assert layer.path_for(s.T) == moe.PATH_PREFILL
    err, near = check_layer(s, lay, y, dbg, threads=os.cpu_count() or 1, sample=512)
    print(f"mixtral_prefill_mxfp8: rel_err={err:.3e} near_ties={near}")


def test_full_int4_prefill_layer_sampled():
    """The Mixtral-shaped layer with int4 experts at the prefill batch (the
    bench's int4 tensor-core workload): routing and dispatch of every token,
    outputs of 512 seeded tokens (every token would take the oracle ~10 min)."""
    s = inputs.CONFIGS["mixtral_prefill_int4"]
    lay = inputs.make_layer(s, seed=0)
    layer, y, dbg = run_layer(s, lay)
    assert layer.path_for(s.T) == moe.PATH_PREFILL
    err, near = check_layer(s, lay, y, dbg, threads=os.cpu_count() or 1, sample=512)
    print(f"mixtral_prefill_int4: rel_err={err:.3e} near_ties={near} tokens_checked=514")


# ---------------------------------------------------------------- stages
def _stage_layer(s, seed):
    lay = inputs.make_layer(s, seed=seed)
    return lay, cuda_layer(lay)


@pytest.mark.parametrize("E,k,act,bias", [(8, 2, "bf16", False), (32, 4, "f32", True),
                                          (64, 4, "bf16", True), (256, 8, "bf16", False),
                                          (200, 7, "f32", False)])
def test_stage_route_topk(E, k, act, bias):
    s = S("route", T=77, d=320, E=E, k=k, f=64, act=act, wdt=act,
          bias="zipf" if bias else "none")
    lay, dev = _stage_layer(s, 21)
    T, d = s.T, s.d
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    gap = torch.empty(T, dtype=torch.float32, device="cuda")
    nb = moe.coli_route_scratch_bytes(T, d, E)
    scratch = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    rc = moe.coli_route_topk(dev["x"], dev["w_router"], dev["b_router"], T, d, E, k, s.act_code,
                             idx, w, gap, scratch, nb)
    assert rc == 0, moe.last_error()
    r_idx, r_w, r_gap, r_inner = oracle_routing(s, lay)
    near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), r_idx, r_w, r_gap, r_inner)
    g = gap.cpu().numpy()
    fin = ~near & np.isfinite(r_gap)
    # a gap is a difference of two fp32 logits: its error bounds the logit
    # accumulation error (tensor-core path for bf16 with E > 32)
    assert np.max(np.abs(g[fin] - r_gap[fin]), initial=0.0) <= 3e-6


@pytest.mark.parametrize("E,k,bias,d", [(3, 1, False, 384), (8, 2, True, 384),
                                        (24, 3, False, 384), (40, 5, True, 384),
                                        (48, 3, True, 384), (64, 4, True, 384),
                                        (64, 4, True, 2048), (96, 2, False, 384),
                                        (112, 6, True, 384), (128, 8, False, 768),
                                        (200, 7, False, 384), (256, 8, False, 384)])
def test_stage_route_topk_many_tokens(E, k, bias, d):
    """bf16 batches of 1024+ tokens take a one-launch router: E <= 32, 32
    tokens per block with mma.sync logits; E a multiple of 16 up to 128, 128
    tokens per CTA with tcgen05 logits in tensor memory (d = 2048 wraps its
    stage ring and accumulator buffers many times); other E, 64 tokens per
    block with mma.sync. Expert counts that fill one, some or all of a block's
    warps, a ragged last block, with and without bias."""
    T = 1100
    s = S("route_many", T=T, d=d, E=E, k=k, f=64, bias="zipf" if bias else "none")
    lay, dev = _stage_layer(s, 22)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    gap = torch.empty(T, dtype=torch.float32, device="cuda")
    nb = moe.coli_route_scratch_bytes(T, d, E)
    scratch = torch.empty(max(nb, 1), dtype=torch.uint8, device="cuda")
    rc = moe.coli_route_topk(dev["x"], dev["w_router"], dev["b_router"], T, d, E, k, s.act_code,
                             idx, w, gap, scratch, nb)
    assert rc == 0, moe.last_error()
    r_idx, r_w, r_gap, r_inner = oracle_routing(s, lay)
    near = check_routing(idx.cpu().numpy(), w.cpu().numpy(), r_idx, r_w, r_gap, r_inner)
    g = gap.cpu().numpy()
    fin = ~near & np.isfinite(r_gap)
    assert np.max(np.abs(g[fin] - r_gap[fin]), initial=0.0) <= 3e-6
    assert moe.coli_device_status() == moe.COLI_OK


@pytest.mark.parametrize("T,E,k,act", [(37, 8, 2, "bf16"), (300, 64, 4, "f32"),
                                       (5000, 64, 4, "bf16"), (3000, 256, 8, "bf16"),
                                       (1, 1, 1, "bf16")])
def test_stage_permute(T, E, k, act):
    d = 128
    idx = inputs.random_assignments(T, E, k, seed=T).cuda()
    x = inputs.random_rows(T, d, inputs.DTYPE_CODE[act], seed=3).cuda()
    n = T * k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.empty(n, dtype=torch.int32, device="cuda")
    assign_row = torch.empty(n, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(n, d, dtype=x.dtype, device="cuda")
    nb = moe.coli_permute_scratch_bytes(T, k, E)
    scratch = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    rc = moe.coli_permute(idx, x, T, d, E, k, inputs.DTYPE_CODE[act], counts, offsets, row_token,
                          assign_row, x_perm, scratch, nb)
    assert rc == 0, moe.last_error()
    c, o, rt, ar = oracle.dispatch(idx.cpu().numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(row_token.cpu().numpy(), rt)
    assert np.array_equal(assign_row.cpu().numpy(), ar)
    assert torch.equal(x_perm.cpu(), x.cpu()[torch.from_numpy(rt).long()])
    assert moe.coli_device_status() == 0


@pytest.mark.parametrize("T,E,k", [(37, 8, 2), (5000, 64, 4)])
def test_stage_permute_without_row_copy(T, E, k):
    # x_perm NULL: the maps alone, x never read (the forward's decode path)
    idx = inputs.random_assignments(T, E, k, seed=T + 1).cuda()
    n = T * k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_token = torch.empty(n, dtype=torch.int32, device="cuda")
    assign_row = torch.empty(n, dtype=torch.int32, device="cuda")
    nb = moe.coli_permute_scratch_bytes(T, k, E)
    scratch = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    rc = moe.coli_permute(idx, None, T, 128, E, k, moe.BF16, counts, offsets, row_token,
                          assign_row, None, scratch, nb)
    assert rc == 0, moe.last_error()
    c, o, rt, ar = oracle.dispatch(idx.cpu().numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(row_token.cpu().numpy(), rt)
    assert np.array_equal(assign_row.cpu().numpy(), ar)
    assert moe.coli_device_status() == 0


@pytest.mark.parametrize("name", ["decode_bf16", "int4", "tiny_fp32", "mxfp8", "mxfp4"])
def test_stage_expert_ffn(name):
    s = SMALL[name]
    lay, dev = _stage_layer(s, 31)
    layer = make_handle(s, dev)
    g = np.random.default_rng(5)
    counts = g.multinomial(s.T * s.k, np.ones(s.E) / s.E)
    counts[0] = 0  # an empty expert
    n = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    xp = inputs.random_rows(n, s.d, s.act_code, seed=6)
    y = torch.empty(n, s.d, dtype=torch.float32, device="cuda")
    rc = moe.coli_expert_ffn(layer.h, xp.cuda(), torch.from_numpy(offsets).cuda(), n, y)
    assert rc == 0, moe.last_error()
    got = y.cpu().numpy().astype(np.float64)
    ref = np.zeros_like(got)
    for e in range(s.E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.expert_ffn(xp[a:b], s.act_code, lay, e, s.d, s.f, s.w_code)
    assert rel_err(got, ref) <= TOL[s.wdt]


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_stage_combine(out):
    T, k, d = 45, 3, 256
    y_perm = inputs.random_rows(T * k, d, inputs.F32, seed=8)
    perm = torch.from_numpy(np.random.default_rng(9).permutation(T * k).astype(np.int32))
    w = inputs.random_gates(T, k, seed=10)
    code = inputs.DTYPE_CODE[out]
    y = torch.empty(T, d, dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
    rc = moe.coli_combine(y_perm.cuda(), perm.cuda(), w.cuda(), T, k, d, code, y)
    assert rc == 0, moe.last_error()
    y64, yo = oracle.combine(y_perm, perm, w, T, k, d, code)
    if out == "f32":
        assert rel_err(y.cpu().numpy(), y64) <= 1e-6
    else:
        # bf16 outputs: at most one unit in the last place from the oracle's rounding
        got = y.cpu().view(torch.int16).numpy().astype(np.int32)
        ref = yo.view(np.int16).astype(np.int32)
        assert np.max(np.abs(got - ref)) <= 1


# ---------------------------------------------------------------- edge cases
EDGE = {
    # tensor-core path with a half-filled last column tile (f % 128 == 64) and
    # a down projection whose last tile runs past d (d % 256 != 0)
    "tc_tails": S("tc_tails", T=300, d=320, E=4, k=2, f=192),
    "min_dims": S("min_dims", T=20, d=64, E=3, k=3, f=64),
    "e256_prefill": S("e256_prefill", T=2048, d=128, E=256, k=8, f=128),
    "int4_min": S("int4_min", T=12, d=128, E=5, k=2, f=128, wdt="i4g128"),
    # int4 on the tensor cores: one scale group along d (K = 128), a down
    # projection whose last 256-column tile is half past the weights, and an
    # odd number of gate/up column tiles
    "int4_tc_tails": S("int4_tc_tails", T=400, d=384, E=3, k=2, f=640, wdt="i4g128"),
}


@pytest.mark.parametrize("name", list(EDGE))
@pytest.mark.parametrize("path", [moe.PATH_DECODE, moe.PATH_PREFILL])
def test_edge_shapes(name, path):
    s = EDGE[name]
    lay = inputs.make_layer(s, seed=41)
    _, y, dbg = run_layer(s, lay, path=path)
    check_layer(s, lay, y, dbg)


def test_int4_prefill_many_tiles_per_cta():
    """int4 experts on the tcgen05 path with several tiles per CTA (the
    accumulator double buffer wraps, the converters cross tile boundaries):
    every token against the oracle."""
    s = S("int4_wrap", T=4096, d=1024, E=8, k=2, f=2048, wdt="i4g128")
    lay = inputs.make_layer(s, seed=43)
    layer, y, dbg = run_layer(s, lay)
    assert layer.path_for(s.T) == moe.PATH_PREFILL
    err, near = check_layer(s, lay, y, dbg, threads=os.cpu_count() or 1)
    print(f"int4_wrap: rel_err={err:.3e} near_ties={near}")


@pytest.mark.parametrize("wdt", ["mxfp8", "mxfp4"])
def test_mx_prefill_many_tiles_per_cta(wdt):
    """MX experts on the tensor-core path with several tiles per CTA (the raw
    slots and tensor-memory stages wrap across tiles): every token."""
    s = S(f"{wdt}_wrap", T=3000, d=1024, E=8, k=2, f=1536, wdt=wdt)
    lay = inputs.make_layer(s, seed=44)
    layer, y, dbg = run_layer(s, lay)
    assert layer.path_for(s.T) == moe.PATH_PREFILL
    err, near = check_layer(s, lay, y, dbg, threads=os.cpu_count() or 1)
    print(f"{s.name}: rel_err={err:.3e} near_ties={near}")


@pytest.mark.parametrize("wdt", ["mxfp8", "mxfp4"])
def test_mx_prefill_special_values(wdt):
    """MX weights outside the converters' fast range, on the tensor-core
    path: block scales of 2^16 and 2^30 and a NaN scale (and, for E4M3, NaN
    codes) take the exact fp32 conversion; outputs are NaN exactly where the
    oracle's are and match it elsewhere."""
    s = S(f"{wdt}_special", T=300, d=256, E=4, k=2, f=256, wdt=wdt)
    lay = inputs.make_layer(s, seed=45)
    sg = lay["s_gate"].clone()
    sg[0, 3, 1] = 127 + 16          # one gate block of expert 0 scaled by 2^16 more
    sg[1, 5, 0] = 127 + 30
    lay["s_gate"] = sg
    sd = lay["s_down"].clone()
    sd[2, 7, 2] = 255               # NaN scale: one block of down row 7 of expert 2
    lay["s_down"] = sd
    if wdt == "mxfp8":
        wd = lay["w_down"].clone()
        wd[3, 11, 40] = 0x7F        # E4M3 NaN code in down row 11 of expert 3
        lay["w_down"] = wd
    layer, y, dbg = run_layer(s, lay, path=moe.PATH_PREFILL)
    assert layer.path_for(s.T) == moe.PATH_PREFILL
    idx, w, gap, inner = oracle_routing(s, lay)
    near = check_routing(dbg["topk_idx"], dbg["topk_w"], idx, w, gap, inner)
    tokens = np.nonzero(~near)[0].astype(np.int32)
    ref = oracle.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f,
                             tokens=tokens)["y_f64"]
    got = y_to_f64(y)[tokens]
    assert np.isnan(ref).any()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    err = np.max(np.abs(got[fin] - ref[fin])) / np.max(np.abs(ref[fin]))
    assert err <= TOL[wdt], err


def test_empty_batch_is_a_no_op():
    s = SMALL["decode_bf16"]
    lay = inputs.make_layer(s, seed=42)
    dev = cuda_layer(lay)
    layer = make_handle(s, dev)
    y = torch.full_like(dev["x"], 7.0)
    assert moe.coli_moe_forward(layer.h, dev["x"], 0, y) == moe.COLI_OK
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    # stage functions accept T == 0 as well
    z = torch.empty(0, dtype=torch.int32, device="cuda")
    assert moe.coli_route_topk(dev["x"], dev["w_router"], None, 0, s.d, s.E, s.k, s.act_code,
                               z, z) == moe.COLI_OK
    assert moe.coli_combine(dev["x"], z, z, 0, s.k, s.d, s.act_code, y) == moe.COLI_OK
    assert layer.status() == moe.COLI_OK
