"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself (CPU only)."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import softmax

from mixture_experts_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- selection
@pytest.mark.parametrize("k", [1, 2, 4, 8])
def test_select_exhaustive_tie_patterns(oracle_mod, k):
    """All 3^8 integer logit patterns over E=8 (ties everywhere): the selected
    set and slot order equal a library sort by (-logit, index)."""
    pats = np.array(list(itertools.product([0.0, 1.0, 2.0], repeat=8)), np.float32)
    idx, w, gap, inner = oracle_mod.select_topk(pats, k)
    for t in range(0, len(pats)):
        order = sorted(range(8), key=lambda e: (-pats[t, e], e))
        assert list(idx[t]) == order[:k]
        expect_gap = math.inf if k == 8 else pats[t, order[k - 1]] - pats[t, order[k]]
        assert gap[t] == expect_gap
    assert np.all(np.diff(w, axis=1) <= 0)


def test_select_distinct_ids_and_gap(oracle_mod):
    rng = np.random.default_rng(1)
    logits = rng.normal(size=(500, 64)).astype(np.float32)
    idx, w, gap, inner = oracle_mod.select_topk(logits, 6)
    for t in range(500):
        assert len(set(idx[t])) == 6 and idx[t].min() >= 0 and idx[t].max() < 64
        s = np.sort(logits[t])[::-1]
        assert gap[t] == s[5] - s[6]
        assert inner[t] == np.min(s[:5] - s[1:6])


# -------------------------------------------------------------------- gates
def test_gates_k2_closed_form(oracle_mod):
    """k=2: g0 = logistic(l0 - l1), g1 = 1 - g0."""
    rng = np.random.default_rng(2)
    logits = (rng.normal(size=(300, 8)) * 3).astype(np.float32)
    idx, w, _, _ = oracle_mod.select_topk(logits, 2)
    for t in range(300):
        l0, l1 = float(logits[t, idx[t, 0]]), float(logits[t, idx[t, 1]])
        g0 = 1.0 / (1.0 + math.exp(l1 - l0))
        assert abs(w[t, 0] - g0) <= 6e-8 and abs(w[t, 1] - (1 - g0)) <= 6e-8


def test_gates_equal_library_softmax_renormalised(oracle_mod):
    """Softmax over all E (scipy), restricted to the top-k and renormalised."""
    rng = np.random.default_rng(3)
    logits = (rng.normal(size=(200, 32)) * 2).astype(np.float32)
    for k in (1, 3, 8, 32):
        idx, w, _, _ = oracle_mod.select_topk(logits, k)
        for t in range(200):
            p = softmax(logits[t].astype(np.float64))
            ref = p[idx[t]] / p[idx[t]].sum()
            assert np.max(np.abs(w[t] - ref)) <= 1e-7
        if k == 1:
            assert np.all(w == 1.0)
        s = w.sum(axis=1, dtype=np.float32)
        assert np.all(np.abs(s - 1) <= 1e-6) and np.all(w > 0)


# ------------------------------------------------------------------- logits
@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_router_logits_match_library_matmul(oracle_mod, act):
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rng.normal(size=(40, 320)).astype(np.float32))
    w = torch.from_numpy((rng.normal(size=(12, 320)) * 0.02).astype(np.float32))
    b = torch.from_numpy(rng.normal(size=12).astype(np.float32))
    code = inputs.DTYPE_CODE[act]
    if act == "bf16":
        x, w = x.to(torch.bfloat16), w.to(torch.bfloat16)
    got = oracle_mod.router_logits(x, code, w, b, 40, 320, 12)
    ref = (x.double() @ w.double().T).float() + b  # fp32 add of the bias
    ulp = np.spacing(np.abs(ref.numpy()))
    assert np.all(np.abs(got - ref.numpy()) <= ulp + 1e-30)


# ----------------------------------------------------------------- dispatch
def test_dispatch_equals_stable_argsort(oracle_mod):
    for (T, E, k, seed) in [(1, 1, 1, 0), (37, 8, 2, 1), (300, 64, 4, 2), (50, 256, 8, 3),
                            (9, 5, 5, 4)]:
        idx = inputs.random_assignments(T, E, k, seed).numpy()
        counts, offsets, row_token, assign_row = oracle_mod.dispatch(idx, E)
        flat = idx.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(row_token, order // k)
        inv = np.empty_like(order)
        inv[order] = np.arange(T * k)
        assert np.array_equal(assign_row, inv)
        # bijection and round trip
        assert np.array_equal(np.sort(assign_row), np.arange(T * k))
        assert np.array_equal(row_token[assign_row], np.repeat(np.arange(T), k))


def test_dispatch_rejects_out_of_range(oracle_mod):
    idx = np.array([[0, 1], [2, 8]], np.int32)
    with pytest.raises(ValueError):
        oracle_mod.dispatch(idx, 8)


# ---------------------------------------------------------------------- FFN
def _dense_swiglu(x, wg, wu, wd):
    x, wg, wu, wd = (t.double() for t in (x, wg, wu, wd))
    return (F.silu(x @ wg.T) * (x @ wu.T)) @ wd.T


@pytest.mark.parametrize("act", ["f32", "bf16"])
def test_single_expert_is_dense_swiglu(oracle_mod, act):
    """E=1, k=1: the layer is a dense SwiGLU FFN (torch float64)."""
    s = inputs.MoEShape("e1", T=6, d=128, E=1, k=1, f=96, act=act, wdt=act)
    lay = inputs.make_layer(s, seed=5)
    out = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f)
    ref = _dense_swiglu(lay["x"], lay["w_gate"][0], lay["w_up"][0], lay["w_down"][0]).numpy()
    assert np.max(np.abs(out["y_f64"] - ref)) <= 1e-12 * np.max(np.abs(ref))
    assert np.all(out["topk_idx"] == 0) and np.all(out["topk_w"] == 1.0)


def test_identical_experts_equal_dense(oracle_mod):
    s = inputs.MoEShape("same", T=10, d=64, E=4, k=2, f=32, act="f32", wdt="f32")
    lay = inputs.make_layer(s, seed=6)
    for key in ("w_gate", "w_up", "w_down"):
        lay[key] = lay[key][:1].repeat(s.E, 1, 1).contiguous()
    out = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f)
    ref = _dense_swiglu(lay["x"], lay["w_gate"][0], lay["w_up"][0], lay["w_down"][0]).numpy()
    assert np.max(np.abs(out["y_f64"] - ref)) <= 1e-6 * np.max(np.abs(ref))


def test_expert_ffn_stage_matches_dense(oracle_mod):
    s = inputs.MoEShape("stage", T=1, d=64, E=3, k=1, f=48, act="bf16", wdt="bf16")
    lay = inputs.make_layer(s, seed=7)
    rows = inputs.random_rows(5, 64, inputs.BF16, seed=8)
    y = oracle_mod.expert_ffn(rows, inputs.BF16, lay, 2, 64, 48, inputs.BF16)
    ref = _dense_swiglu(rows, lay["w_gate"][2], lay["w_up"][2], lay["w_down"][2]).numpy()
    assert np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))


# --------------------------------------------------------------------- int4
def _pack(q: np.ndarray) -> np.ndarray:
    nib = (q.astype(np.int16) & 0xF).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def test_int4_decode_exact(oracle_mod):
    """w = q * s with q the signed nibble (low nibble = even index) and s the
    bf16 scale of its 128-wide group."""
    rng = np.random.default_rng(9)
    E, rows, cols = 2, 5, 256
    q = rng.integers(-8, 8, size=(E, rows, cols))
    s = torch.from_numpy(rng.uniform(1e-3, 1.0, size=(E, rows, cols // 128)).astype(np.float32))
    s_bf = s.to(torch.bfloat16)
    packed = _pack(q)
    sf = s_bf.float().numpy()
    for e in range(E):
        for r in range(rows):
            for c in range(0, cols, 7):
                want = float(np.float32(q[e, r, c]) * sf[e, r, c // 128])
                got = oracle_mod.weight_at(packed, _bits(s_bf), inputs.I4G128, e, rows, cols, r, c)
                assert got == want


def test_int4_ffn_equals_f32_on_decoded_weights(oracle_mod):
    rng = np.random.default_rng(10)
    d, f = 256, 128
    def mk(rows, cols):
        q = rng.integers(-7, 8, size=(1, rows, cols))
        s = torch.from_numpy(rng.uniform(1e-3, 3e-3, size=(1, rows, cols // 128))
                             .astype(np.float32)).to(torch.bfloat16)
        w = torch.from_numpy(q.astype(np.float32)) * s.float().repeat_interleave(128, dim=2)
        return _pack(q), _bits(s), w
    pg, sg, wg = mk(f, d)
    pu, su, wu = mk(f, d)
    pd, sd, wd = mk(d, f)
    x = inputs.random_rows(3, d, inputs.BF16, seed=11)
    y4 = oracle_mod.expert_ffn(x, inputs.BF16, dict(w_gate=pg, w_up=pu, w_down=pd, s_gate=sg,
                                                    s_up=su, s_down=sd), 0, d, f, inputs.I4G128)
    ref = _dense_swiglu(x, wg[0], wu[0], wd[0]).numpy()
    assert np.max(np.abs(y4 - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_quantiser_round_trip():
    rng = np.random.default_rng(12)
    w = torch.from_numpy((rng.normal(size=(7, 384)) * 0.02).astype(np.float32))
    packed, s = inputs.quantize_i4g128(w)
    lo = (packed & 0xF).to(torch.int16)
    hi = (packed >> 4).to(torch.int16)
    q = torch.stack([lo, hi], dim=-1).reshape(7, 384)
    q = torch.where(q >= 8, q - 16, q)
    assert int(q.abs().max()) <= 7
    sf = s.float().repeat_interleave(128, dim=1)
    amax = w.reshape(7, 3, 128).abs().amax(-1)
    assert torch.equal(s, (amax / 7).to(torch.bfloat16))
    err = (w - q.float() * sf).abs()
    unclamped = (w / sf).abs() <= 7
    assert bool((err[unclamped] <= sf[unclamped] / 2 * (1 + 1e-6)).all())


# --------------------------------------------------------------- bf16, merge
# ------------------------------------------------------------------ MX formats
def test_e4m3_decode_matches_torch(oracle_mod):
    """Every E4M3 code decodes to torch's float8_e4m3fn value (NaN codes NaN)."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle_mod.mx_element(inputs.MXFP8, c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], ref[~nan])


def test_e2m1_and_e8m0_decode_match_the_format_tables(oracle_mod):
    """E2M1 codes 0..15 against the value table of the OCP MX format (sign
    bit 3), and E8M0 codes against 2^(c - 127) with 255 = NaN."""
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    want = table + [-v for v in table]
    got = [oracle_mod.mx_element(inputs.MXFP4, c) for c in range(16)]
    assert got == want
    assert math.copysign(1.0, got[8]) == -1.0          # code 8 is -0
    for c in (0, 1, 100, 127, 128, 200, 254):
        assert oracle_mod.mx_element(inputs.F32, c) == math.ldexp(1.0, c - 127)
    assert math.isnan(oracle_mod.mx_element(inputs.F32, 255))


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_weight_decode_is_element_times_scale(oracle_mod, fmt):
    """weight_at of packed MX weights = element value x 2^(s - 127), with the
    E2M1 nibble order low = even index and one scale per 32 indices."""
    rng = np.random.default_rng(7)
    rows, cols = 3, 96
    if fmt == "mxfp8":
        codes = rng.integers(0, 256, size=(1, rows, cols), dtype=np.uint8)
        codes[codes & 0x7F == 0x7F] = 0x11            # no NaN codes
        elem = lambda r, c: oracle_mod.mx_element(inputs.MXFP8, codes[0, r, c])  # noqa: E731
        code = inputs.MXFP8
    else:
        nib = rng.integers(0, 16, size=(rows, cols), dtype=np.uint8)
        codes = (nib[:, 0::2] | (nib[:, 1::2] << 4))[None].astype(np.uint8)
        elem = lambda r, c: [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0][nib[r, c] & 7] * (  # noqa: E731
            -1.0 if nib[r, c] & 8 else 1.0)
        code = inputs.MXFP4
    scales = rng.integers(100, 140, size=(1, rows, cols // 32), dtype=np.uint8)
    for r in range(rows):
        for c in range(0, cols, 7):
            want = elem(r, c) * 2.0 ** (int(scales[0, r, c // 32]) - 127)
            assert oracle_mod.weight_at(codes, scales, code, 0, rows, cols, r, c) == want


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_quantiser_round_trip_and_ties(oracle_mod, fmt):
    """The harness quantiser: decoded weights within half an element step of
    the input clipped to the format's largest normal (the shared exponent
    floor(log2 max|w|) - emax lets a block maximum reach just under 2^(emax+1),
    above 448 or 6), and exact midpoints go to the even code."""
    g = torch.Generator().manual_seed(8)
    w = torch.randn(6, 128, generator=g) * 0.02
    q, s = inputs.quantize_mx(w, fmt)
    code = inputs.DTYPE_CODE[fmt]
    wq = q.numpy()[None]
    sc = s.numpy()[None]
    mant = 3 if fmt == "mxfp8" else 1
    for r in range(6):
        for c in range(128):
            deq = oracle_mod.weight_at(wq, sc, code, 0, 6, 128, r, c)
            scale = 2.0 ** (int(sc[0, r, c // 32]) - 127)
            top = 448.0 if fmt == "mxfp8" else 6.0
            x = math.copysign(min(abs(float(w[r, c])), top * scale), float(w[r, c]))
            a = abs(x) / scale
            step = 2.0 ** (max(math.floor(math.log2(a)), 0 if fmt == "mxfp4" else -6) - mant) \
                if a > 0 else 0.0
            assert abs(deq - x) <= step / 2 * scale * (1 + 1e-12) + 1e-30
    # ties: in block units, E2M1 1.25 (between 1 and 1.5) -> 1 (even code 2),
    # 1.75 -> 2; E4M3 1.0625 (between 1 and 1.125) -> 1, 1.1875 -> 1.25
    vals = [1.25, 1.75, 2.5, 5.0] if fmt == "mxfp4" else [1.0625, 1.1875, 17.0, 19.0]
    want = [1.0, 2.0, 2.0, 4.0] if fmt == "mxfp4" else [1.0, 1.25, 16.0, 20.0]
    row = torch.zeros(1, 32)
    row[0, :4] = torch.tensor(vals)
    row[0, 31] = 6.0 if fmt == "mxfp4" else 448.0   # fixes the block exponent at 0
    q, s = inputs.quantize_mx(row, fmt)
    assert int(s[0, 0]) == 127
    got = [oracle_mod.weight_at(q.numpy()[None], s.numpy()[None], code, 0, 1, 32, 0, c)
           for c in range(4)]
    assert got == want


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_ffn_equals_f32_ffn_on_decoded_weights(oracle_mod, fmt):
    s = inputs.MoEShape("mx", T=5, d=128, E=2, k=1, f=64, wdt=fmt)
    lay = inputs.make_layer(s, seed=18)
    code = inputs.DTYPE_CODE[fmt]
    dec = {}
    for key, rows, cols in (("w_gate", s.f, s.d), ("w_up", s.f, s.d), ("w_down", s.d, s.f)):
        skey = "s_" + key[2:]
        m = np.zeros((s.E, rows, cols), np.float32)
        for e in range(s.E):
            for r in range(rows):
                for c in range(cols):
                    m[e, r, c] = oracle_mod.weight_at(lay[key], lay[skey], code, e, rows, cols,
                                                      r, c)
        dec[key] = torch.from_numpy(m)
    x = lay["x"]
    for e in range(s.E):
        got = oracle_mod.expert_ffn(x, s.act_code, lay, e, s.d, s.f, code)
        ref = oracle_mod.expert_ffn(x, s.act_code, dec, e, s.d, s.f, inputs.F32)
        assert np.max(np.abs(got - ref)) <= 1e-12 * max(1.0, np.max(np.abs(ref)))


def test_bf16_rounding_matches_torch(oracle_mod):
    vals = [0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20,
            -2.5e-3, 3.4e38, 1e-40, float("inf"), -float("inf")]
    rng = np.random.default_rng(13)
    vals += list(rng.normal(size=200).astype(np.float32) * 10.0)
    for v in vals:
        want = int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16)
                   .view(torch.int16).item()) & 0xFFFF
        assert oracle_mod.float_to_bf16(v) == want, v
        assert oracle_mod.bf16_to_float(want) == float(
            torch.tensor([want], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float())
    assert math.isnan(oracle_mod.bf16_to_float(oracle_mod.float_to_bf16(float("nan"))))


def test_combine_one_hot_is_gather(oracle_mod):
    T, d = 9, 64
    y_perm = inputs.random_rows(T, d, inputs.F32, seed=14).numpy()
    perm = np.random.default_rng(15).permutation(T).astype(np.int32)
    y64, yo = oracle_mod.combine(y_perm, perm, np.ones((T, 1), np.float32), T, 1, d, inputs.F32)
    assert np.array_equal(yo, y_perm[perm])
    y64, yb = oracle_mod.combine(y_perm, perm, np.ones((T, 1), np.float32), T, 1, d, inputs.BF16)
    assert np.array_equal(yb, _bits(torch.from_numpy(y_perm[perm]).to(torch.bfloat16)))


def test_combine_k2_k3_hand_computed(oracle_mod):
    """The weighted merge y[t] = sum_j g[t][j] * y_perm[assign_row[t*k+j]] on
    values worked out by hand (gates and rows exact in binary, so the expected
    outputs are exact): a transposed gather index, a swapped gate or a dropped
    slot each change at least one of them."""
    # k = 2, T = 2, d = 3; assign_row sends token 0 to rows (2, 0), token 1 to (1, 3)
    y_perm = np.array([[4.0, -8.0, 1.0],
                       [2.0, 6.0, -2.0],
                       [-4.0, 0.5, 8.0],
                       [16.0, -1.0, 0.0]], np.float32)
    assign = np.array([2, 0, 1, 3], np.int32)
    gates = np.array([[0.75, 0.25], [0.5, 0.5]], np.float32)
    # token 0: 0.75*(-4, 0.5, 8) + 0.25*(4, -8, 1) = (-3+1, 0.375-2, 6+0.25)
    # token 1: 0.5*(2, 6, -2) + 0.5*(16, -1, 0)     = (1+8, 3-0.5, -1+0)
    want = np.array([[-2.0, -1.625, 6.25], [9.0, 2.5, -1.0]])
    y64, yo = oracle_mod.combine(y_perm, assign, gates, 2, 2, 3, inputs.F32)
    assert np.array_equal(y64, want) and np.array_equal(yo, want.astype(np.float32))
    # k = 3, T = 1, d = 2; slots read rows 1, 2, 0 with gates 1/2, 1/4, 1/4
    y_perm = np.array([[8.0, 1.0], [2.0, -4.0], [-16.0, 3.0]], np.float32)
    assign = np.array([1, 2, 0], np.int32)
    gates = np.array([[0.5, 0.25, 0.25]], np.float32)
    # 0.5*(2, -4) + 0.25*(-16, 3) + 0.25*(8, 1) = (1-4+2, -2+0.75+0.25)
    want = np.array([[-1.0, -1.0]])
    y64, yo = oracle_mod.combine(y_perm, assign, gates, 1, 3, 2, inputs.F32)
    assert np.array_equal(y64, want) and np.array_equal(yo, want.astype(np.float32))
    # bf16 output: 0.5*1 + 0.5*(1 + 2^-8) = 1 + 2^-9, halfway between the bf16
    # values 1 and 1 + 2^-7: round to nearest even gives 1.0 (0x3F80); and
    # 0.5*(1 + 2^-7) + 0.5*(1 + 2^-6) = 1 + 3*2^-8 rounds up to 1 + 2^-6 (0x3F82)
    y_perm = np.array([[1.0, 1 + 2.0 ** -7], [1 + 2.0 ** -8, 1 + 2.0 ** -6]], np.float32)
    assign = np.array([0, 1], np.int32)
    gates = np.array([[0.5, 0.5]], np.float32)
    y64, yb = oracle_mod.combine(y_perm, assign, gates, 1, 2, 2, inputs.BF16)
    assert np.array_equal(y64, [[1 + 2.0 ** -9, 1 + 3 * 2.0 ** -8]])
    assert yb.tolist() == [[0x3F80, 0x3F82]]


@pytest.mark.parametrize("act,wdt,bias", [("bf16", "bf16", "zipf"), ("f32", "f32", "none"),
                                          ("bf16", "i4g128", "none")])
def test_threaded_forward_is_bit_identical(oracle_mod, act, wdt, bias):
    """The N-thread forward (token list split over std::threads) returns the
    single-threaded call's bits for every thread count, with and without a
    token list, including more threads than tokens."""
    s = inputs.MoEShape("mt", T=23, d=256, E=8, k=3, f=128, act=act, wdt=wdt, bias=bias)
    lay = inputs.make_layer(s, seed=17)
    one = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f)
    for n in (2, 3, 7, 40):
        many = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f,
                                      threads=n)
        for key in one:
            assert np.array_equal(one[key], many[key]), (n, key)
    tok = [5, 0, 22, 5, 11]
    sub1 = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f, tokens=tok)
    sub4 = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f, tokens=tok,
                                  threads=4)
    for key in sub1:
        assert np.array_equal(sub1[key], sub4[key]), key
    assert np.array_equal(sub1["y_f64"], one["y_f64"][tok])
    with pytest.raises(ValueError):
        oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f,
                               tokens=[0, 23], threads=2)


def test_forward_equals_staged_composition(oracle_mod):
    s = inputs.MoEShape("mini", T=20, d=128, E=6, k=3, f=64, act="bf16", wdt="bf16")
    lay = inputs.make_layer(s, seed=16)
    full = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f)
    logits = oracle_mod.router_logits(lay["x"], s.act_code, lay["w_router"], None, s.T, s.d, s.E)
    idx, w, gap, _ = oracle_mod.select_topk(logits, s.k)
    assert np.array_equal(idx, full["topk_idx"]) and np.array_equal(w, full["topk_w"])
    counts, offsets, row_token, assign_row = oracle_mod.dispatch(idx, s.E)
    xb = lay["x"][torch.from_numpy(row_token).long()]
    y_perm = np.zeros((s.T * s.k, s.d))
    for e in range(s.E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            y_perm[a:b] = oracle_mod.expert_ffn(xb[a:b], s.act_code, lay, e, s.d, s.f, s.w_code)
    y64, _ = oracle_mod.combine(y_perm.astype(np.float32), assign_row, w, s.T, s.k, s.d, s.act_code)
    assert np.max(np.abs(y64 - full["y_f64"])) <= 1e-6 * np.max(np.abs(full["y_f64"]))
    sub = oracle_mod.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f,
                                 tokens=[3, 17, 0])
    assert np.array_equal(sub["y_f64"], full["y_f64"][[3, 17, 0]])


# ------------------------------------------------------------ closed forms
def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def test_closed_form_cases(oracle_mod):
    cases = json.load(open(os.path.join(HERE, "golden", "closed_form_cases.json")))["cases"]
    for c in cases:
        d, E, k, f = c["d"], c["E"], c["k"], c["f"]
        lay = {key: torch.tensor(c[key], dtype=torch.float32)
               for key in ("x", "w_router", "w_gate", "w_up", "w_down")}
        out = oracle_mod.moe_forward(lay, inputs.F32, inputs.F32, 1, d, E, k, f)
        assert out["topk_idx"].tolist() == c["expect"]["topk_idx"]
        if c["name"] == "one_expert_k1":
            h = 6.0 / (1.0 + math.exp(-2.0))
            gates, gap, y = [1.0], 1.0, [h, 0.5 * h]
        else:
            g = [_sig(1.0), _sig(-1.0)]
            h1, h0 = 2.0 * _sig(2.0), 2.0 * _sig(1.0)
            # the gates enter the merge as the fp32 values the layer outputs
            g32 = [float(np.float32(v)) for v in g]
            gates, gap, y = g, 5.0, [g32[1] * h0, g32[0] * h1]
        assert np.allclose(out["topk_w"][0], gates, rtol=0, atol=6e-8)
        assert out["gap"][0] == gap
        assert np.allclose(out["y_f64"][0], y, rtol=1e-12, atol=0)


# ----------------------------------------------------------- skewed alpha
def test_skewed_alpha_constant_matches_script_record():
    rec = json.load(open(os.path.join(HERE, "golden", "skewed_alpha.json")))
    assert rec["alpha"] == inputs.SKEWED_ALPHA
    assert rec["hottest_share"] >= 0.24 and rec["empty_experts"] >= 3


@pytest.mark.slow
def test_skewed_alpha_is_smallest_on_grid(oracle_mod):
    s = inputs.CONFIGS["skewed"]

    def stats(alpha):
        lay = inputs.make_layer(s.with_(alpha=alpha), experts=False)
        lg = oracle_mod.router_logits(lay["x"], s.act_code, lay["w_router"], lay["b_router"],
                                      s.T, s.d, s.E)
        idx, _, _, _ = oracle_mod.select_topk(lg, s.k)
        c = np.bincount(idx.reshape(-1), minlength=s.E)
        return c.max() / c.sum(), int((c == 0).sum())

    share, empty = stats(inputs.SKEWED_ALPHA)
    assert share >= 0.24 and empty >= 3
    share0, empty0 = stats(round(inputs.SKEWED_ALPHA - 0.05, 2))
    assert not (share0 >= 0.24 and empty0 >= 3)
