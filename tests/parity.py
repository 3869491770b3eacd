"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import mixture_experts_gb300 as moe
import oracle
from mixture_experts_gb300 import inputs

# max|err| / max|ref| bounds on the layer output per expert weight type
TOL = {"f32": 1e-5, "bf16": 2e-2, "i4g128": 3e-2, "mxfp8": 3e-2, "mxfp4": 3e-2}
GATE_TOL = 1e-6   # absolute, on the renormalised gates
NEAR_TIE = 1e-5   # fp32 logit gap below which several selections are correct


def cuda_layer(layer: dict) -> dict:
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in layer.items()}


def make_handle(s: inputs.MoEShape, dev: dict, path=moe.PATH_AUTO, max_tokens=None):
    return moe.MoELayer(s.d, s.f, s.E, s.k, max_tokens or s.T, s.act_code, s.w_code, dev,
                        path=path)


def oracle_routing(s: inputs.MoEShape, layer: dict):
    logits = oracle.router_logits(layer["x"], s.act_code, layer["w_router"], layer["b_router"],
                                  s.T, s.d, s.E)
    return oracle.select_topk(logits, s.k)


def check_routing(gpu_idx, gpu_w, ref_idx, ref_w, gap, inner):
    """Selected ids bit-exact and gates within GATE_TOL, except tokens whose
    k-th/(k+1)-th gap is a near-tie (returned as a mask, reported not failed).
    Where two selected logits near-tie, the slot order is compared as a set."""
    gpu_idx, gpu_w = np.asarray(gpu_idx), np.asarray(gpu_w)
    near = gap < NEAR_TIE
    swap = (inner < NEAR_TIE) & ~near
    firm = ~near & ~swap
    assert np.array_equal(gpu_idx[firm], ref_idx[firm]), "top-k ids differ from the oracle"
    assert np.max(np.abs(gpu_w[firm] - ref_w[firm]), initial=0.0) <= GATE_TOL
    for t in np.nonzero(swap)[0]:
        a = sorted(zip(gpu_idx[t], gpu_w[t]))
        b = sorted(zip(ref_idx[t], ref_w[t]))
        assert [i for i, _ in a] == [i for i, _ in b]
        assert max(abs(x[1] - y[1]) for x, y in zip(a, b)) <= GATE_TOL
    return near


def check_dispatch_valid(idx, counts, offsets, row_token, assign_row, E):
    """Properties any correct stable dispatch of `idx` has."""
    idx = np.asarray(idx)
    T, k = idx.shape
    flat = idx.reshape(-1)
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(np.sort(assign_row), np.arange(T * k))
    assert np.array_equal(row_token[assign_row], np.repeat(np.arange(T), k))
    for e in range(E):
        rows = row_token[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(rows) > 0), "rows of one expert must keep token order"


def check_dispatch(gpu: dict, ref_idx, near, E):
    """Bit-exact against the oracle's dispatch when no token near-tied; else
    validity of the GPU's own dispatch of its own selection."""
    g = {k: np.asarray(v) for k, v in gpu.items()}
    if not near.any():
        counts, offsets, row_token, assign_row = oracle.dispatch(ref_idx, E)
        assert np.array_equal(g["counts"], counts)
        assert np.array_equal(g["offsets"], offsets)
        assert np.array_equal(g["row_token"], row_token)
        assert np.array_equal(g["assign_row"], assign_row)
    check_dispatch_valid(g["topk_idx"], g["counts"], g["offsets"], g["row_token"],
                         g["assign_row"], E)


def y_to_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def rel_err(y, ref) -> float:
    y, ref = np.asarray(y, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(y - ref)) / max(np.max(np.abs(ref)), 1e-30))


def host_dict(d: dict) -> dict:
    return {k: v.cpu().numpy() for k, v in d.items()}


def check_layer(s, lay, y, dbg, threads=1, sample=None):
    """Routing and dispatch of every token against the oracle, then the output
    of every token that is not a near-tie (or of `sample` seeded tokens),
    element by element."""
    idx, w, gap, inner = oracle_routing(s, lay)
    near = check_routing(dbg["topk_idx"], dbg["topk_w"], idx, w, gap, inner)
    check_dispatch(dbg, idx, near, s.E)
    assert np.allclose(dbg["gap"][~near], gap[~near], rtol=0, atol=1e-5)
    tokens = np.nonzero(~near)[0].astype(np.int32)
    if sample is not None and sample < len(tokens):
        pick = np.random.default_rng(0).choice(len(tokens), sample, replace=False)
        tokens = np.sort(np.concatenate([tokens[pick], tokens[[0, -1]]]))
        tokens = np.unique(tokens).astype(np.int32)
    ref = oracle.moe_forward(lay, s.act_code, s.w_code, s.T, s.d, s.E, s.k, s.f, tokens=tokens,
                             threads=threads)
    got = y_to_f64(y)[tokens]
    err = rel_err(got, ref["y_f64"])
    assert err <= TOL[s.wdt], f"{s.name}: max|err|/max|ref| = {err:.3e}"
    return err, int(near.sum())
