"""Seeded random-shape sweep: layers whose sizes, expert format, path,
router bias and residency tier are drawn at random within the library's
limits, each checked on every token against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import mixture_experts_gb300 as moe
from mixture_experts_gb300 import inputs
from parity import check_layer, cuda_layer, host_dict

pytestmark = pytest.mark.gpu

N_CASES = 32  # cases 24..31 force the tensor-core (prefill) path


def draw(i: int) -> tuple:
    """Case i: (shape, path, expert_slots, max_promotions)."""
    g = np.random.default_rng(1000 + i)
    wdt = ["bf16", "bf16", "i4g128", "mxfp8", "mxfp4", "f32"][g.integers(6)]
    act = "f32" if wdt == "f32" else "bf16"
    step = 128 if wdt in ("i4g128", "mxfp8", "mxfp4") else 64
    d = int(step * g.integers(1, 7))
    f = int(step * g.integers(1, 7))
    E = int(g.choice([1, 2, 3, 5, 8, 16, 33, 64, 100, 256]))
    k = int(g.integers(1, min(E, 8) + 1))
    T = int(g.choice([1, 7, 40, 130, 700, 1500]))
    bias = ["none", "zipf", "hot0"][g.integers(3)]
    path = moe.PATH_AUTO
    if wdt in ("bf16", "i4g128") and g.random() < 0.4:
        path = [moe.PATH_DECODE, moe.PATH_PREFILL][g.integers(2)]
    if i >= 24:
        wdt = ["bf16", "bf16", "i4g128"][g.integers(3)]
        act, step = "bf16", 128
        d, f = int(step * g.integers(1, 9)), int(step * g.integers(1, 9))
        T = int(g.choice([300, 700, 1500, 3000]))
        path = moe.PATH_PREFILL
    slots = promotions = 0
    if wdt != "f32" and path != moe.PATH_PREFILL and E > 1 and g.random() < 0.3:
        slots = int(g.integers(1, E))
        promotions = int(g.integers(0, slots + 1))
    s = inputs.MoEShape(f"sweep{i}", T=T, d=d, E=E, k=k, f=f, act=act, wdt=wdt, bias=bias,
                        slots=slots, promotions=promotions)
    return s, path


@pytest.fixture(scope="module", autouse=True)
def built():
    moe.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_layer_matches_the_oracle(i):
    s, path = draw(i)
    lay = inputs.make_layer(s, seed=2000 + i)
    dev = cuda_layer(lay)
    layer = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev, path=path,
                         expert_slots=s.slots, max_promotions=s.promotions)
    for rep in range(2 if s.slots else 1):  # a tier handle twice: after its first update
        y = layer(dev["x"])
        dbg = host_dict(layer.debug(s.T))
        torch.cuda.synchronize()
        assert layer.status() == moe.COLI_OK, s
        err, near = check_layer(s, lay, y, dbg, threads=4)
    print(f"{s} path={layer.path_for(s.T)} rel_err={err:.2e} near={near}")
