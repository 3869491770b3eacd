"""Expert residency tier (experts in pinned host memory, a hot set in HBM
slots, streamed over NVLink-C2C otherwise): placement never changes the
results, the hot set follows the routing, promotions stay within their
per-forward bound (GPU)."""
import numpy as np
import pytest
import torch

import mixture_experts_gb300 as moe
from mixture_experts_gb300 import inputs
from parity import check_layer, cuda_layer, host_dict

pytestmark = pytest.mark.gpu

S = inputs.MoEShape


@pytest.fixture(scope="module", autouse=True)
def built():
    moe.build()
    assert torch.cuda.is_available()


def _handles(s, lay, slots, promotions):
    dev = cuda_layer(lay)
    full = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev)
    tier = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev,
                        expert_slots=slots, max_promotions=promotions)
    return full, tier


@pytest.mark.parametrize("wdt", ["bf16", "i4g128", "mxfp8"])
def test_placement_does_not_change_results(wdt):
    """Forwards over batches whose routing shifts: the tier handle (3 of 8
    experts in HBM, up to 2 promotions per forward) gives the bits of the
    fully resident handle every time, while its hot set moves."""
    s = S("tier", T=24, d=256, E=8, k=2, f=256, wdt=wdt)
    lay = inputs.make_layer(s, seed=51)
    full, tier = _handles(s, lay, slots=3, promotions=2)
    slots0, n0 = tier.residency()
    assert slots0 == [0, 1, 2, -1, -1, -1, -1, -1] and n0 == 0
    moves = 0
    for i in range(6):
        x = inputs.random_rows(s.T, s.d, s.act_code, seed=100 + i).cuda()
        y_full = full(x)
        y_tier = tier(x)
        torch.cuda.synchronize()
        assert torch.equal(y_full, y_tier), f"forward {i}"
        slots, n = tier.residency()
        assert sorted(v for v in slots if v >= 0) == [0, 1, 2]   # three slots, all used
        assert n <= 2 * (i + 1)                                 # bounded promotions
        moves = n
    assert moves > 0
    assert full.status() == moe.COLI_OK and tier.status() == moe.COLI_OK


def test_hot_set_follows_the_routing():
    """A router that sends every token to expert 0: after one forward expert 0
    is promoted into a slot (it starts on the host side: slots hold 0..S-1,
    so the layer is built with expert 0 made hot through a shifted bias)."""
    s = S("tier_hot", T=32, d=256, E=8, k=2, f=128)
    lay = inputs.make_layer(s, seed=52)
    b = torch.zeros(s.E, dtype=torch.float32)
    b[6] = 30.0                       # expert 6: outside the initial slots 0, 1
    lay["b_router"] = b
    full, tier = _handles(s, lay, slots=2, promotions=1)
    slots, _ = tier.residency()
    assert slots[6] == -1
    x = lay["x"].cuda()
    assert torch.equal(full(x), tier(x))
    slots, n = tier.residency()
    assert slots[6] >= 0 and n == 1   # promoted after the first forward, one copy
    y_full, y_tier = full(x), tier(x)
    torch.cuda.synchronize()
    assert torch.equal(y_full, y_tier)
    assert tier.residency()[0][6] == slots[6]   # stays resident while hot


def test_streamed_layer_matches_the_oracle():
    """The tier handle with no promotions (one expert in HBM, the others read
    over C2C every forward) against the oracle, element by element."""
    s = S("tier_oracle", T=40, d=512, E=6, k=2, f=256, wdt="i4g128")
    lay = inputs.make_layer(s, seed=53)
    dev = cuda_layer(lay)
    tier = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev, expert_slots=1,
                        max_promotions=0)
    y = tier(dev["x"])
    dbg = host_dict(tier.debug(s.T))
    torch.cuda.synchronize()
    assert tier.status() == moe.COLI_OK
    check_layer(s, lay, y, dbg)
    assert tier.residency() == ([0, -1, -1, -1, -1, -1], 0)


def test_tier_expert_ffn_stage_and_host_api():
    s = S("tier_stage", T=16, d=256, E=4, k=2, f=128, wdt="mxfp8")
    lay = inputs.make_layer(s, seed=54)
    full, tier = _handles(s, lay, slots=1, promotions=1)
    xh = lay["x"].pin_memory()
    a = torch.empty_like(xh).pin_memory()
    b = torch.empty_like(xh).pin_memory()
    full.forward_host(xh, a)
    tier.forward_host(xh, b)
    assert torch.equal(a, b)
    g = np.random.default_rng(5)
    counts = g.multinomial(s.T * s.k, np.ones(s.E) / s.E)
    n = int(counts.sum())
    offsets = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    xp = inputs.random_rows(n, s.d, s.act_code, seed=6).cuda()
    ya = torch.empty(n, s.d, dtype=torch.float32, device="cuda")
    yb = torch.empty_like(ya)
    assert moe.coli_expert_ffn(full.h, xp, offsets, n, ya) == moe.COLI_OK
    assert moe.coli_expert_ffn(tier.h, xp, offsets, n, yb) == moe.COLI_OK
    torch.cuda.synchronize()
    assert torch.equal(ya, yb)
