"""Device-side failure handling without faulting the GPU: bad data is skipped
and latched, a bounded wait gives up and reports, and the context stays
usable afterwards (GPU)."""
import numpy as np
import pytest
import torch

import mixture_experts_gb300 as moe
from mixture_experts_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    moe.build()


def _permute(idx, E, k, d=64):
    T = idx.shape[0]
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    n = T * k
    bufs = [torch.full((E,), -7, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.zeros(n, dtype=torch.int32, device="cuda"),
            torch.zeros(n, dtype=torch.int32, device="cuda")]
    x_perm = torch.empty(n, d, dtype=torch.bfloat16, device="cuda")
    nb = moe.coli_permute_scratch_bytes(T, k, E)
    scratch = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    rc = moe.coli_permute(idx.cuda(), x, T, d, E, k, moe.BF16, *bufs, x_perm, scratch, nb)
    return rc, bufs


@pytest.mark.parametrize("T", [6, 9000])
def test_out_of_range_expert_id_is_latched(T):
    assert moe.coli_device_status() == moe.COLI_OK
    idx = inputs.random_assignments(T, 8, 2, seed=1)
    idx[T // 2, 1] = 8      # one id past the last expert
    idx[0, 0] = -3
    rc, bufs = _permute(idx, 8, 2)
    assert rc == moe.COLI_OK  # launch is fine; the kernel found the bad ids
    assert moe.coli_device_status() == moe.COLI_EDEVICE
    counts = bufs[0].cpu().numpy()
    assert counts.sum() == T * 2 - 2   # the two bad assignments were skipped
    assert moe.coli_device_status() == moe.COLI_OK   # cleared by the query
    good = inputs.random_assignments(T, 8, 2, seed=2)
    rc, bufs = _permute(good, 8, 2)
    assert rc == moe.COLI_OK and moe.coli_device_status() == moe.COLI_OK
    assert np.array_equal(bufs[0].cpu().numpy(), np.bincount(good.numpy().ravel(), minlength=8))


def test_combine_after_skipped_ids_reads_nothing_out_of_range():
    """A bad id skipped by the dispatch leaves assign_row = -1; the combine on
    that output adds nothing for it, latches the error and reads no row."""
    assert moe.coli_device_status() == moe.COLI_OK
    T, E, k, d = 40, 8, 2, 64
    idx = inputs.random_assignments(T, E, k, seed=5)
    idx[7, 1] = 1 << 20     # far outside [0, E)
    rc, bufs = _permute(idx, E, k, d)
    assert rc == moe.COLI_OK
    assert moe.coli_device_status() == moe.COLI_EDEVICE
    assign_row = bufs[3]
    ar = assign_row.cpu().numpy()
    assert ar[7 * k + 1] == -1 and (np.delete(ar, 7 * k + 1) >= 0).all()
    y_perm = inputs.random_rows(T * k, d, inputs.F32, seed=6).cuda()
    gates = inputs.random_gates(T, k, seed=7).cuda()
    y = torch.empty(T, d, dtype=torch.float32, device="cuda")
    assert moe.coli_combine(y_perm, assign_row, gates, T, k, d, moe.F32, y) == moe.COLI_OK
    assert moe.coli_device_status() == moe.COLI_EDEVICE
    yc = y.cpu().numpy()
    g = gates.cpu().numpy()
    yp = y_perm.cpu().numpy()
    # the skipped slot contributes nothing; the other slot is there
    assert np.allclose(yc[7], g[7, 0] * yp[ar[7 * k]], rtol=1e-6, atol=1e-7)
    assert moe.coli_device_status() == moe.COLI_OK


@pytest.mark.parametrize("E,k,T", [(8, 2, 20), (64, 4, 20), (64, 4, 1100), (40, 3, 1100)])
def test_nan_router_row_still_gives_k_distinct_ids(E, k, T):
    """A NaN in a token's activations makes its logits NaN: the router ranks
    them as -inf, so the token still gets k distinct ids in [0, E), and the
    data error is latched (the fused E <= 32 router, the two-launch E > 32
    router, and the one-launch tensor-core routers of 1024+ tokens)."""
    assert moe.coli_device_status() == moe.COLI_OK
    d = 256
    s = inputs.MoEShape("nan", T=T, d=d, E=E, k=k, f=64)
    lay = inputs.make_layer(s, seed=8, experts=False)
    x = lay["x"].clone()
    x[3, 17] = float("nan")
    xd, wr = x.cuda(), lay["w_router"].cuda()
    idx = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    nb = moe.coli_route_scratch_bytes(T, d, E)
    scratch = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    assert moe.coli_route_topk(xd, wr, None, T, d, E, k, moe.BF16, idx, w, None, scratch,
                               nb) == moe.COLI_OK
    assert moe.coli_device_status() == moe.COLI_EDEVICE
    ids = idx.cpu().numpy()
    for t in range(T):
        assert len(set(ids[t])) == k and ids[t].min() >= 0 and ids[t].max() < E
    assert np.isfinite(w.cpu().numpy()[np.arange(T) != 3]).all()
    assert moe.coli_device_status() == moe.COLI_OK


def test_mx_activation_beyond_fp16_is_saturated_and_latched():
    """MX experts take fp16 activations: a bf16 input above the fp16 range is
    saturated (no inf reaches the output) and latches a data error."""
    assert moe.coli_device_status() == moe.COLI_OK
    s = inputs.MoEShape("mxbig", T=8, d=256, E=4, k=2, f=128, wdt="mxfp8")
    lay = inputs.make_layer(s, seed=9)
    lay["x"][2, 5] = 1.0e6
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in lay.items()}
    layer = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev)
    y = layer(dev["x"])
    assert layer.status() == moe.COLI_EDEVICE
    assert torch.isfinite(y.float()).all()
    assert layer.status() == moe.COLI_OK


def test_bounded_wait_times_out_and_context_survives():
    assert moe.coli_device_status() == moe.COLI_OK
    assert moe.coli_selftest_bounded_wait(2000) == moe.COLI_OK
    assert moe.coli_device_status() == moe.COLI_ETIMEOUT
    # the context still works: a full layer runs and reports no error
    s = inputs.MoEShape("after", T=16, d=256, E=8, k=2, f=128)
    lay = inputs.make_layer(s, seed=3)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in lay.items()}
    layer = moe.MoELayer(s.d, s.f, s.E, s.k, s.T, s.act_code, s.w_code, dev)
    y = layer(dev["x"])
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()
    assert layer.status() == moe.COLI_OK


def test_forward_rejects_oversized_batch():
    s = inputs.MoEShape("small", T=8, d=128, E=4, k=2, f=64)
    lay = inputs.make_layer(s, seed=4)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in lay.items()}
    layer = moe.MoELayer(s.d, s.f, s.E, s.k, 8, s.act_code, s.w_code, dev)
    x = torch.zeros(9, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    assert moe.coli_moe_forward(layer.h, x, 9, y) == moe.COLI_EINVAL
    assert "max_tokens" in moe.last_error()
    assert moe.coli_moe_forward(layer.h, x[1:], 8, y) in (moe.COLI_OK, moe.COLI_EINVAL)
