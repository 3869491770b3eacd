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
