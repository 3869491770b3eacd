"""coli_permute_noalloc against coli_permute (GPU).

coli_permute_noalloc serves callers that cannot allocate device memory at
the call site (a plugin whose host program owns the device memory pool, a
real-time loop that may not allocate after start-up): it keeps its scratch
table in a fixed area inside the library. This file is collected last so a
run that stops at its first failure has run every other test before it; it
passes on its own in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import mixture_experts_gb300 as moe
from mixture_experts_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    moe.build()
    assert torch.cuda.is_available()


def _outputs(T, E, k, d, dtype):
    n = T * k
    return [torch.full((E,), -1, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((n,), -1, dtype=torch.int32, device="cuda"),
            torch.full((n,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros(n, d, dtype=dtype, device="cuda")]


def _with_caller_scratch(idx, x, T, d, E, k, act):
    out = _outputs(T, E, k, d, x.dtype)
    nb = moe.coli_permute_scratch_bytes(T, k, E)
    scratch = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    rc = moe.coli_permute(idx, x, T, d, E, k, act, *out, scratch, nb)
    assert rc == moe.COLI_OK, moe.last_error()
    return out


def _without_scratch(idx, x, T, d, E, k, act):
    out = _outputs(T, E, k, d, x.dtype)
    rc = moe.coli_permute_noalloc(idx, x, T, d, E, k, act, *out)
    assert rc == moe.COLI_OK, moe.last_error()
    return out


def test_noalloc_matches_coli_permute_on_two_calls_in_a_row():
    # both calls need the scratch table (more than 16384 assignments), with
    # different shapes so the second call cannot pass on the first one's data
    cases = [(5000, 128, 64, 4, "bf16", 1), (3000, 256, 256, 8, "f32", 2)]
    for T, d, E, k, act, seed in cases:
        assert T * k > 16384
        assert moe.coli_permute_scratch_bytes(T, k, E) <= moe.COLI_PERMUTE_STATIC_SCRATCH_BYTES
        code = inputs.DTYPE_CODE[act]
        idx = inputs.random_assignments(T, E, k, seed=seed).cuda()
        x = inputs.random_rows(T, d, code, seed=seed).cuda()
        ref = _with_caller_scratch(idx, x, T, d, E, k, code)
        got = _without_scratch(idx, x, T, d, E, k, code)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):  # integer / copied data: bit-exact
            assert torch.equal(a, b)
        assert moe.coli_device_status() == moe.COLI_OK


@pytest.mark.parametrize("T,E,k", [
    (2048, 64, 8),     # 16384 assignments: the single-block path, no table
    (16384, 256, 8),   # 64 blocks x 256 experts x 4 B = exactly the 65536-byte area
    (131072, 64, 4),   # 524288 assignments at E = 64: 256 blocks x 64 x 4 B, also exactly full
])
def test_noalloc_boundary_shapes(T, E, k):
    """The path that needs no table, and the two largest batches whose table
    fills the area exactly: bit-exact against coli_permute with caller scratch."""
    d = 64
    need = moe.coli_permute_scratch_bytes(T, k, E)
    assert need <= moe.COLI_PERMUTE_STATIC_SCRATCH_BYTES
    if T * k > 16384:
        assert need == moe.COLI_PERMUTE_STATIC_SCRATCH_BYTES
    idx = inputs.random_assignments(T, E, k, seed=T % 97).cuda()
    x = inputs.random_rows(T, d, moe.BF16, seed=3).cuda()
    ref = _with_caller_scratch(idx, x, T, d, E, k, moe.BF16)
    got = _without_scratch(idx, x, T, d, E, k, moe.BF16)
    torch.cuda.synchronize()
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
    assert moe.coli_device_status() == moe.COLI_OK


def test_noalloc_rejects_batches_beyond_its_area():
    T, k, E = 16385, 8, 256  # needs 65 blocks x 256 experts x 4 bytes > 65536
    assert moe.coli_permute_scratch_bytes(T, k, E) > moe.COLI_PERMUTE_STATIC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = moe.coli_permute_noalloc(fake, fake, T, 64, E, k, moe.BF16, fake, fake, fake, fake,
                                  fake)
    assert rc == moe.COLI_EINVAL
    assert "static" in moe.last_error()
    # one row past the E = 64 limit as well
    T, k, E = 131073, 4, 64
    assert moe.coli_permute_scratch_bytes(T, k, E) > moe.COLI_PERMUTE_STATIC_SCRATCH_BYTES
    rc = moe.coli_permute_noalloc(fake, fake, T, 64, E, k, moe.BF16, fake, fake, fake, fake,
                                  fake)
    assert rc == moe.COLI_EINVAL
    # a size outside the general limits names the sizes and the T*k bound
    rc = moe.coli_permute_noalloc(fake, fake, 1 << 22, 64, 8, 8, moe.BF16, fake, fake, fake,
                                  fake, fake)
    assert rc == moe.COLI_EINVAL and "16777216" in moe.last_error()
