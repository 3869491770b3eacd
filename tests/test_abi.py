"""The C-ABI library builds, loads without a GPU, exports every declared
symbol and rejects bad arguments before launching anything (CPU only)."""
import ctypes

import pytest

import mixture_experts_gb300 as moe
from mixture_experts_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def test_exports_every_header_symbol(lib):
    names = moe.header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    for n in ("coli_moe_create", "coli_moe_forward", "coli_route_topk", "coli_permute",
              "coli_expert_ffn", "coli_combine"):
        assert n in names


def test_version_and_status_strings(lib):
    assert "sm_103a" in moe.coli_version()
    for code in moe.STATUS:
        assert moe.coli_status_string(code) != "unknown status"


@pytest.mark.parametrize("field,value", [
    ("d_model", 100), ("d_ff", 0), ("n_experts", 0), ("n_experts", 300), ("top_k", 0),
    ("top_k", 9), ("max_tokens", 0), ("act_dtype", 2), ("weight_dtype", 0), ("path", 7)])
def test_create_rejects_bad_config(lib, field, value):
    cfg = moe.coli_moe_config(256, 512, 8, 2, 16, moe.BF16, moe.BF16, 0, 0)
    setattr(cfg, field, value)
    rc, h, msg = moe.coli_moe_create(cfg, moe.coli_moe_weights(), stream=0)
    assert rc == moe.COLI_EINVAL and h.value is None and msg


def test_create_rejects_int4_with_bad_group(lib):
    cfg = moe.coli_moe_config(192, 512, 8, 2, 16, moe.BF16, moe.I4G128, 0, 0)
    rc, _, msg = moe.coli_moe_create(cfg, moe.coli_moe_weights(), stream=0)
    assert rc == moe.COLI_EINVAL and "128" in msg


@pytest.mark.parametrize("wdt", [moe.MXFP8, moe.MXFP4])
def test_create_checks_mx_shapes(lib, wdt):
    cfg = moe.coli_moe_config(192, 512, 8, 2, 16, moe.BF16, wdt, 0, 0)
    rc, _, msg = moe.coli_moe_create(cfg, moe.coli_moe_weights(), stream=0)
    assert rc == moe.COLI_EINVAL and "128" in msg
    # both paths serve MX experts: the configuration passes, the missing
    # weights are what the call rejects
    cfg = moe.coli_moe_config(256, 512, 8, 2, 16, moe.BF16, wdt, 0, moe.PATH_PREFILL)
    rc, _, msg = moe.coli_moe_create(cfg, moe.coli_moe_weights(), stream=0)
    assert rc == moe.COLI_EINVAL and "weights" in msg
    cfg = moe.coli_moe_config(256, 512, 8, 2, 16, moe.F32, wdt, 0, 0)
    rc, _, msg = moe.coli_moe_create(cfg, moe.coli_moe_weights(), stream=0)
    assert rc == moe.COLI_EINVAL


def test_create_rejects_bad_residency_tiers(lib):
    base = dict(d=256, f=512, E=8, k=2, T=16)

    def cfg(act, wdt, path, slots, promo):
        return moe.coli_moe_config(base["d"], base["f"], base["E"], base["k"], base["T"], act,
                                   wdt, 0, path, slots, promo)
    for c, code, word in [
            (cfg(moe.BF16, moe.BF16, 0, 9, 0), moe.COLI_EINVAL, "expert_slots"),
            (cfg(moe.BF16, moe.BF16, 0, -1, 0), moe.COLI_EINVAL, "expert_slots"),
            (cfg(moe.BF16, moe.BF16, 0, 4, 5), moe.COLI_EINVAL, "max_promotions"),
            (cfg(moe.F32, moe.F32, 0, 4, 1), moe.COLI_EUNSUPPORTED, "bf16"),
            (cfg(moe.BF16, moe.I4G128, moe.PATH_PREFILL, 4, 1), moe.COLI_EUNSUPPORTED,
             "decode")]:
        rc, _, msg = moe.coli_moe_create(c, moe.coli_moe_weights(), stream=0)
        assert rc == code and word in msg, (rc, msg)
    assert moe.coli_moe_residency(None, 8)[0] == moe.COLI_EINVAL


def test_create_rejects_missing_weights(lib):
    cfg = moe.coli_moe_config(256, 512, 8, 2, 16, moe.BF16, moe.BF16, 0, 0)
    rc, _, msg = moe.coli_moe_create(cfg, moe.coli_moe_weights(), stream=0)
    assert rc == moe.COLI_EINVAL and "weights" in msg


def test_stage_argument_validation(lib):
    fake = 1 << 20  # never dereferenced: validation fails first
    assert moe.coli_route_topk(None, None, None, -1, 64, 8, 2, moe.BF16, None, None,
                               stream=0) == moe.COLI_EINVAL
    assert moe.coli_route_topk(fake, fake, None, 4, 64, 8, 9, moe.BF16, fake, fake,
                               stream=0) == moe.COLI_EINVAL
    assert moe.coli_route_topk(fake + 8, fake, None, 4, 64, 8, 2, moe.BF16, fake, fake,
                               stream=0) == moe.COLI_EINVAL  # misaligned x
    assert moe.coli_route_topk(fake, fake, None, 4, 64, 64, 2, moe.BF16, fake, fake,
                               stream=0) == moe.COLI_EINVAL  # E > 32 needs scratch
    assert moe.coli_permute(None, None, 4, 64, 8, 2, moe.BF16, None, None, None, None, None,
                            stream=0) == moe.COLI_EINVAL
    n = moe.coli_permute_scratch_bytes(8000, 4, 64)
    assert n > 0
    assert moe.coli_permute(fake, fake, 8000, 64, 64, 4, moe.BF16, fake, fake, fake, fake, fake,
                            scratch=fake + 64, scratch_bytes=n, stream=0) == moe.COLI_EINVAL
    assert moe.coli_combine(fake, fake, fake, 4, 2, 64, 5, fake, stream=0) == moe.COLI_EINVAL
    assert moe.coli_expert_ffn(None, fake, fake, 4, fake, stream=0) == moe.COLI_EINVAL
    assert moe.coli_selftest_bounded_wait(0, stream=0) == moe.COLI_EINVAL
    assert "spin_limit" in moe.last_error()


def test_scratch_sizes(lib):
    assert moe.coli_route_scratch_bytes(256, 4096, 8) == 0
    assert moe.coli_route_scratch_bytes(256, 6144, 256) >= 12 * 256 * 256 * 4
    assert moe.coli_permute_scratch_bytes(32, 2, 8) == 0
    big = moe.coli_permute_scratch_bytes(16384, 4, 64)
    assert big > 0 and big % 256 == 0


def test_handle_calls_reject_null(lib):
    assert moe.coli_moe_forward(None, None, 1, None, stream=0) == moe.COLI_EINVAL
    assert moe.coli_moe_path_for(None, 4) == moe.COLI_EINVAL
    assert lib.coli_moe_set_timing(None, 1) == moe.COLI_EINVAL
    moe.coli_moe_destroy(None)  # no-op


def _declarations():
    """name -> list of parameter types, parsed from include/coli_moe.h."""
    import re
    text = open(moe.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"#.*", "", text)
    out = {}
    for m in re.finditer(r"([\w\s\*]+?)\b(coli_\w+)\s*\(([^;{]*?)\)\s*;", text):
        params = " ".join(m.group(3).split())
        out[m.group(2)] = ([] if params in ("", "void") else
                           [p.strip() for p in params.split(",")])
    return out


def _kind(param: str) -> str:
    """The ctypes class a C parameter needs: P pointer, Z size_t, I 32-bit int."""
    if "*" in param:
        return "P"
    words = param.split()
    if words[0] == "size_t":
        return "Z"
    if words[0] in ("int", "int32_t"):
        return "I"
    raise AssertionError(f"unexpected parameter type: {param}")


def test_binding_signatures_match_header():
    # every ctypes signature of the binding has the header's parameter count
    # and kinds, so no call passes arguments of the wrong size
    decl = _declarations()
    assert set(moe._SIGS) == set(decl) == set(moe.header_functions())
    for name, (_, args) in moe._SIGS.items():
        want = [_kind(p) for p in decl[name]]
        assert args == want, (name, args, want)
