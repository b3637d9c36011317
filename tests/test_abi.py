"""The C-ABI library loads, exports every function include/mla.h declares, and
rejects malformed arguments on the host before touching the GPU. CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import head_latent_attention_24_b300 as m
    return ctypes.CDLL(m.LIB_PATH)


def test_header_declares_the_four_steps():
    names = declared_functions()
    for n in ("mla_append_cache", "mla_absorb_q", "mla_decode_attn", "mla_out_proj", "mla_create",
              "mla_destroy", "mla_decode_workspace_size", "mla_get_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_abi_version_and_status_strings():
    import head_latent_attention_24_b300 as m
    assert m.mla_abi_version() == 1
    for s in (m.MLA_OK, m.MLA_ERR_INVALID_ARG, m.MLA_ERR_UNSUPPORTED, m.MLA_ERR_CUDA, m.MLA_ERR_DEVICE,
              m.MLA_ERR_TIMEOUT, m.MLA_ERR_WORKSPACE):
        assert m.mla_status_string(s).startswith("MLA_")
    assert "unknown" in m.mla_status_string(12345)


@pytest.mark.parametrize("bad", [
    dict(d_r=15),            # odd rope width
    dict(d_c=0),             # empty latent
    dict(n_h=-1),
    dict(dtype=7),
    dict(max_pos=0),
    dict(rope_base=1.0),
    dict(d_c=60),            # not a multiple of 8
])
def test_create_rejects_bad_shapes_on_host(bad):
    import head_latent_attention_24_b300 as m
    cfg = dict(d=256, n_h=4, d_h=32, d_c=64, d_r=16, d_cq=96, dtype=m.MLA_F32, max_pos=256, rope_base=10000.0)
    cfg.update(bad)
    with pytest.raises(m.MLAError) as ei:
        m.mla_create(**cfg)
    assert ei.value.status == m.MLA_ERR_INVALID_ARG


def test_null_handle_is_rejected():
    import head_latent_attention_24_b300 as m
    for fn, args in ((m._c["mla_destroy"], (None,)),
                     (m._c["mla_decode_attn"], (None, None, None, 1, 1, None, None, None, None, 0, None)),
                     (m._c["mla_append_cache"], (None, None, 1, None, None, None, None, None, 1, 1, None)),
                     (m._c["mla_out_proj"], (None, None, 1, None, None, None, None, 0, None))):
        assert fn(*args) == m.MLA_ERR_INVALID_ARG
    n = ctypes.c_size_t(0)
    assert m._c["mla_decode_step_workspace_size"](None, 1, 1, ctypes.byref(n)) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_decode_step"](None, None, 1, *([None] * 8), None, None, None, 1, None, None, 0,
                                   None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_set_decode_chunks"](None, 4) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_set_wait_limit"](None, 1000) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_set_fault_injection"](None, 0) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_set_kv_norm"](None, None, 1e-5) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_premerge_query_weights"](None, None, None, None, None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_premerge_output_weights"](None, None, None, None, None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_absorb_q_premerged"](None, None, 1, None, None, None, None, None, None, 0,
                                          None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_out_proj_premerged"](None, None, 1, None, None, None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_project_q"](None, None, 1, None, None, None, None, None, None, 0, None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_materialise_kv"](None, None, 1, None, None, None, None, None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_mha_attn"](None, None, 1, 1, None, None, None, 1, None, None, None,
                                None) == m.MLA_ERR_INVALID_ARG
    assert m._c["mla_project_out"](None, None, 1, None, None, None) == m.MLA_ERR_INVALID_ARG


def test_binding_has_every_declared_function():
    """The Python binding carries each C entry point under its own name."""
    import head_latent_attention_24_b300 as m
    missing = [n for n in declared_functions() if n not in m._c]
    assert not missing, missing
