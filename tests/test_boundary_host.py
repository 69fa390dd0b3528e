"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every symbol that include/*.h declares, and rejects bad arguments with the
documented codes before touching CUDA."""
import ctypes
import os
import re

import pytest

from attention_block_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in ("cf.h", "cf_test.h"):
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(cf_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_library_loads_and_exports_every_declared_symbol():
    L = binding.lib()
    declared = _declared_functions()
    assert "cf_create" in declared and "cf_decode_attn_block" in declared
    for name in declared:
        assert hasattr(L, name), f"libcf.so does not export {name}"
    assert set(declared) <= set(binding.SIGNATURES), "binding misses a declared function"


def test_error_strings():
    for code in range(0, -8, -1):
        s = binding.strerror(code)
        assert s and "unknown" not in s
    assert "unknown" in binding.strerror(-99)


def _cfg(**kw):
    base = dict(hidden=4096, n_q_heads=32, n_kv_heads=32, head_dim=128, max_batch=1,
                s_max=1025, dtype="f16")
    base.update(kw)
    return binding.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=0), binding.CF_ERR_INVALID_ARG),
    (dict(hidden=100), binding.CF_ERR_INVALID_ARG),
    (dict(n_kv_heads=5), binding.CF_ERR_INVALID_ARG),
    (dict(n_q_heads=0), binding.CF_ERR_INVALID_ARG),
    (dict(head_dim=63), binding.CF_ERR_INVALID_ARG),
    (dict(head_dim=96), binding.CF_ERR_UNSUPPORTED),
    (dict(max_batch=0), binding.CF_ERR_INVALID_ARG),
    (dict(s_max=0), binding.CF_ERR_INVALID_ARG),
    (dict(dtype=7), binding.CF_ERR_INVALID_ARG),
    (dict(cluster_size=3), binding.CF_ERR_INVALID_ARG),
    (dict(cluster_size=32), binding.CF_ERR_INVALID_ARG),
    (dict(head_dim=64, cluster_size=32), binding.CF_ERR_INVALID_ARG),
    (dict(stage_bytes=100), binding.CF_ERR_INVALID_ARG),
    (dict(ctas_per_sm=3), binding.CF_ERR_INVALID_ARG),
    (dict(rope_theta=0.0), binding.CF_ERR_INVALID_ARG),
    (dict(rms_eps=float("nan")), binding.CF_ERR_INVALID_ARG),
    (dict(hidden=64, cluster_size=16), binding.CF_ERR_INVALID_ARG),
])
def test_create_rejects_bad_config_before_cuda(kw, code):
    rc, h = binding.cf_create_rc(_cfg(**kw))
    assert rc == code
    assert not h


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=0), binding.CF_ERR_INVALID_ARG),
    (dict(hidden=100), binding.CF_ERR_INVALID_ARG),        # not a multiple of 8
    (dict(intermediate=0), binding.CF_ERR_INVALID_ARG),
    (dict(max_batch=0), binding.CF_ERR_INVALID_ARG),
    (dict(dtype=7), binding.CF_ERR_INVALID_ARG),
    (dict(rms_eps=float("nan")), binding.CF_ERR_INVALID_ARG),
    (dict(stage_bytes=-1), binding.CF_ERR_INVALID_ARG),
    (dict(hidden=8192), binding.CF_ERR_UNSUPPORTED),       # above the registers' 4096
    (dict(max_batch=65), binding.CF_ERR_UNSUPPORTED),      # the pair's tile is 64 rows
    (dict(max_batch=3, dtype=binding.CF_F32), binding.CF_ERR_UNSUPPORTED),
    (dict(max_batch=16, hidden=320), binding.CF_ERR_UNSUPPORTED),  # not 128 | H
])
def test_ffn_create_rejects_bad_config_before_cuda(kw, code):
    base = dict(hidden=4096, intermediate=11008, max_batch=1, rms_eps=1e-6,
                dtype=binding.CF_F16, stage_bytes=0)
    base.update(kw)
    c = binding.CfFfnConfig(base["hidden"], base["intermediate"], base["max_batch"],
                            base["rms_eps"], base["dtype"], base["stage_bytes"])
    h = binding._vp()
    assert binding.lib().cf_ffn_create(ctypes.byref(c), ctypes.byref(h)) == code
    assert not h.value


def test_ffn_null_arguments():
    L = binding.lib()
    assert L.cf_ffn_create(None, None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_ffn_forward(None, 1, *([None] * 7)) == binding.CF_ERR_INVALID_ARG
    assert L.cf_ffn_get_status(None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_ffn_launch_info(None, None, None, None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_ffn_kernels(None, 1, None, None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_ffn_set_timeline(None, None) == binding.CF_ERR_INVALID_ARG
    L.cf_ffn_destroy(None)  # NULL-safe


def test_null_arguments():
    rc, _ = binding.cf_create_rc(None)
    assert rc == binding.CF_ERR_INVALID_ARG
    L = binding.lib()
    assert L.cf_create(ctypes.byref(_cfg()), None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_decode_attn_block(None, 1, *([None] * 9)) == binding.CF_ERR_INVALID_ARG
    assert L.cf_get_status(None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_set_debug(None, None) == binding.CF_ERR_INVALID_ARG
    assert L.cf_get_launch_info(None, None) == binding.CF_ERR_INVALID_ARG
    L.cf_destroy(None)  # NULL-safe


def test_package_import_loads_no_library_and_fails_loudly_when_missing(tmp_path, monkeypatch):
    import attention_block_gb300.build as b
    monkeypatch.setattr(b, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError):
        binding.lib(build_if_missing=False)


MLA_BASE = dict(hidden=2048, n_heads=16, d_nope=128, d_rope=64, d_v=128, d_latent=512,
                max_batch=1, s_max=4097, rope_theta=1e4, rms_eps=1e-6, dtype=binding.CF_BF16)


@pytest.mark.parametrize("kw,code", [
    (dict(hidden=0), binding.CF_ERR_INVALID_ARG),
    (dict(s_max=0), binding.CF_ERR_INVALID_ARG),
    (dict(rope_theta=0.0), binding.CF_ERR_INVALID_ARG),
    (dict(rms_eps=-1.0), binding.CF_ERR_INVALID_ARG),
    (dict(dtype=7), binding.CF_ERR_INVALID_ARG),
    (dict(d_latent=256), binding.CF_ERR_UNSUPPORTED),
    (dict(d_rope=32), binding.CF_ERR_UNSUPPORTED),
    (dict(dtype=binding.CF_F32), binding.CF_ERR_UNSUPPORTED),
    (dict(n_heads=12), binding.CF_ERR_UNSUPPORTED),
    (dict(n_heads=64), binding.CF_ERR_UNSUPPORTED),
    (dict(hidden=2000), binding.CF_ERR_UNSUPPORTED),
    (dict(hidden=32768), binding.CF_ERR_UNSUPPORTED),
    (dict(max_batch=5), binding.CF_ERR_UNSUPPORTED),
])
def test_mla_create_rejects_bad_config_before_cuda(kw, code):
    cfg = dict(MLA_BASE)
    cfg.update(kw)
    c = binding.CfMlaConfig(*(cfg[k] for k in ("hidden", "n_heads", "d_nope", "d_rope", "d_v",
                                               "d_latent", "max_batch", "s_max", "rope_theta",
                                               "rms_eps", "dtype")))
    rc, h = binding.cf_mla_create_rc(c)
    assert rc == code and not h


def test_mla_null_arguments():
    assert binding.cf_mla_create_rc(None)[0] == binding.CF_ERR_INVALID_ARG
    lib = binding.lib()
    assert lib.cf_mla_decode(None, 1, *([None] * 11)) == binding.CF_ERR_INVALID_ARG
    assert lib.cf_mla_get_status(None) == binding.CF_ERR_INVALID_ARG
    lib.cf_mla_destroy(None)
