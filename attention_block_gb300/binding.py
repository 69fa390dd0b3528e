"""ctypes binding of libcf.so (include/cf.h, include/cf_test.h).

Argument marshalling only: every step of the decode block runs in the CUDA
library.  There is no fallback of any kind -- if the library is missing or
was not built, ``lib()`` raises.  Tensors may be passed as torch tensors
(their ``data_ptr()`` is used) or as raw integer addresses.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

CF_OK = 0
CF_ERR_INVALID_ARG = -1
CF_ERR_UNSUPPORTED = -2
CF_ERR_ALIAS = -3
CF_ERR_CLUSTER = -4
CF_ERR_CUDA = -5
CF_ERR_DEVICE_POS_RANGE = -6
CF_ERR_DEVICE_TIMEOUT = -7

CF_F32, CF_F16, CF_BF16 = 0, 1, 2


class CfConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "n_q_heads", "n_kv_heads", "head_dim", "max_batch", "s_max")] + [
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)] + [
        (n, ctypes.c_int32) for n in (
            "dtype", "cluster_size", "batch_tile", "stage_bytes", "ctas_per_sm",
            "pdl", "max_stages", "rows_per_block", "adaptive")]


class CfFfnConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("max_batch", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("dtype", ctypes.c_int32), ("stage_bytes", ctypes.c_int32)]


class CfMlaConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "n_heads", "d_nope", "d_rope", "d_v", "d_latent", "max_batch", "s_max")] + [
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("dtype", ctypes.c_int32)]


class CfLaunchInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "cluster_size", "batch_tile", "group", "rows_per_wtile", "pos_per_ktile",
        "wo_rows_per_tile", "wo_cols_per_tile", "stages", "stage_bytes", "smem_bytes",
        "threads", "max_active_clusters", "sm_count", "mode", "rows_per_block")]


class CfError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else
                         f"{strerror(code)} ({code})")


_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p

# Exported symbols, with (restype, argtypes).
SIGNATURES = {
    "cf_create": (ctypes.c_int, [ctypes.POINTER(CfConfig), ctypes.POINTER(_vp)]),
    "cf_decode_attn_block": (ctypes.c_int, [_vp, ctypes.c_int32] + [_vp] * 9),
    "cf_decode_attn_block_unfused": (ctypes.c_int, [_vp, ctypes.c_int32] + [_vp] * 9),
    "cf_get_status": (ctypes.c_int, [_vp]),
    "cf_set_debug": (ctypes.c_int, [_vp, _vp]),
    "cf_get_launch_info": (ctypes.c_int, [_vp, ctypes.POINTER(CfLaunchInfo)]),
    "cf_get_launch_info_batch": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.POINTER(CfLaunchInfo)]),
    "cf_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "cf_destroy": (None, [_vp]),
    "cf_test_cluster_allreduce": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 _vp, _vp, _vp, _vp]),
    "cf_test_cluster_reduce_scatter": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _vp, _vp,
                                                      _vp, _vp]),
    "cf_test_cluster_gather": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp]),
    "cf_test_tc05_gemm": (ctypes.c_int, [ctypes.c_int] * 4 + [_vp] * 5),
    "cf_test_lost_transfer": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_longlong,
                                             _vp, _vp, _vp, _vp]),
    "cf_bench_cluster_collective": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                   _vp, _vp, _vp, _vp, _vp]),
    "cf_set_timeline": (ctypes.c_int, [_vp, _vp]),
    "cf_ffn_create": (ctypes.c_int, [ctypes.POINTER(CfFfnConfig), ctypes.POINTER(_vp)]),
    "cf_ffn_forward": (ctypes.c_int, [_vp, ctypes.c_int32] + [_vp] * 7),
    "cf_ffn_get_status": (ctypes.c_int, [_vp]),
    "cf_ffn_launch_info": (ctypes.c_int, [_vp] + [ctypes.POINTER(ctypes.c_int32)] * 3),
    "cf_ffn_destroy": (None, [_vp]),
    "cf_ffn_kernels": (ctypes.c_int, [_vp, ctypes.c_int32] + [ctypes.POINTER(ctypes.c_int32)] * 2),
    "cf_ffn_set_timeline": (ctypes.c_int, [_vp, _vp]),
    "cf_ffn_debug_a": (ctypes.c_int, [_vp, ctypes.c_int32, _vp]),
    "cf_decode_attn_block_noalloc": (ctypes.c_int, [ctypes.POINTER(CfConfig), ctypes.c_int32]
                                     + [_vp] * 9),
    "cf_noalloc_get_status": (ctypes.c_int, []),
    "cf_mla_create": (ctypes.c_int, [ctypes.POINTER(CfMlaConfig), ctypes.POINTER(_vp)]),
    "cf_mla_decode": (ctypes.c_int, [_vp, ctypes.c_int32] + [_vp] * 11),
    "cf_mla_get_status": (ctypes.c_int, [_vp]),
    "cf_mla_launch_info": (ctypes.c_int, [_vp] + [ctypes.POINTER(ctypes.c_int32)] * 5),
    "cf_mla_destroy": (None, [_vp]),
    "cf_mla_set_timeline": (ctypes.c_int, [_vp, _vp]),
}

TIMELINE_SLOTS = 32
TIMELINE_NAMES = ["start", "norm", "proj", "reduce_scatter", "gather", "attn", "merge", "sum",
                  "oproj", "final", "prod_w", "prod_kv", "prod_all", "end", "proj_loop",
                  "proj_loop_last_warp", "rinv", "attn_first_tile", "oproj_first_tile",
                  "oproj_loop", "ticket", "oproj_tile1", "oproj_tile2", "oproj_tile3",
                  "attn_loop", "attn_warps"]
MLA_TIMELINE_NAMES = ["start", "norm", "A", "bar1", "B", "bar2", "C_first_tile", "C_tiles",
                      "C_merged", "bar3", "D_wuv", "D_allreduce", "D_wo", "end", "prod_A",
                      "prod_C", "prod_D"]
# Timeline slot holding the block's SM id (a value, not a time).
TIMELINE_SMID = 26


def lib_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """Load libcf.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            if build_if_missing and _build.is_stale():
                _build.build()
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing; run "
                                   "attention_block_gb300.build.build() (needs nvcc)")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def strerror(code: int) -> str:
    try:
        return lib().cf_strerror(int(code)).decode()
    except Exception:  # message lookup must never mask the original error
        return f"error {code}"


def make_config(hidden, n_q_heads, n_kv_heads, head_dim, max_batch, s_max, rope_theta=1e4,
                rms_eps=1e-6, dtype=CF_F16, cluster_size=0, batch_tile=0, stage_bytes=0,
                ctas_per_sm=0, pdl=0, max_stages=0, rows_per_block=0,
                adaptive=0) -> CfConfig:
    if isinstance(dtype, str):
        dtype = {"f32": CF_F32, "f16": CF_F16, "bf16": CF_BF16}[dtype]
    return CfConfig(int(hidden), int(n_q_heads), int(n_kv_heads), int(head_dim),
                    int(max_batch), int(s_max), float(rope_theta), float(rms_eps), int(dtype),
                    int(cluster_size), int(batch_tile), int(stage_bytes), int(ctas_per_sm),
                    int(pdl), int(max_stages), int(rows_per_block), int(adaptive))


def cf_create(cfg: CfConfig) -> int:
    h = _vp()
    rc = lib().cf_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc != CF_OK:
        raise CfError(rc, "cf_create")
    return h.value


def cf_create_rc(cfg: CfConfig | None) -> tuple[int, int | None]:
    """Return code and handle without raising (boundary tests)."""
    h = _vp()
    rc = lib().cf_create(ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(h))
    return rc, h.value


def cf_decode_attn_block(handle, batch, hidden_states, ln_weight, w_qkv, w_o, k_cache, v_cache,
                         positions, out, stream=None) -> int:
    return lib().cf_decode_attn_block(handle, int(batch), _ptr(hidden_states), _ptr(ln_weight),
                                      _ptr(w_qkv), _ptr(w_o), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(positions), _ptr(out), _stream(stream))


def cf_decode_attn_block_unfused(handle, batch, hidden_states, ln_weight, w_qkv, w_o, k_cache,
                                 v_cache, positions, out, stream=None) -> int:
    """The same step as three kernels with HBM intermediates (fusion baseline)."""
    return lib().cf_decode_attn_block_unfused(handle, int(batch), _ptr(hidden_states),
                                              _ptr(ln_weight), _ptr(w_qkv), _ptr(w_o),
                                              _ptr(k_cache), _ptr(v_cache), _ptr(positions),
                                              _ptr(out), _stream(stream))


def cf_decode_attn_block_noalloc(cfg: CfConfig, batch, hidden_states, ln_weight, w_qkv, w_o,
                                 k_cache, v_cache, positions, out, stream=None) -> int:
    """Allocation-free decode step (no handle; scratch in a static device array)."""
    return lib().cf_decode_attn_block_noalloc(
        ctypes.byref(cfg), int(batch), _ptr(hidden_states), _ptr(ln_weight), _ptr(w_qkv),
        _ptr(w_o), _ptr(k_cache), _ptr(v_cache), _ptr(positions), _ptr(out), _stream(stream))


def cf_noalloc_get_status() -> int:
    """Read and clear the error word of the allocation-free calls (current device)."""
    return lib().cf_noalloc_get_status()


def cf_get_status(handle) -> int:
    return lib().cf_get_status(handle)


def cf_set_debug(handle, dbg) -> int:
    return lib().cf_set_debug(handle, _ptr(dbg))


def cf_get_launch_info(handle, batch=None) -> dict:
    """What the handle launches for max_batch rows, or for `batch` rows."""
    info = CfLaunchInfo()
    if batch is None:
        rc = lib().cf_get_launch_info(handle, ctypes.byref(info))
    else:
        rc = lib().cf_get_launch_info_batch(handle, int(batch), ctypes.byref(info))
    if rc != CF_OK:
        raise CfError(rc, "cf_get_launch_info")
    return {n: getattr(info, n) for n, _ in CfLaunchInfo._fields_}


def cf_set_timeline(handle, stamps) -> int:
    return lib().cf_set_timeline(handle, _ptr(stamps))


def cf_strerror(code: int) -> str:
    return strerror(code)


def cf_destroy(handle) -> None:
    lib().cf_destroy(handle)


def cf_test_cluster_allreduce(cluster_size, op, n, inp, out, errflag, stream=None) -> int:
    return lib().cf_test_cluster_allreduce(int(cluster_size), int(op), int(n), _ptr(inp),
                                           _ptr(out), _ptr(errflag), _stream(stream))


def cf_test_cluster_reduce_scatter(cluster_size, n, inp, out, errflag, stream=None) -> int:
    return lib().cf_test_cluster_reduce_scatter(int(cluster_size), int(n), _ptr(inp), _ptr(out),
                                                _ptr(errflag), _stream(stream))


def cf_test_cluster_gather(cluster_size, n, inp, out, errflag, stream=None) -> int:
    return lib().cf_test_cluster_gather(int(cluster_size), int(n), _ptr(inp), _ptr(out),
                                        _ptr(errflag), _stream(stream))


def cf_test_lost_transfer(n, drop_rank, limit_cycles, inp, out, errflag, stream=None) -> int:
    return lib().cf_test_lost_transfer(int(n), int(drop_rank), int(limit_cycles), _ptr(inp),
                                       _ptr(out), _ptr(errflag), _stream(stream))


def cf_test_tc05_gemm(dtype, n, k, a, b, d, errflag, stream=None, a_mn=False) -> int:
    return lib().cf_test_tc05_gemm(int(dtype), int(bool(a_mn)), int(n), int(k), _ptr(a), _ptr(b),
                                   _ptr(d), _ptr(errflag), _stream(stream))


def cf_bench_cluster_collective(kind, cluster_size, n, inp, out, errflag, cycles,
                                stream=None) -> int:
    return lib().cf_bench_cluster_collective(int(kind), int(cluster_size), int(n), _ptr(inp),
                                             _ptr(out), _ptr(errflag), _ptr(cycles),
                                             _stream(stream))


class DecodeAttnBlock:
    """Owns one cf_handle; calling it enqueues one fused decode step.

    Raises CfError on any non-zero return code.  ``status()`` synchronizes
    the current device and reads (and clears) the device error flag.
    """

    def __init__(self, **cfg):
        self.cfg = make_config(**cfg)
        self.handle = cf_create(self.cfg)

    def __call__(self, batch, hidden_states, ln_weight, w_qkv, w_o, k_cache, v_cache, positions,
                 out, stream=None):
        rc = cf_decode_attn_block(self.handle, batch, hidden_states, ln_weight, w_qkv, w_o,
                                  k_cache, v_cache, positions, out, stream)
        if rc != CF_OK:
            raise CfError(rc, "cf_decode_attn_block")
        return out

    def unfused(self, batch, hidden_states, ln_weight, w_qkv, w_o, k_cache, v_cache, positions,
                out, stream=None):
        """The same step through the three-kernel path (the fusion baseline)."""
        rc = cf_decode_attn_block_unfused(self.handle, batch, hidden_states, ln_weight, w_qkv, w_o,
                                          k_cache, v_cache, positions, out, stream)
        if rc != CF_OK:
            raise CfError(rc, "cf_decode_attn_block_unfused")
        return out

    def launch_info(self, batch=None) -> dict:
        return cf_get_launch_info(self.handle, batch)

    def set_debug(self, dbg) -> None:
        rc = cf_set_debug(self.handle, dbg)
        if rc != CF_OK:
            raise CfError(rc, "cf_set_debug")

    def status(self) -> int:
        import torch
        torch.cuda.synchronize()
        return cf_get_status(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            cf_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------- FFN --
def cf_ffn_create(cfg: CfFfnConfig) -> int:
    h = _vp()
    rc = lib().cf_ffn_create(ctypes.byref(cfg), ctypes.byref(h))
    if rc != CF_OK:
        raise CfError(rc, "cf_ffn_create")
    return h.value


def cf_ffn_forward(handle, batch, hidden, ln_weight, w_gate, w_up, w_down, out,
                   stream=None) -> int:
    return lib().cf_ffn_forward(handle, int(batch), _ptr(hidden), _ptr(ln_weight), _ptr(w_gate),
                                _ptr(w_up), _ptr(w_down), _ptr(out), _stream(stream))


class FfnBlock:
    """Owns one cf_ffn_handle; calling it enqueues the second RMSNorm, the
    gated FFN and the residual for ``batch`` rows.  Raises CfError on any
    non-zero return code."""

    def __init__(self, hidden, intermediate, max_batch, rms_eps=1e-6, dtype=CF_F16,
                 stage_bytes=0):
        if isinstance(dtype, str):
            dtype = {"f32": CF_F32, "f16": CF_F16, "bf16": CF_BF16}[dtype]
        self.cfg = CfFfnConfig(int(hidden), int(intermediate), int(max_batch), float(rms_eps),
                               int(dtype), int(stage_bytes))
        self.handle = cf_ffn_create(self.cfg)

    def __call__(self, batch, hidden, ln_weight, w_gate, w_up, w_down, out, stream=None):
        rc = cf_ffn_forward(self.handle, batch, hidden, ln_weight, w_gate, w_up, w_down, out,
                            stream)
        if rc != CF_OK:
            raise CfError(rc, "cf_ffn_forward")
        return out

    def launch_info(self) -> dict:
        b, r, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        rc = lib().cf_ffn_launch_info(self.handle, ctypes.byref(b), ctypes.byref(r),
                                      ctypes.byref(s))
        if rc != CF_OK:
            raise CfError(rc, "cf_ffn_launch_info")
        return {"blocks": b.value, "rows_per_stage": r.value, "stages": s.value}

    def kernels(self, batch) -> dict:
        """Kernels (1: the one- and two-row kernel, 2: the tensor-core pair)
        and grids a call of ``batch`` rows launches."""
        b1, b2 = ctypes.c_int32(), ctypes.c_int32()
        n = lib().cf_ffn_kernels(self.handle, int(batch), ctypes.byref(b1), ctypes.byref(b2))
        if n < 0:
            raise CfError(n, "cf_ffn_kernels")
        return {"kernels": n, "blocks1": b1.value, "blocks2": b2.value}

    def debug_a(self, batch):
        """The last call's intermediate activations [batch, I] (tensor-core
        pair only), read back from the device as a float64 numpy array."""
        import numpy as np
        a = np.empty((int(batch), int(self.cfg.intermediate)), dtype=np.float32)
        rc = lib().cf_ffn_debug_a(self.handle, int(batch), a.ctypes.data)
        if rc != CF_OK:
            raise CfError(rc, "cf_ffn_debug_a")
        return a.astype(np.float64)

    def status(self) -> int:
        import torch
        torch.cuda.synchronize()
        return lib().cf_ffn_get_status(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().cf_ffn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------- MLA --
def cf_mla_create_rc(cfg: CfMlaConfig | None) -> tuple[int, int | None]:
    """Return code and handle without raising (boundary tests)."""
    h = _vp()
    rc = lib().cf_mla_create(ctypes.byref(cfg) if cfg is not None else None, ctypes.byref(h))
    return rc, h.value


def cf_mla_decode(handle, batch, hidden, ln_weight, w_q, w_dkv, kv_norm_weight, w_ukv, w_o,
                  latent_cache, positions, out, stream=None) -> int:
    return lib().cf_mla_decode(handle, int(batch), _ptr(hidden), _ptr(ln_weight), _ptr(w_q),
                               _ptr(w_dkv), _ptr(kv_norm_weight), _ptr(w_ukv), _ptr(w_o),
                               _ptr(latent_cache), _ptr(positions), _ptr(out), _stream(stream))


class MlaBlock:
    """Owns one cf_mla_handle; calling it enqueues one MLA decode step
    (include/cf_mla.h).  Raises CfError on any non-zero return code."""

    def __init__(self, hidden, n_heads, max_batch, s_max, rope_theta=1e4, rms_eps=1e-6,
                 dtype=CF_BF16, d_nope=128, d_rope=64, d_v=128, d_latent=512):
        if isinstance(dtype, str):
            dtype = {"f32": CF_F32, "f16": CF_F16, "bf16": CF_BF16}[dtype]
        self.cfg = CfMlaConfig(int(hidden), int(n_heads), int(d_nope), int(d_rope), int(d_v),
                               int(d_latent), int(max_batch), int(s_max), float(rope_theta),
                               float(rms_eps), int(dtype))
        rc, h = cf_mla_create_rc(self.cfg)
        if rc != CF_OK:
            raise CfError(rc, "cf_mla_create")
        self.handle = h

    def __call__(self, batch, hidden, ln_weight, w_q, w_dkv, kv_norm_weight, w_ukv, w_o,
                 latent_cache, positions, out, stream=None):
        rc = cf_mla_decode(self.handle, batch, hidden, ln_weight, w_q, w_dkv, kv_norm_weight,
                           w_ukv, w_o, latent_cache, positions, out, stream)
        if rc != CF_OK:
            raise CfError(rc, "cf_mla_decode")
        return out

    def set_timeline(self, stamps) -> None:
        rc = lib().cf_mla_set_timeline(self.handle, _ptr(stamps))
        if rc != CF_OK:
            raise CfError(rc, "cf_mla_set_timeline")

    def launch_info(self) -> dict:
        v = [ctypes.c_int32() for _ in range(5)]
        rc = lib().cf_mla_launch_info(self.handle, *[ctypes.byref(x) for x in v])
        if rc != CF_OK:
            raise CfError(rc, "cf_mla_launch_info")
        return dict(zip(("clusters", "cluster_size", "stages", "stage_bytes", "smem_bytes"),
                        (x.value for x in v)))

    def status(self) -> int:
        import torch
        torch.cuda.synchronize()
        return lib().cf_mla_get_status(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            lib().cf_mla_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
