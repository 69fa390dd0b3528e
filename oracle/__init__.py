"""float64 CPU oracle of the decode attention block -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding in ``attention_block_gb300``) never imports, links or calls it,
and this package imports nothing from the product path.

The arithmetic lives in ``oracle.c`` (plain single-threaded float64 C); this
module only compiles it, loads it with ctypes and marshals numpy arrays.
Setting ``CF_ORACLE_LIB`` loads another build of oracle.c instead (used by
the mutation tests, which plant mistakes in temporary copies).
See ``oracle.h`` for the definitions and the page passages each one follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


class OrcConfig(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int),
        ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("s_max", ctypes.c_int),
        ("rope_theta", ctypes.c_double),
        ("rms_eps", ctypes.c_double),
    ]


class OrcMlaConfig(ctypes.Structure):
    _fields_ = [
        ("hidden", ctypes.c_int),
        ("n_heads", ctypes.c_int),
        ("d_nope", ctypes.c_int),
        ("d_rope", ctypes.c_int),
        ("d_v", ctypes.c_int),
        ("d_latent", ctypes.c_int),
        ("s_max", ctypes.c_int),
        ("rope_theta", ctypes.c_double),
        ("rms_eps", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (no fast-math, no FMA contraction)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            override = os.environ.get("CF_ORACLE_LIB")
            lib = ctypes.CDLL(override if override else build())
            lib.orc_rmsnorm.argtypes = [ctypes.c_int, _dp, _dp, ctypes.c_double, _dp]
            lib.orc_matvec.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp, _dp]
            lib.orc_rope.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_int, _dp]
            lib.orc_attention.argtypes = [ctypes.c_int, ctypes.c_int, _dp, _dp,
                                          ctypes.c_ssize_t, _dp, ctypes.c_ssize_t,
                                          _dp, _dp]
            lib.orc_attention_split.argtypes = [
                ctypes.c_int, ctypes.c_int, _dp, _dp, ctypes.c_ssize_t, _dp,
                ctypes.c_ssize_t, ctypes.c_int, ctypes.POINTER(ctypes.c_int), _dp]
            lib.orc_decode_row.argtypes = [ctypes.POINTER(OrcConfig), _dp, _dp, _dp,
                                           _dp, _dp, _dp, ctypes.c_int, _dp, _dp,
                                           _dp, _dp, _dp, _dp, _dp]
            lib.orc_decode_row.restype = ctypes.c_int
            lib.orc_silu.argtypes = [ctypes.c_double]
            lib.orc_silu.restype = ctypes.c_double
            lib.orc_ffn_row.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double] + [_dp] * 9
            lib.orc_ffn_row.restype = ctypes.c_int
            lib.orc_mla_row.argtypes = [ctypes.POINTER(OrcMlaConfig)] + [_dp] * 8 + [
                ctypes.c_int] + [_dp] * 5
            lib.orc_mla_row.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x, g = _f64(x), _f64(g)
    n = np.empty_like(x)
    _load().orc_rmsnorm(x.shape[0], _p(x), _p(g), float(eps), _p(n))
    return n


def matvec(x, W) -> np.ndarray:
    """y = x . W for W [K, N] row-major."""
    x, W = _f64(x), _f64(W)
    K, N = W.shape
    assert x.shape == (K,)
    y = np.empty(N, dtype=np.float64)
    _load().orc_matvec(K, N, _p(x), _p(W), _p(y))
    return y


def rope(u, pos: int, theta: float) -> np.ndarray:
    u = _f64(u).copy()
    _load().orc_rope(u.shape[0], float(theta), int(pos), _p(u))
    return u


def attention(q, K, V):
    """Two-pass softmax attention of q [d] over K, V [ntok, d] -> (o, w)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    ntok, d = K.shape
    o = np.empty(d, dtype=np.float64)
    w = np.empty(ntok, dtype=np.float64)
    _load().orc_attention(d, ntok, _p(q), _p(K), d, _p(V), d, _p(o), _p(w))
    return o, w


def attention_split(q, K, V, chunk_ends) -> np.ndarray:
    q, K, V = _f64(q), _f64(K), _f64(V)
    ntok, d = K.shape
    ends = (ctypes.c_int * len(chunk_ends))(*[int(e) for e in chunk_ends])
    assert list(chunk_ends)[-1] == ntok
    o = np.empty(d, dtype=np.float64)
    _load().orc_attention_split(d, ntok, _p(q), _p(K), d, _p(V), d,
                                len(chunk_ends), ends, _p(o))
    return o


def decode_row(cfg: dict, x, g, wqkv, wo, kc, vc, pos: int):
    """One batch row.  kc, vc: float64 [S, nkv, d] arrays, updated in place.

    cfg keys: hidden, n_q_heads, n_kv_heads, head_dim, s_max, rope_theta,
    rms_eps.  Returns a dict with out, n, q, k, v, o, proj (float64).
    """
    c = OrcConfig(int(cfg["hidden"]), int(cfg["n_q_heads"]), int(cfg["n_kv_heads"]),
                  int(cfg["head_dim"]), int(cfg["s_max"]), float(cfg["rope_theta"]),
                  float(cfg["rms_eps"]))
    H, nq, nkv, d = c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim
    x, g, wqkv, wo = _f64(x), _f64(g), _f64(wqkv), _f64(wo)
    assert kc.dtype == np.float64 and kc.flags.c_contiguous
    assert vc.dtype == np.float64 and vc.flags.c_contiguous
    assert kc.shape == (c.s_max, nkv, d) and vc.shape == kc.shape
    res = {k: np.empty(n, dtype=np.float64) for k, n in (
        ("out", H), ("n", H), ("q", nq * d), ("k", nkv * d), ("v", nkv * d),
        ("o", nq * d), ("proj", H))}
    rc = _load().orc_decode_row(ctypes.byref(c), _p(x), _p(g), _p(wqkv), _p(wo),
                                _p(kc), _p(vc), int(pos), _p(res["out"]), _p(res["n"]),
                                _p(res["q"]), _p(res["k"]), _p(res["v"]), _p(res["o"]),
                                _p(res["proj"]))
    if rc != 0:
        raise ValueError(f"oracle rejected row (pos={pos}, cfg={cfg})")
    return res


def decode(cfg: dict, X, g, wqkv, wo, KC, VC, positions, rows=None):
    """Batch form: X [B, H]; KC, VC float64 [B, S, nkv, d] (updated in place).

    ``rows`` selects a subset of batch rows (default: all).  Returns a dict of
    stacked per-row results for the selected rows.
    """
    rows = range(X.shape[0]) if rows is None else rows
    outs = [decode_row(cfg, X[b], g, wqkv, wo, KC[b], VC[b], int(positions[b]))
            for b in rows]
    return {k: np.stack([o[k] for o in outs]) for k in outs[0]}


def silu(z: float) -> float:
    return float(_load().orc_silu(float(z)))


def ffn_row(h, g2, wg, wu, wd, eps: float):
    """Second RMSNorm + SwiGLU FFN + residual for one row h [H]; wg, wu, wd
    are [I, H].  Returns a dict with out, n, a, proj (float64)."""
    h, g2, wg, wu, wd = _f64(h), _f64(g2), _f64(wg), _f64(wu), _f64(wd)
    H = h.shape[0]
    I = wg.shape[0]
    assert wg.shape == (I, H) and wu.shape == (I, H) and wd.shape == (I, H)
    res = {"out": np.empty(H), "n": np.empty(H), "a": np.empty(I), "proj": np.empty(H)}
    rc = _load().orc_ffn_row(H, I, float(eps), _p(h), _p(g2), _p(wg), _p(wu), _p(wd),
                             _p(res["out"]), _p(res["n"]), _p(res["a"]), _p(res["proj"]))
    if rc != 0:
        raise ValueError("oracle rejected the FFN shape")
    return res


def ffn(Hs, g2, wg, wu, wd, eps: float, rows=None):
    """Batch form of ffn_row over the rows of Hs [B, H] (or the selected rows)."""
    rows = range(Hs.shape[0]) if rows is None else rows
    outs = [ffn_row(Hs[b], g2, wg, wu, wd, eps) for b in rows]
    return {k: np.stack([o[k] for o in outs]) for k in outs[0]}


def mla_row(cfg: dict, x, g, wq, wdkv, g_kv, wukv, wo, lc, pos: int):
    """One batch row of the MLA decode block (oracle.h, orc_mla_row).  lc is
    this row's latent cache, a float64 [S, dc+dr] array updated in place.

    cfg keys: hidden, n_heads, d_nope, d_rope, d_v, d_latent, s_max,
    rope_theta, rms_eps.  Returns a dict with out, q, lat, o, proj.
    """
    c = OrcMlaConfig(*(int(cfg[k]) for k in ("hidden", "n_heads", "d_nope", "d_rope", "d_v",
                                              "d_latent", "s_max")),
                     float(cfg["rope_theta"]), float(cfg["rms_eps"]))
    H, nh, dn, dr, dv, dc = c.hidden, c.n_heads, c.d_nope, c.d_rope, c.d_v, c.d_latent
    x, g, wq, wdkv, g_kv, wukv, wo = (_f64(a) for a in (x, g, wq, wdkv, g_kv, wukv, wo))
    assert wq.shape == (H, nh * (dn + dr)) and wdkv.shape == (H, dc + dr)
    assert wukv.shape == (dc, nh * (dn + dv)) and wo.shape == (nh * dv, H)
    assert lc.dtype == np.float64 and lc.flags.c_contiguous and lc.shape == (c.s_max, dc + dr)
    res = {k: np.empty(n, dtype=np.float64) for k, n in (
        ("out", H), ("q", nh * (dn + dr)), ("lat", dc + dr), ("o", nh * dv), ("proj", H))}
    rc = _load().orc_mla_row(ctypes.byref(c), _p(x), _p(g), _p(wq), _p(wdkv), _p(g_kv),
                             _p(wukv), _p(wo), _p(lc), int(pos), _p(res["out"]), _p(res["q"]),
                             _p(res["lat"]), _p(res["o"]), _p(res["proj"]))
    if rc != 0:
        raise ValueError(f"oracle rejected the MLA row (pos={pos}, cfg={cfg})")
    return res
