"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI, run the float64 oracle on the same seeded inputs, compare.

Tolerance (stated for fp16/bf16 storage with fp32 accumulation, used for
every storage type): max |gpu - ref| <= 1e-2 * max |ref| + 1e-3, and mean
relative error sum|gpu - ref| / sum|ref| <= 1e-3.  Values the GPU rounds to
the storage type (out, the appended K/V slot) are compared with the oracle's
float64 result rounded once (round-to-nearest-even) to that same type, so
the bound measures the arithmetic of the path and not the storage rounding
itself; fp32 intermediates are compared with the unrounded oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from attention_block_gb300 import binding, synth

MAX_ABS_REL = 1e-2
MAX_ABS_ADD = 1e-3
MEAN_REL = 1e-3


def round_to(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once (RNE) to the storage dtype, back to float64."""
    t = torch.from_numpy(np.ascontiguousarray(ref)).to(synth.DTYPES[dtype])
    return t.to(torch.float64).numpy()


def storage_ulp(values: np.ndarray, dtype: str) -> float:
    """One unit in the last place of the storage type at the largest
    magnitude of `values` (0 for fp32 storage)."""
    bits = {"f16": 10, "bf16": 7}.get(dtype)
    m = float(np.max(np.abs(values))) if np.size(values) else 0.0
    if bits is None or m == 0.0:
        return 0.0
    return 2.0 ** (np.floor(np.log2(m)) - bits)


def check(gpu, ref, what: str, mean_rel: float = MEAN_REL, floor: float = 0.0):
    """`floor` widens the max bound for differences of values that were each
    rounded to the storage type (e.g. out - hidden): one rounding flip of
    the output moves such a difference by one storage ulp of the output."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    err = np.abs(gpu - ref)
    bound = MAX_ABS_REL * np.max(np.abs(ref)) + MAX_ABS_ADD + floor
    mre = err.sum() / max(np.abs(ref).sum(), 1e-300)
    assert err.max() <= bound, f"{what}: max|err| {err.max():.3e} > {bound:.3e}"
    assert mre <= mean_rel, f"{what}: mean rel err {mre:.3e} > {mean_rel:.1e}"
    return float(err.max()), float(mre)


def dbg_size(w: synth.Workload, batch: int) -> int:
    d = w.head_dim
    return batch * (2 * w.n_q_heads * d + 2 * w.n_kv_heads * d + w.hidden)


def split_dbg(dbg: torch.Tensor, w: synth.Workload, batch: int) -> dict:
    d, nq, nkv, H = w.head_dim, w.n_q_heads, w.n_kv_heads, w.hidden
    sizes = [("q", nq * d), ("k", nkv * d), ("v", nkv * d), ("o", nq * d), ("proj", H)]
    out, off = {}, 0
    flat = dbg.double().cpu().numpy()
    for name, n in sizes:
        out[name] = flat[off: off + batch * n].reshape(batch, n)
        off += batch * n
    return out


def make_block(w: synth.Workload, **tune) -> binding.DecodeAttnBlock:
    return binding.DecodeAttnBlock(
        hidden=w.hidden, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
        max_batch=w.batch, s_max=w.s_max, rope_theta=w.rope_theta, rms_eps=w.rms_eps,
        dtype=w.dtype, **tune)


def run_gpu(w: synth.Workload, t: dict, block=None, debug: bool = False, unfused: bool = False,
            **tune):
    """One fused decode step on the GPU; returns (out, k_cache, v_cache, dbg).

    ``t`` holds the layer's device tensors (they are cloned, not modified).
    """
    blk = block or make_block(w, **tune)
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    out = torch.empty_like(t["hidden"])
    dbg = None
    if debug:
        dbg = torch.full((dbg_size(w, w.batch),), float("nan"), dtype=torch.float32,
                         device=t["hidden"].device)
        blk.set_debug(dbg)
    step = blk.unfused if unfused else blk
    step(w.batch, t["hidden"], t["ln_weight"], t["w_qkv"], t["w_o"], kc, vc, t["positions"], out)
    torch.cuda.synchronize()
    st = binding.cf_get_status(blk.handle)
    if debug:
        blk.set_debug(None)
    return out, kc, vc, dbg, st


def run_oracle(w: synth.Workload, t: dict, rows=None, hidden=None):
    """Oracle on the same inputs (rows: subset of batch rows).

    Returns dict of stacked float64 results plus the updated cache slots.
    """
    rows = list(range(w.batch)) if rows is None else list(rows)
    x = synth.to_f64(t["hidden"] if hidden is None else hidden)
    g = synth.to_f64(t["ln_weight"])
    wqkv = synth.to_f64(t["w_qkv"])
    wo = synth.to_f64(t["w_o"])
    pos = t["positions"].cpu().numpy()
    res = {k: [] for k in ("out", "q", "k", "v", "o", "proj", "kslot", "vslot")}
    for b in rows:
        kc = synth.to_f64(t["k_cache"][b])
        vc = synth.to_f64(t["v_cache"][b])
        r = oracle.decode_row(w.oracle_cfg(), x[b], g, wqkv, wo, kc, vc, int(pos[b]))
        for k in ("out", "q", "k", "v", "o", "proj"):
            res[k].append(r[k])
        res["kslot"].append(kc[int(pos[b])].reshape(-1).copy())
        res["vslot"].append(vc[int(pos[b])].reshape(-1).copy())
    return {k: np.stack(v) for k, v in res.items()}


def check_cache_untouched_except_slot(before: torch.Tensor, after: torch.Tensor, positions):
    """Bit-exact: every cache byte except [b, positions[b]] is unchanged."""
    mask = torch.ones(before.shape[:2], dtype=torch.bool, device=before.device)
    for b, p in enumerate(positions):
        if 0 <= p < before.shape[1]:
            mask[b, p] = False
    assert torch.equal(before[mask], after[mask]), "cache bytes outside the new slot changed"


def full_check(w, seed=0, rows=None, debug=True, t=None, **tune):
    t = t if t is not None else synth.make_layer(w, seed, device="cuda")
    out, kc, vc, dbg, st = run_gpu(w, t, debug=debug, **tune)
    assert st == binding.CF_OK, binding.strerror(st)
    rows = list(range(w.batch)) if rows is None else list(rows)
    ref = run_oracle(w, t, rows)
    pos = t["positions"].tolist()
    check(out[rows].double().cpu().numpy(), round_to(ref["out"], w.dtype), "out")
    check_cache_untouched_except_slot(t["k_cache"], kc, pos)
    check_cache_untouched_except_slot(t["v_cache"], vc, pos)
    ks = torch.stack([kc[b, pos[b]].reshape(-1) for b in rows]).double().cpu().numpy()
    vs = torch.stack([vc[b, pos[b]].reshape(-1) for b in rows]).double().cpu().numpy()
    check(ks, round_to(ref["kslot"], w.dtype), "k slot")
    check(vs, round_to(ref["vslot"], w.dtype), "v slot")
    if debug:
        d = split_dbg(dbg, w, w.batch)
        # fp32 on-chip intermediates against the unrounded oracle
        for name in ("q", "k", "v", "o", "proj"):
            check(d[name][rows], ref[name], name)
    return out, ref
