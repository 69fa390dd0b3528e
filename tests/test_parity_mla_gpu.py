"""GPU parity of the DeepSeek multi-head latent attention (MLA) variant
(cf_mla_decode, include/cf_mla.h) against the float64 oracle (orc_mla_row).

Page: "ClusterFusion框架深度解析" (devpress.csdn.net), §5.2 DeepSeek-MLA特殊处理.
Tolerance as in parity_util: max |gpu - ref| <= 1e-2 * max |ref| + 1e-3 and
sum |gpu - ref| / sum |ref| <= 1e-3, the storage-typed results against the
oracle rounded once to the storage type.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_block_gb300 import binding, synth
from parity_util import check, check_cache_untouched_except_slot, round_to, storage_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.lib()


def make_mla(w):
    return binding.MlaBlock(w.hidden, w.n_heads, w.batch, w.s_max, w.rope_theta, w.rms_eps,
                            w.dtype)


ARGS = ("hidden", "ln_weight", "w_q", "w_dkv", "kv_norm_weight", "w_ukv", "w_o")


def run_mla(w, t, blk=None, batch=None, x=None):
    blk = blk if blk is not None else make_mla(w)
    B = w.batch if batch is None else batch
    lc = t["latent_cache"].clone()
    out = torch.full_like(t["hidden"], float("nan"))
    args = [t[k] for k in ARGS]
    if x is not None:
        args[0] = x
    blk(B, *args, lc, t["positions"], out)
    return out, lc, blk.status()


def oracle_mla(w, t, rows=None, x=None):
    f = {k: synth.to_f64(t[k]) for k in ARGS}
    if x is not None:
        f["hidden"] = synth.to_f64(x)
    pos = t["positions"].tolist()
    rows = range(w.batch) if rows is None else rows
    res = {"out": [], "lat": []}
    for b in rows:
        lc = synth.to_f64(t["latent_cache"][b]).copy()
        r = oracle.mla_row(w.oracle_cfg(), f["hidden"][b], f["ln_weight"], f["w_q"], f["w_dkv"],
                           f["kv_norm_weight"], f["w_ukv"], f["w_o"], lc, int(pos[b]))
        res["out"].append(r["out"])
        res["lat"].append(r["lat"])
    return {k: np.stack(v) for k, v in res.items()}


def full_mla_check(w, seed=0, rows=None, t=None):
    t = t if t is not None else synth.make_mla_layer(w, seed, device="cuda")
    out, lc, st = run_mla(w, t)
    assert st == binding.CF_OK, binding.strerror(st)
    rows = list(range(w.batch)) if rows is None else rows
    ref = oracle_mla(w, t, rows)
    pos = t["positions"].tolist()
    got = out[rows].double().cpu().numpy()
    check(got, round_to(ref["out"], w.dtype), "out")
    # the attention's contribution, unmasked by the residual
    x = synth.to_f64(t["hidden"][rows])
    want = round_to(ref["out"], w.dtype)
    check(got - x, want - x, "out - hidden", floor=storage_ulp(want, w.dtype))
    slots = torch.stack([lc[b, pos[b]] for b in rows]).double().cpu().numpy()
    check(slots, round_to(ref["lat"], w.dtype), "latent slot")
    check_cache_untouched_except_slot(t["latent_cache"], lc, pos)
    return out, ref


def test_tiny_workload():
    full_mla_check(synth.MLA_WORKLOADS[synth.MLA_TINY])


# dtype, H, heads, batch, positions
SHAPES = [
    ("bf16", 2048, 16, 1, "fixed:300"),              # the DeepSeek-V2-Lite shape, short context
    ("f16", 1024, 8, 3, "list:0,57,1000"),           # position 0: only the new token
    ("bf16", 512, 8, 2, "list:31,32"),               # one head per warp; ragged 32-row tiles
    ("bf16", 1536, 16, 4, "list:600,5,129,64"),      # three W_o boxes per band, four rows
    ("f16", 4096, 8, 2, "list:700,701"),             # widest hidden
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}-H{s[1]}-h{s[2]}-B{s[3]}")
def test_scaled_shapes(shape):
    dt, H, nh, B, pos = shape
    s_max = max(int(v) for v in pos.split(":")[1].split(",")) + 3
    w = synth.custom_mla(name="mla", hidden=H, n_heads=nh, batch=B, s_max=s_max, dtype=dt,
                         positions=pos)
    full_mla_check(w, seed=7)


def test_deepseek_v2_lite_4k_full_size():
    """The 4096-position workload bench.py times, at full size, all outputs."""
    full_mla_check(synth.MLA_WORKLOADS[synth.MLA_4K], seed=0)


def test_deepseek_v2_lite_16k_full_size():
    """The 16384-position workload bench.py times, at full size."""
    full_mla_check(synth.MLA_WORKLOADS[synth.MLA_16K], seed=0)


def test_zero_output_projection_returns_hidden_bit_exact():
    for dt in ("bf16", "f16"):
        w = synth.custom_mla(name="mla0", hidden=1024, n_heads=16, batch=2, s_max=80, dtype=dt,
                             positions="list:79,3")
        t = synth.make_mla_layer(w, 3, device="cuda")
        t["w_o"].zero_()
        out, _, st = run_mla(w, t)
        assert st == binding.CF_OK
        assert torch.equal(out, t["hidden"]), dt


def test_out_of_range_position_flags_and_skips_the_row():
    w = synth.custom_mla(name="mla_bad", hidden=512, n_heads=8, batch=3, s_max=40,
                         positions="list:39,40,-1")
    t = synth.make_mla_layer(w, 4, device="cuda")
    blk = make_mla(w)
    out, lc, st = run_mla(w, t, blk)
    assert st == binding.CF_ERR_DEVICE_POS_RANGE
    assert blk.status() == binding.CF_OK  # the read cleared it
    assert torch.equal(out[1:], t["hidden"][1:])
    assert torch.equal(lc[1:], t["latent_cache"][1:])
    ref = oracle_mla(w, t, rows=[0])
    check(out[:1].double().cpu().numpy(), round_to(ref["out"], w.dtype), "good row")


def test_repeats_smaller_batches_and_graph_replay_leave_the_workspace_clean():
    w = synth.custom_mla(name="mla_rep", hidden=1024, n_heads=16, batch=4, s_max=200,
                         positions="list:199,3,77,150")
    t = synth.make_mla_layer(w, 5, device="cuda")
    blk = make_mla(w)
    first, _, st = run_mla(w, t, blk)
    assert st == binding.CF_OK
    check(first.double().cpu().numpy(), round_to(oracle_mla(w, t)["out"], w.dtype), "first call")
    for B in (4, 1, 3, 4):
        out, _, st = run_mla(w, t, blk, batch=B)
        assert st == binding.CF_OK
        assert torch.isnan(out[B:]).all()
        check(out[:B].double().cpu().numpy(), first[:B].double().cpu().numpy(), f"B={B}",
              mean_rel=1e-5)
    lc = t["latent_cache"].clone()
    out = torch.empty_like(t["hidden"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk(w.batch, *[t[k] for k in ARGS], lc, t["positions"], out, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert blk.status() == binding.CF_OK
    check(out.double().cpu().numpy(), first.double().cpu().numpy(), "graph", mean_rel=1e-5)


def test_back_to_back_launches_on_one_cache_agree():
    """Launches that follow one another with nothing in between (each may
    start while the previous one drains) and graph replays separated by
    host synchronizations, all on the cache the first launch appended to,
    give the first launch's output."""
    w = synth.custom_mla(name="mla_b2b", hidden=1024, n_heads=16, batch=4, s_max=200,
                         positions="list:199,3,77,150")
    t = synth.make_mla_layer(w, 5, device="cuda")
    blk = make_mla(w)
    first, lc, st = run_mla(w, t, blk)
    assert st == binding.CF_OK
    ref = first.double().cpu().numpy()
    outs = [torch.full_like(first, float("nan")) for _ in range(6)]
    for o in outs:
        blk(w.batch, *[t[k] for k in ARGS], lc, t["positions"], o)
    torch.cuda.synchronize()
    assert blk.status() == binding.CF_OK
    for i, o in enumerate(outs):
        check(o.double().cpu().numpy(), ref, f"launch {i}", mean_rel=1e-5)
    out = torch.full_like(first, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk(w.batch, *[t[k] for k in ARGS], lc, t["positions"], out, s)
    for i in range(4):
        g.replay()
        torch.cuda.synchronize()
        check(out.double().cpu().numpy(), ref, f"replay {i}", mean_rel=1e-5)
    assert blk.status() == binding.CF_OK


def test_layers_chained_on_one_handle_under_programmatic_dependent_launch():
    """Four layers back to back on one stream and one handle (each launch may
    start while the previous one drains; the grid barrier's words are read
    only after the dependency wait), each checked against the oracle fed that
    layer's GPU input."""
    w = synth.custom_mla(name="mla_chain", hidden=2048, n_heads=16, batch=2, s_max=160,
                         positions="list:159,40")
    ts = [synth.make_mla_layer(w, 20 + l, device="cuda") for l in range(4)]
    blk = make_mla(w)
    outs, caches = [], []
    x = ts[0]["hidden"]
    for t in ts:
        lc = t["latent_cache"].clone()
        out = torch.full_like(x, float("nan"))
        blk(w.batch, x, *[t[k] for k in ARGS[1:]], lc, t["positions"], out)
        outs.append(out)
        caches.append(lc)
        x = out
    torch.cuda.synchronize()
    assert blk.status() == binding.CF_OK
    for l, t in enumerate(ts):
        x_in = ts[0]["hidden"] if l == 0 else outs[l - 1]
        ref = oracle_mla(w, t, x=x_in)
        check(outs[l].double().cpu().numpy(), round_to(ref["out"], w.dtype), f"layer {l}")


def test_argument_errors():
    w = synth.custom_mla(name="mla_err", hidden=512, n_heads=8, batch=2, s_max=16,
                         positions="list:3,4")
    t = synth.make_mla_layer(w, 0, device="cuda")
    blk = make_mla(w)
    args = [t[k] for k in ARGS]
    lc = t["latent_cache"].clone()
    out = torch.empty_like(t["hidden"])
    f = binding.cf_mla_decode
    assert f(blk.handle, 0, *args, lc, t["positions"], out) == binding.CF_OK
    assert f(blk.handle, 3, *args, lc, t["positions"], out) == binding.CF_ERR_INVALID_ARG
    assert f(blk.handle, 2, *args, lc, t["positions"], t["hidden"]) == binding.CF_ERR_ALIAS
    assert f(blk.handle, 2, *args, lc, t["positions"], lc) == binding.CF_ERR_ALIAS
    bad = [t["hidden"].data_ptr() + 2] + args[1:]
    assert f(blk.handle, 2, *bad, lc, t["positions"], out) == binding.CF_ERR_INVALID_ARG
