"""GPU parity of the second RMSNorm + gated FFN + residual (cf_ffn_forward)
against the float64 oracle, alone and after the attention block (one whole
decoder layer on one stream, the FFN launched as a programmatic dependent of
the attention kernel).
"""
import numpy as np
import pytest
import torch

import oracle
from attention_block_gb300 import binding, synth
from parity_util import check, make_block, round_to, run_gpu, run_oracle, storage_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.lib()


def make_ffn_block(w, **kw):
    return binding.FfnBlock(w.hidden, w.intermediate, w.batch, w.rms_eps, w.dtype, **kw)


def run_ffn(w, t, blk=None, batch=None, out=None):
    blk = blk if blk is not None else make_ffn_block(w)
    B = w.batch if batch is None else batch
    if out is None:
        out = torch.full_like(t["hidden"], float("nan"))
    blk(B, t["hidden"], t["ln_weight"], t["w_gate"], t["w_up"], t["w_down"], out)
    st = blk.status()
    return out, st


def oracle_ffn(w, t, rows=None):
    f = {k: synth.to_f64(t[k]) for k in ("hidden", "ln_weight", "w_gate", "w_up", "w_down")}
    return oracle.ffn(f["hidden"], f["ln_weight"], f["w_gate"], f["w_up"], f["w_down"],
                      w.rms_eps, rows)


def full_ffn_check(w, seed=0, rows=None, **kw):
    t = synth.make_ffn(w, seed, device="cuda")
    out, st = run_ffn(w, t, make_ffn_block(w, **kw))
    assert st == binding.CF_OK
    rows = list(range(w.batch)) if rows is None else rows
    ref = oracle_ffn(w, t, rows)
    got = out[rows].double().cpu().numpy()
    want = round_to(ref["out"], w.dtype)
    check(got, want, "out")
    # the FFN's own contribution, unmasked by the residual (both sides carry
    # the output's rounding to the storage type)
    x = synth.to_f64(t["hidden"][rows])
    check(got - x, want - x, "out - hidden", floor=storage_ulp(want, w.dtype))
    return out, ref


@pytest.mark.parametrize("name", sorted(synth.FFN_WORKLOADS))
def test_ffn_workloads(name):
    full_ffn_check(synth.FFN_WORKLOADS[name])


SHAPES = [
    # dtype, H, I, B, stage_bytes
    ("f16", 1024, 300, 1, 0),
    ("bf16", 2048, 5632, 2, 0),
    ("f32", 512, 152, 2, 0),       # one unit per block on a 152-SM part
    ("f16", 4096, 100, 2, 0),      # fewer units than SMs
    ("bf16", 64, 1000, 1, 0),      # H below one 4-element chunk per thread
    ("f16", 4096, 11008, 2, 8192),  # one weight row per stage
    ("bf16", 3072, 777, 1, 40000),  # stage of 6 rows, ragged last group
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}-H{s[1]}-I{s[2]}-B{s[3]}-S{s[4]}")
def test_scaled_shapes(shape):
    dt, H, I, B, sb = shape
    w = synth.custom_ffn(name="ffn", hidden=H, intermediate=I, batch=B, dtype=dt)
    full_ffn_check(w, seed=3, stage_bytes=sb)


# batched decode on the tensor-core pair: dtype, H, I, max_batch, batch
TC_SHAPES = [
    ("f16", 2048, 5632, 64, 64),    # the 64-row layer's FFN
    ("bf16", 4096, 14336, 16, 16),  # the Llama-3 layer's FFN at 16 rows
    ("f16", 1024, 777, 16, 3),      # 3 rows (smallest batch of the pair), ragged I
    ("bf16", 512, 152, 32, 21),     # one unit per block, 21 of 32 rows
    ("f16", 384, 4000, 64, 40),     # H of three column tiles, UB 32
    ("bf16", 4096, 100, 16, 9),     # fewer units than SMs, more columns than units
]


@pytest.mark.parametrize("shape", TC_SHAPES,
                         ids=lambda s: f"{s[0]}-H{s[1]}-I{s[2]}-M{s[3]}-B{s[4]}")
def test_tensor_core_pair_scaled_shapes(shape):
    dt, H, I, M, B = shape
    w = synth.custom_ffn(name="ffn_tc", hidden=H, intermediate=I, batch=B, dtype=dt)
    t = synth.make_ffn(w, 11, device="cuda")
    blk = binding.FfnBlock(H, I, M, w.rms_eps, dt)
    assert blk.kernels(B)["kernels"] == 2 and blk.kernels(2)["kernels"] == 1
    out, st = run_ffn(w, t, blk)
    assert st == binding.CF_OK
    rows = list(range(B))  # every row
    ref = oracle_ffn(w, t, rows)
    got = out[rows].double().cpu().numpy()
    want = round_to(ref["out"], w.dtype)
    check(got, want, "out")
    x = synth.to_f64(t["hidden"][rows])
    check(got - x, want - x, "out - hidden", floor=storage_ulp(want, w.dtype))
    # the intermediate activations the pair hands from one kernel to the next
    check(blk.debug_a(B), ref["a"], "a = silu(gate) * up")


def test_tensor_core_pair_small_batches_and_repeats_on_one_handle():
    """One handle of max_batch 64 serves 1, 2 (the CUDA-core kernel), 3, 17
    and 64 rows (the pair), in any order, leaving its workspace clean."""
    w64 = synth.FFN_WORKLOADS[synth.B64_FFN]
    t = synth.make_ffn(w64, 12, device="cuda")
    blk = make_ffn_block(w64)
    firsts = {}
    for B in (64, 3, 1, 17, 2, 64, 3):
        out = torch.full_like(t["hidden"], float("nan"))
        blk(B, t["hidden"], t["ln_weight"], t["w_gate"], t["w_up"], t["w_down"], out)
        assert blk.status() == binding.CF_OK
        assert torch.isnan(out[B:]).all()
        if B in firsts:
            # The row sums of squares meet by fp32 atomics in any order, so a
            # repeat may round a few single-fp16 activations one ulp apart,
            # which moves outputs by about one fp16 ulp: bound the mean
            # relative difference at 1e-4 (stale workspace state would show
            # as errors of the order of the values themselves).
            check(out[:B].double().cpu().numpy(), firsts[B], f"repeat B={B}", mean_rel=1e-4)
            continue
        firsts[B] = out[:B].double().cpu().numpy()
        rows = sorted({0, B - 1})
        ref = oracle_ffn(w64, t, rows)
        check(out[rows].double().cpu().numpy(), round_to(ref["out"], w64.dtype), f"out B={B}")


def test_tensor_core_pair_zero_down_projection_returns_hidden_bit_exact():
    w = synth.custom_ffn(name="ffn_tc0", hidden=1024, intermediate=3000, batch=32, dtype="bf16")
    t = synth.make_ffn(w, 13, device="cuda")
    t["w_down"].zero_()
    out, st = run_ffn(w, t, make_ffn_block(w))
    assert st == binding.CF_OK and torch.equal(out, t["hidden"])


def test_tensor_core_pair_graph_replay():
    w = synth.FFN_WORKLOADS[synth.LLAMA3_FFN_B16]
    t = synth.make_ffn(w, 14, device="cuda")
    blk = make_ffn_block(w)
    first, st = run_ffn(w, t, blk)
    assert st == binding.CF_OK
    out = torch.empty_like(t["hidden"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk(w.batch, t["hidden"], t["ln_weight"], t["w_gate"], t["w_up"], t["w_down"], out, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert blk.status() == binding.CF_OK
    check(out.double().cpu().numpy(), first.double().cpu().numpy(), "graph", mean_rel=1e-5)


def test_zero_down_projection_returns_hidden_bit_exact_and_batch_below_max():
    w = synth.custom_ffn(name="ffn0", hidden=2048, intermediate=3000, batch=2, dtype="bf16")
    t = synth.make_ffn(w, 1, device="cuda")
    t["w_down"].zero_()
    blk = make_ffn_block(w)
    out, st = run_ffn(w, t, blk)
    assert st == binding.CF_OK and torch.equal(out, t["hidden"])
    out1 = torch.full_like(t["hidden"], float("nan"))
    out1, st = run_ffn(w, t, blk, batch=1, out=out1)
    assert st == binding.CF_OK and torch.equal(out1[0], t["hidden"][0])
    assert torch.isnan(out1[1]).all()


def test_repeat_and_graph_replay_leave_the_workspace_clean():
    w = synth.FFN_WORKLOADS[synth.LLAMA2_FFN]
    t = synth.make_ffn(w, 2, device="cuda")
    blk = make_ffn_block(w)
    first, _ = run_ffn(w, t, blk)
    second, _ = run_ffn(w, t, blk)
    check(second.double().cpu().numpy(), first.double().cpu().numpy(), "repeat", mean_rel=1e-5)
    out = torch.empty_like(t["hidden"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk(w.batch, t["hidden"], t["ln_weight"], t["w_gate"], t["w_up"], t["w_down"], out, s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert blk.status() == binding.CF_OK
    check(out.double().cpu().numpy(), first.double().cpu().numpy(), "graph", mean_rel=1e-5)


def test_argument_errors():
    w = synth.custom_ffn(name="ffn_err", hidden=256, intermediate=64, batch=2, dtype="f16")
    t = synth.make_ffn(w, 0, device="cuda")
    blk = make_ffn_block(w)
    args = [t["hidden"], t["ln_weight"], t["w_gate"], t["w_up"], t["w_down"]]
    out = torch.empty_like(t["hidden"])
    assert binding.cf_ffn_forward(blk.handle, 0, *args, out) == binding.CF_OK
    assert binding.cf_ffn_forward(blk.handle, 3, *args, out) == binding.CF_ERR_INVALID_ARG
    assert binding.cf_ffn_forward(blk.handle, 2, *args, t["hidden"]) == binding.CF_ERR_ALIAS
    assert binding.cf_ffn_forward(blk.handle, 2, *args, t["w_up"]) == binding.CF_ERR_ALIAS
    bad = [t["hidden"].data_ptr() + 2] + args[1:]
    assert binding.cf_ffn_forward(blk.handle, 2, *bad, out) == binding.CF_ERR_INVALID_ARG
    for cfg in (dict(hidden=4100), dict(hidden=8192), dict(max_batch=65), dict(intermediate=0),
                dict(max_batch=3, dtype=binding.CF_F32), dict(max_batch=3, hidden=320)):
        base = dict(hidden=256, intermediate=64, max_batch=1, rms_eps=1e-6, dtype=binding.CF_F16,
                    stage_bytes=0)
        base.update(cfg)
        c = binding.CfFfnConfig(base["hidden"], base["intermediate"], base["max_batch"],
                                base["rms_eps"], base["dtype"], base["stage_bytes"])
        h = binding._vp()
        rc = binding.lib().cf_ffn_create(c, binding.ctypes.byref(h))
        assert rc in (binding.CF_ERR_INVALID_ARG, binding.CF_ERR_UNSUPPORTED), cfg
        assert not h.value


@pytest.mark.parametrize("B", [1, 2])
def test_whole_decoder_layer_attention_then_ffn(B):
    """One decoder layer of the Llama-2-7B shape on one stream: the attention
    block's output feeds the FFN (launched as its programmatic dependent);
    the oracle runs the same two steps in float64 from the same inputs."""
    w = synth.custom(name="layer", hidden=4096, n_q_heads=32, n_kv_heads=32, head_dim=128,
                     batch=B, s_max=1025, dtype="f16", positions="fixed:1024")
    wf = synth.custom_ffn(name="layer_ffn", hidden=4096, intermediate=11008, batch=B,
                          dtype="f16")
    t = synth.make_layer(w, 5, device="cuda")
    tf = synth.make_ffn(wf, 6, device="cuda")
    attn = make_block(w)
    ffn = make_ffn_block(wf)
    h = torch.empty_like(t["hidden"])
    out = torch.empty_like(t["hidden"])
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    attn(B, t["hidden"], t["ln_weight"], t["w_qkv"], t["w_o"], kc, vc, t["positions"], h)
    ffn(B, h, tf["ln_weight"], tf["w_gate"], tf["w_up"], tf["w_down"], out)
    torch.cuda.synchronize()
    assert attn.status() == binding.CF_OK and ffn.status() == binding.CF_OK
    ref_attn = run_oracle(w, t)
    ref = oracle.ffn(ref_attn["out"], synth.to_f64(tf["ln_weight"]), synth.to_f64(tf["w_gate"]),
                     synth.to_f64(tf["w_up"]), synth.to_f64(tf["w_down"]), wf.rms_eps)
    check(out.double().cpu().numpy(), round_to(ref["out"], "f16"), "layer out")
    # and the FFN on exactly the GPU's layer-norm input (no compounding)
    ref_h = oracle.ffn(synth.to_f64(h), synth.to_f64(tf["ln_weight"]),
                       synth.to_f64(tf["w_gate"]), synth.to_f64(tf["w_up"]),
                       synth.to_f64(tf["w_down"]), wf.rms_eps)
    check(out.double().cpu().numpy(), round_to(ref_h["out"], "f16"), "ffn on the GPU's h")


# Decoder layers chained through ONE attention handle and ONE FFN handle:
# dtype, H, nq, nkv, d, position, I, batch
CHAIN_SHAPES = [
    # fewer FFN units than SMs: the gate/up grid leaves SMs free, so the next
    # layer's kernels can become resident while this layer's FFN still runs
    ("bf16", 4096, 32, 8, 128, 200, 100, 9),
    # the Llama-3 layer's FFN at 16 rows (one gate/up block per SM)
    ("bf16", 4096, 32, 8, 128, 256, 14336, 16),
]


@pytest.mark.parametrize("shape", CHAIN_SHAPES,
                         ids=lambda s: f"{s[0]}-H{s[1]}-I{s[6]}-B{s[7]}")
def test_decoder_layers_chained_under_programmatic_dependent_launch(shape):
    """Three decoder layers back to back on one stream, each the attention
    block then the FFN, with no host synchronization between launches and
    programmatic dependent launch on (the default): a kernel may become
    resident while earlier ones still run, including the previous layer's
    FFN with its grid barrier.  Every layer's attention output and FFN
    output is checked, all rows, against the oracle fed that layer's actual
    GPU input, so errors do not compound."""
    dt, H, nq, nkv, d, pos, I, B = shape
    layers = 3
    w = synth.custom(name="chain", hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, batch=B,
                     s_max=pos + 1, dtype=dt, rope_theta=5e5, positions=f"fixed:{pos}")
    wf = synth.custom_ffn(name="chain_ffn", hidden=H, intermediate=I, batch=B, dtype=dt)
    ts = [synth.make_layer(w, 30 + l, device="cuda") for l in range(layers)]
    tfs = [synth.make_ffn(wf, 60 + l, device="cuda") for l in range(layers)]
    attn = make_block(w)
    ffn = make_ffn_block(wf)
    assert ffn.kernels(B)["kernels"] == 2
    mids = [torch.full_like(ts[0]["hidden"], float("nan")) for _ in range(layers)]
    outs = [torch.full_like(ts[0]["hidden"], float("nan")) for _ in range(layers)]
    caches = [(t["k_cache"].clone(), t["v_cache"].clone()) for t in ts]
    x = ts[0]["hidden"]
    for l in range(layers):
        t, tf = ts[l], tfs[l]
        attn(B, x, t["ln_weight"], t["w_qkv"], t["w_o"], caches[l][0], caches[l][1],
             t["positions"], mids[l])
        ffn(B, mids[l], tf["ln_weight"], tf["w_gate"], tf["w_up"], tf["w_down"], outs[l])
        x = outs[l]
    torch.cuda.synchronize()
    assert attn.status() == binding.CF_OK
    assert ffn.status() == binding.CF_OK
    for l in range(layers):
        t, tf = ts[l], tfs[l]
        x_in = ts[0]["hidden"] if l == 0 else outs[l - 1]
        ref_a = run_oracle(w, t, hidden=x_in)
        check(mids[l].double().cpu().numpy(), round_to(ref_a["out"], dt), f"layer {l} attention")
        ref_f = oracle.ffn(synth.to_f64(mids[l]), synth.to_f64(tf["ln_weight"]),
                           synth.to_f64(tf["w_gate"]), synth.to_f64(tf["w_up"]),
                           synth.to_f64(tf["w_down"]), wf.rms_eps)
        got = outs[l].double().cpu().numpy()
        check(got, round_to(ref_f["out"], dt), f"layer {l} FFN")
        h = synth.to_f64(mids[l])
        want = round_to(ref_f["out"], dt)
        check(got - h, want - h, f"layer {l} FFN - its input", floor=storage_ulp(want, dt))
