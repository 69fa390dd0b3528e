"""GPU parity of the batched row-split kernel (4 to 64 batch rows per
cluster, tensor-core projections and attention) against the float64 oracle.

Every compiled (dtype, head_dim, group, batch tile, rows per block) instance
runs on a scaled shape with a ragged last batch tile and positions that hit
0, the last cache slot and the K/V tile edges; the two batched benchmark
workloads run at full size (sampled rows for the 64-row one) in every
instance that serves them, and with the sequence-split kernel forced for
comparison.  The degenerate cases (zero output projection, out-of-range
positions, batch below the handle's maximum, graph replay) are repeated for
this kernel because its row ownership and finalization differ.
"""
import numpy as np
import pytest
import torch

from attention_block_gb300 import binding, synth
from parity_util import check, full_check, make_block, round_to, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.lib()


def _positions(batch, S):
    """Mix of edge positions (0, 1, S-1, around 64/128-position tiles) and
    spread values, one per row."""
    edge = [0, S - 1, 1, 63, 64, 65, 127, 128, 129, S - 2]
    return [edge[i] if i < len(edge) and edge[i] < S else (i * 37 + 11) % S
            for i in range(batch)]


def _custom(dtype, H, nq, nkv, d, B, S):
    return synth.custom(name="batched", hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d,
                        batch=B, s_max=S, dtype=dtype,
                        positions="list:" + ",".join(str(p) for p in _positions(B, S)))


# (dtype, head_dim, group, batch tile, rows per block) of every instance, with
# a shape whose hidden size splits into 64-column bands over the cluster
INSTANCES = [
    ("f16", 64, 1, 64, 16),
    ("f16", 64, 1, 32, 8),
    ("f16", 64, 1, 16, 4),
    ("f16", 128, 1, 16, 4),
    ("f16", 128, 4, 16, 4),
    ("f16", 128, 4, 4, 1),
    ("bf16", 128, 4, 4, 1),
    ("bf16", 128, 4, 8, 2),
    ("bf16", 128, 4, 16, 4),
    ("bf16", 64, 1, 16, 4),
]


def _shape_for(dt, d, G, BT, RPC):
    N = BT // RPC
    H = max(512, 64 * N)
    nkv = 4 if G > 1 else 8
    B = BT + BT // 2 + 3  # two tiles, the second ragged
    return _custom(dt, H, nkv * G, nkv, d, B, 300)


@pytest.mark.parametrize("inst", INSTANCES, ids=lambda s: f"{s[0]}-d{s[1]}-G{s[2]}-BT{s[3]}-R{s[4]}")
def test_every_instance_scaled_shape(inst):
    dt, d, G, BT, RPC = inst
    w = _shape_for(*inst)
    blk = make_block(w, batch_tile=BT, rows_per_block=RPC)
    info = blk.launch_info()
    assert info["mode"] == 1 and info["batch_tile"] == BT and info["rows_per_block"] == RPC
    assert info["cluster_size"] == BT // RPC
    full_check(w, seed=11, batch_tile=BT, rows_per_block=RPC)


@pytest.mark.parametrize("inst,stages", [
    (("f16", 64, 1, 16, 4), 2), (("f16", 64, 1, 16, 4), 3),
    (("bf16", 128, 4, 4, 1), 2), (("bf16", 128, 4, 4, 1), 3),
    (("bf16", 128, 4, 16, 4), 3), (("f16", 64, 1, 64, 16), 3)],
    ids=lambda v: "-".join(map(str, v)) if isinstance(v, tuple) else f"stages{v}")
def test_ring_depths(inst, stages):
    # Ring slots and fill parities are advanced by counting in every loop
    # (projection, attention tiles, O projection, producer); a shallow ring
    # wraps many times per launch, so every slot reuses its barrier phases.
    dt, d, G, BT, RPC = inst
    w = _shape_for(*inst)
    blk = make_block(w, batch_tile=BT, rows_per_block=RPC, max_stages=stages)
    assert blk.launch_info()["stages"] == stages
    full_check(w, seed=17, batch_tile=BT, rows_per_block=RPC, max_stages=stages)


def test_tcgen05_ring_must_hold_a_k_slice():
    # The 16-row bf16 GQA instance stages each K slice of W_qkv as 3 ring
    # stages and only its MMA issuer waits for the second and third: a
    # 2-stage ring is refused rather than run.
    w = _shape_for("bf16", 128, 4, 16, 4)
    cfg = binding.make_config(w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim, w.batch, w.s_max,
                              w.rope_theta, w.rms_eps, w.dtype, batch_tile=16, rows_per_block=4,
                              max_stages=2)
    rc, h = binding.cf_create_rc(cfg)
    assert rc == binding.CF_ERR_UNSUPPORTED and not h


def test_default_picks_batched_kernel_for_batched_workloads():
    for name, bt in ((synth.SMALL_HEAD_B64, 64), (synth.LLAMA3_GQA, 4)):
        w = synth.WORKLOADS[name]
        info = make_block(w).launch_info()
        assert info["mode"] == 1 and info["batch_tile"] == bt, (name, info)
    # batch 1 and fp32 stay on the sequence-split kernel
    for name in (synth.LLAMA2_1K, synth.TINY):
        assert make_block(synth.WORKLOADS[name]).launch_info()["mode"] == 0


@pytest.mark.parametrize("bt,rpc", [(64, 16), (32, 8), (16, 4)])
def test_small_head_dim_batch64_every_batched_instance(bt, rpc):
    w = synth.WORKLOADS[synth.SMALL_HEAD_B64]
    t = synth.make_layer(w, 0, device="cuda")
    pos = t["positions"].cpu().numpy()
    rows = sorted({int(np.argmin(pos)), int(np.argmax(pos)), 0, 15, 16, 31, 33, 47, 62, 63})
    full_check(w, rows=rows, t=t, batch_tile=bt, rows_per_block=rpc)


@pytest.mark.parametrize("bt,rpc", [(4, 1), (8, 2), (16, 4)])
def test_llama3_gqa_layer_full_batched(bt, rpc):
    full_check(synth.WORKLOADS[synth.LLAMA3_GQA], batch_tile=bt, rows_per_block=rpc)


def test_batched_workloads_on_sequence_split_kernel():
    w = synth.WORKLOADS[synth.SMALL_HEAD_B64]
    t = synth.make_layer(w, 0, device="cuda")
    full_check(w, rows=[0, 21, 63], t=t, batch_tile=4)
    full_check(synth.WORKLOADS[synth.LLAMA3_GQA], batch_tile=2)


def test_batched_zero_output_projection_returns_hidden_bit_exact():
    for dt, G in (("f16", 1), ("bf16", 4)):
        w = _custom(dt, 1024, 8 * G, 8, 128, 20, 64)
        t = synth.make_layer(w, 1, device="cuda")
        t["w_o"].zero_()
        blk = make_block(w, batch_tile=16)
        assert blk.launch_info()["mode"] == 1
        out, _, _, _, st = run_gpu(w, t, block=blk)
        assert st == binding.CF_OK
        assert torch.equal(out, t["hidden"]), dt


def test_batched_out_of_range_positions_flag_and_skip_rows():
    B, S = 18, 70
    pos = [(5 * i + 3) % S for i in range(B)]
    bad = [2, 9, 17]
    pos[2], pos[9], pos[17] = S, -1, S + 100
    w = synth.custom(name="batched_oob", hidden=512, n_q_heads=8, n_kv_heads=8, head_dim=64,
                     batch=B, s_max=S, dtype="f16",
                     positions="list:" + ",".join(str(p) for p in pos))
    t = synth.make_layer(w, 2, device="cuda")
    blk = make_block(w, batch_tile=16, rows_per_block=4)
    assert blk.launch_info()["mode"] == 1
    out, kc, vc, _, st = run_gpu(w, t, block=blk)
    assert st == binding.CF_ERR_DEVICE_POS_RANGE
    assert binding.cf_get_status(blk.handle) == binding.CF_OK
    for b in bad:
        assert torch.equal(out[b], t["hidden"][b])
        assert torch.equal(kc[b], t["k_cache"][b]) and torch.equal(vc[b], t["v_cache"][b])
    good = [b for b in range(B) if b not in bad]
    ref = run_oracle(w, t, rows=good)
    check(out[good].double().cpu().numpy(), round_to(ref["out"], w.dtype), "good rows")


def test_batched_batch_below_max_batch():
    w = _custom("f16", 512, 8, 8, 64, 21, 90)
    blk = binding.DecodeAttnBlock(hidden=512, n_q_heads=8, n_kv_heads=8, head_dim=64,
                                  max_batch=64, s_max=90, dtype="f16")
    assert blk.launch_info()["mode"] == 1
    t = synth.make_layer(w, 7, device="cuda")
    out, kc, vc, _, st = run_gpu(w, t, block=blk)
    assert st == binding.CF_OK
    ref = run_oracle(w, t)
    check(out.double().cpu().numpy(), round_to(ref["out"], w.dtype), "out")


def test_batched_graph_replay_matches_eager():
    w = _custom("bf16", 1024, 16, 4, 128, 16, 200)
    t = synth.make_layer(w, 4, device="cuda")
    blk = make_block(w)
    assert blk.launch_info()["mode"] == 1
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    args = (t["hidden"], t["ln_weight"], t["w_qkv"], t["w_o"], kc, vc, t["positions"])
    out_e = torch.empty_like(t["hidden"])
    blk(w.batch, *args, out_e)
    torch.cuda.synchronize()
    out_g = torch.empty_like(t["hidden"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        blk(w.batch, *args, out_g)
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        check(out_g.double().cpu().numpy(), out_e.double().cpu().numpy(), "graph vs eager",
              mean_rel=1e-4)
    assert binding.cf_get_status(blk.handle) == binding.CF_OK


def test_runtime_choice_per_batch_matches_oracle_and_changes_kernel():
    """A handle sized for 64 rows plans for batch caps 1, 2, 4, ... as well and
    gives each call the smallest plan that holds its batch: a one-row call runs
    the sequence-split kernel, a 64-row call the batched one; every call
    matches the oracle on its rows.  adaptive = -1 keeps the single plan."""
    w = synth.WORKLOADS[synth.SMALL_HEAD_B64]
    t = synth.make_layer(w, 7, device="cuda")
    blk = make_block(w)
    assert blk.launch_info(1)["mode"] == 0
    assert blk.launch_info(64)["mode"] == 1 and blk.launch_info(64)["batch_tile"] == 64
    assert blk.launch_info() == blk.launch_info(64)
    fixed = make_block(w, adaptive=-1)
    assert fixed.launch_info(1) == fixed.launch_info(64)
    for b in (1, 5, 16, 64):
        out = torch.full_like(t["hidden"], float("nan"))
        kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
        blk(b, t["hidden"], t["ln_weight"], t["w_qkv"], t["w_o"], kc, vc, t["positions"], out)
        assert blk.status() == binding.CF_OK
        rows = sorted({0, b // 2, b - 1})
        ref = run_oracle(w, t, rows=rows)
        check(out[rows].double().cpu().numpy(), round_to(ref["out"], w.dtype), f"batch {b}")
        if b < w.batch:
            assert torch.isnan(out[b:]).all()
