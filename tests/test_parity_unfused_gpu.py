"""GPU parity of the three-kernel (unfused) decode step -- the fusion
baseline, cf_decode_attn_block_unfused -- against the float64 oracle, and its
agreement with the fused kernel on the same inputs.
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


@pytest.mark.parametrize("name", [synth.TINY, synth.LLAMA2_1K, synth.LLAMA3_GQA])
def test_benchmark_workloads(name):
    full_check(synth.WORKLOADS[name], debug=False, unfused=True)


def test_small_head_dim_batch64_sampled_rows():
    w = synth.WORKLOADS[synth.SMALL_HEAD_B64]
    t = synth.make_layer(w, 0, device="cuda")
    pos = t["positions"].cpu().numpy()
    rows = sorted({int(np.argmin(pos)), int(np.argmax(pos)), 0, 7, 8, 33, 63})
    full_check(w, rows=rows, t=t, debug=False, unfused=True)


def test_long_context_layer():
    w = synth.custom(name="long", hidden=4096, n_q_heads=32, n_kv_heads=32, head_dim=128, batch=1,
                     s_max=16385, dtype="f16", positions="fixed:16384")
    full_check(w, debug=False, unfused=True)


SHAPES = [
    # dtype, H, nq, nkv, d, batch, S, positions
    ("f32", 512, 8, 2, 128, 3, 200, [0, 77, 199]),
    ("f16", 1024, 8, 8, 64, 11, 257, [256, 0, 31, 33, 129, 1, 2, 3, 64, 65, 200]),
    ("bf16", 1024, 16, 4, 128, 9, 300, [299, 128, 127, 0, 200, 1, 64, 65, 298]),
    ("bf16", 512, 4, 4, 64, 1, 70, [33]),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}-H{s[1]}-{s[2]}x{s[3]}-d{s[4]}-B{s[5]}")
def test_scaled_shapes(shape):
    dt, H, nq, nkv, d, B, S, pos = shape
    w = synth.custom(name="uf", hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, batch=B,
                     s_max=S, dtype=dt, positions="list:" + ",".join(str(p) for p in pos))
    full_check(w, seed=5, debug=False, unfused=True)


def test_agrees_with_fused_and_repeats():
    w = synth.WORKLOADS[synth.LLAMA3_GQA]
    t = synth.make_layer(w, 3, device="cuda")
    blk = make_block(w)
    outs = []
    for unfused in (False, True, True):
        out, _, _, _, st = run_gpu(w, t, block=blk, unfused=unfused)
        assert st == binding.CF_OK
        outs.append(out.double().cpu().numpy())
    check(outs[1], outs[0], "unfused vs fused", mean_rel=1e-4)
    check(outs[2], outs[1], "unfused twice (workspace left clean)", mean_rel=1e-5)


def test_zero_output_projection_and_out_of_range_rows():
    pos = [5, 40, -1, 3]
    w = synth.custom(name="uf_oob", hidden=512, n_q_heads=8, n_kv_heads=8, head_dim=64, batch=4,
                     s_max=40, dtype="f16", positions="list:" + ",".join(str(p) for p in pos))
    t = synth.make_layer(w, 2, device="cuda")
    blk = make_block(w)
    out, kc, vc, _, st = run_gpu(w, t, block=blk, unfused=True)
    assert st == binding.CF_ERR_DEVICE_POS_RANGE
    assert binding.cf_get_status(blk.handle) == binding.CF_OK
    for b in (1, 2):
        assert torch.equal(out[b], t["hidden"][b])
        assert torch.equal(kc[b], t["k_cache"][b]) and torch.equal(vc[b], t["v_cache"][b])
    ref = run_oracle(w, t, rows=[0, 3])
    check(out[[0, 3]].double().cpu().numpy(), round_to(ref["out"], w.dtype), "good rows")
    t["w_o"].zero_()
    out, _, _, _, st = run_gpu(w, t, block=blk, unfused=True)
    assert torch.equal(out, t["hidden"])
