"""The allocation-free entry point against the regular one.

cf_decode_attn_block_noalloc serves callers that cannot allocate device
memory (e.g. under a no-allocation graph-capture policy, or when another
allocator owns the device): it uses a fixed static device array as scratch
instead of a handle's workspace.  This test calls it through the C ABI twice
in a row on the same inputs and checks both outputs (and the appended cache
slot) against cf_decode_attn_block's, with the tolerance used by the parity
tests.  The file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from attention_block_gb300 import binding, synth
from parity_util import check, check_cache_untouched_except_slot

pytestmark = pytest.mark.gpu


def _workloads():
    return [synth.WORKLOADS[synth.LLAMA2_1K],
            synth.custom(name="gqa_small", hidden=1024, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         batch=3, s_max=300, dtype="bf16", positions="list:299,0,150")]


@pytest.mark.parametrize("w", _workloads(), ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point_twice(w):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    t = synth.make_layer(w, seed=11, device="cuda")
    cfg = binding.make_config(w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim, w.batch,
                              w.s_max, w.rope_theta, w.rms_eps, w.dtype)
    # regular entry point
    blk = binding.DecodeAttnBlock(hidden=w.hidden, n_q_heads=w.n_q_heads,
                                  n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                                  max_batch=w.batch, s_max=w.s_max, rope_theta=w.rope_theta,
                                  rms_eps=w.rms_eps, dtype=w.dtype)
    kc_r, vc_r = t["k_cache"].clone(), t["v_cache"].clone()
    out_r = torch.empty_like(t["hidden"])
    blk(w.batch, t["hidden"], t["ln_weight"], t["w_qkv"], t["w_o"], kc_r, vc_r, t["positions"],
        out_r)
    torch.cuda.synchronize()
    assert blk.status() == binding.CF_OK
    pos = t["positions"].tolist()
    for call in range(2):
        kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
        out = torch.full_like(t["hidden"], float("nan"))
        rc = binding.cf_decode_attn_block_noalloc(cfg, w.batch, t["hidden"], t["ln_weight"],
                                                  t["w_qkv"], t["w_o"], kc, vc, t["positions"],
                                                  out)
        assert rc == binding.CF_OK, binding.strerror(rc)
        torch.cuda.synchronize()
        check(out.double().cpu().numpy(), out_r.double().cpu().numpy(), f"out, call {call}")
        for b, p in enumerate(pos):
            check(kc[b, p].double().cpu().numpy(), kc_r[b, p].double().cpu().numpy(),
                  f"k slot, call {call}")
            check(vc[b, p].double().cpu().numpy(), vc_r[b, p].double().cpu().numpy(),
                  f"v slot, call {call}")
        check_cache_untouched_except_slot(t["k_cache"], kc, pos)
        check_cache_untouched_except_slot(t["v_cache"], vc, pos)
        assert binding.cf_noalloc_get_status() == binding.CF_OK
    blk.close()


def _regular(w, t, batch, positions):
    blk = binding.DecodeAttnBlock(hidden=w.hidden, n_q_heads=w.n_q_heads,
                                  n_kv_heads=w.n_kv_heads, head_dim=w.head_dim,
                                  max_batch=w.batch, s_max=w.s_max, rope_theta=w.rope_theta,
                                  rms_eps=w.rms_eps, dtype=w.dtype)
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    out = torch.empty_like(t["hidden"])
    blk(batch, t["hidden"], t["ln_weight"], t["w_qkv"], t["w_o"], kc, vc, positions, out)
    assert blk.status() == binding.CF_OK
    blk.close()
    return out, kc, vc


def test_noalloc_recovers_after_a_flagged_call_and_serves_a_smaller_batch():
    """The shared array keeps what earlier calls left.  A call with a position
    outside the cache (the kernel's own range check flags it and skips that
    row) is reported once by cf_noalloc_get_status; the valid calls that
    follow -- the full batch, then a smaller batch after the larger one --
    match the regular entry point and write nothing outside their new
    cache slots."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = _workloads()[1]
    t = synth.make_layer(w, seed=12, device="cuda")
    cfg = binding.make_config(w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim, w.batch,
                              w.s_max, w.rope_theta, w.rms_eps, w.dtype)
    assert binding.cf_noalloc_get_status() == binding.CF_OK

    def call(batch, positions):
        kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
        out = torch.full_like(t["hidden"], float("nan"))
        rc = binding.cf_decode_attn_block_noalloc(cfg, batch, t["hidden"], t["ln_weight"],
                                                  t["w_qkv"], t["w_o"], kc, vc, positions, out)
        assert rc == binding.CF_OK, binding.strerror(rc)
        torch.cuda.synchronize()
        return out, kc, vc

    bad = torch.tensor([w.s_max, 0, 150], dtype=torch.int32, device="cuda")
    out, kc, vc = call(w.batch, bad)
    assert binding.cf_noalloc_get_status() == binding.CF_ERR_DEVICE_POS_RANGE
    assert binding.cf_noalloc_get_status() == binding.CF_OK  # the read cleared it
    assert torch.equal(out[0], t["hidden"][0])  # the flagged row: out = hidden, cache untouched
    assert torch.equal(kc[0], t["k_cache"][0]) and torch.equal(vc[0], t["v_cache"][0])
    for batch in (w.batch, 2, 1):
        pos = t["positions"][:batch]
        out, kc, vc = call(batch, pos)
        assert binding.cf_noalloc_get_status() == binding.CF_OK
        out_r, kc_r, vc_r = _regular(w, t, batch, pos)
        check(out[:batch].double().cpu().numpy(), out_r[:batch].double().cpu().numpy(),
              f"out, batch {batch}")
        assert torch.isnan(out[batch:]).all()
        plist = pos.tolist()
        for b, p in enumerate(plist):
            check(kc[b, p].double().cpu().numpy(), kc_r[b, p].double().cpu().numpy(), "k slot")
            check(vc[b, p].double().cpu().numpy(), vc_r[b, p].double().cpu().numpy(), "v slot")
        check_cache_untouched_except_slot(t["k_cache"][:batch], kc[:batch], plist)
        check_cache_untouched_except_slot(t["v_cache"][:batch], vc[:batch], plist)
        assert torch.equal(kc[batch:], t["k_cache"][batch:])
        assert torch.equal(vc[batch:], t["v_cache"][batch:])


def test_noalloc_rejects_oversized_problem_without_launching():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cfg = binding.make_config(4096, 32, 32, 128, 256, 1025, dtype="f16")  # 256*4096 > 524288
    x = torch.zeros(16, device="cuda")
    rc = binding.cf_decode_attn_block_noalloc(cfg, 1, x, x, x, x, x, x, x, x)
    assert rc == binding.CF_ERR_INVALID_ARG
