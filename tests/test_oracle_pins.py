"""Pins of the float64 oracle to facts fixed by the pages and by mathematics.

Nothing here compares the oracle with a retyped copy of its own formula: each
test uses a closed form, a hand-worked value, an invariant, a special case
that reduces to a library routine (numpy), or brute force on a tiny input.
Each is chosen so that a plausible slip in the oracle (eps outside the sqrt,
a dropped ln_weight, a transposed weight, interleaved instead of rotate-half
RoPE, a wrong frequency exponent or sign, a missing 1/sqrt(d), a wrong GQA
grouping, an off-by-one in the attended positions, a wrong head order in the
output projection, a dropped residual) fails at least one of them.

Pages: [CF] "ClusterFusion框架深度解析" (devpress.csdn.net);
[LNA] "大模型推理中的算子融合优化：LayerNorm + Attention" (asdsk.com).
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- RMSNorm --
def test_rmsnorm_constant_vector_closed_form():
    # [LNA §三 stage 1]: x = c*1 gives n_i = g_i * c / sqrt(c^2 + eps).  A large
    # eps separates "inside the sqrt" from "added to the rms".
    H, c, eps = 8, -1.5, 0.25
    g = RNG.normal(size=H)
    n = oracle.rmsnorm(np.full(H, c), g, eps)
    np.testing.assert_allclose(n, g * c / math.sqrt(c * c + eps), rtol=1e-14)


def test_rmsnorm_hand_example():
    # x = (3, 4): mean square = 12.5 (mean over H = 2, not the sum 25).
    n = oracle.rmsnorm([3.0, 4.0], [1.0, 2.0], 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(n, [3.0 / r, 8.0 / r], rtol=1e-15)


def test_rmsnorm_scale_invariance():
    x = RNG.normal(size=64)
    g = RNG.normal(size=64)
    np.testing.assert_allclose(oracle.rmsnorm(7.0 * x, g, 0.0),
                               oracle.rmsnorm(x, g, 0.0), rtol=1e-13)


# ----------------------------------------------------------------- matvec --
def test_matvec_matches_numpy_on_nonsquare():
    # x . W with W [K, N] row-major; K != N so a transposed read cannot pass.
    x = RNG.normal(size=7)
    W = RNG.normal(size=(7, 5))
    np.testing.assert_allclose(oracle.matvec(x, W), x @ W, rtol=1e-13, atol=1e-14)


def test_matvec_brute_force_integers():
    x = np.arange(1, 4, dtype=np.float64)             # [1,2,3]
    W = np.arange(6, dtype=np.float64).reshape(3, 2)  # [[0,1],[2,3],[4,5]]
    # y_0 = 1*0 + 2*2 + 3*4 = 16; y_1 = 1*1 + 2*3 + 3*5 = 22.
    np.testing.assert_array_equal(oracle.matvec(x, W), [16.0, 22.0])


# ------------------------------------------------------------------- RoPE --
def test_rope_position_zero_is_identity():
    u = RNG.normal(size=128)
    np.testing.assert_array_equal(oracle.rope(u, 0, 1e4), u)


def test_rope_d2_direction():
    # d = 2: one pair (0, 1), frequency theta^0 = 1, angle = pos.
    np.testing.assert_allclose(oracle.rope([1.0, 0.0], 1, 1e4),
                               [math.cos(1.0), math.sin(1.0)], rtol=1e-15)
    np.testing.assert_allclose(oracle.rope([0.0, 1.0], 1, 1e4),
                               [-math.sin(1.0), math.cos(1.0)], rtol=1e-15)


def test_rope_rotate_half_pairing_and_frequency():
    # d = 4: pairs (0,2) and (1,3); pair 1 turns at theta^(-2/4) = 0.01 rad per
    # position, so pos = 100 turns it by exactly 1 rad.  Interleaved pairing
    # would move e_1 into index 0; theta^(-i/d) would turn it by 10 rad.
    u = oracle.rope([0.0, 1.0, 0.0, 0.0], 100, 1e4)
    np.testing.assert_allclose(u, [0.0, math.cos(1.0), 0.0, math.sin(1.0)],
                               atol=1e-13)
    u = oracle.rope([1.0, 0.0, 0.0, 0.0], 100, 1e4)
    np.testing.assert_allclose(u, [math.cos(100.0), 0.0, math.sin(100.0), 0.0],
                               atol=1e-13)


def test_rope_preserves_pair_norms():
    d = 64
    u = RNG.normal(size=d)
    r = oracle.rope(u, 777, 5e5)
    h = d // 2
    np.testing.assert_allclose(r[:h] ** 2 + r[h:] ** 2, u[:h] ** 2 + u[h:] ** 2,
                               rtol=1e-12)


def test_rope_relative_position_property():
    d = 128
    q, k = RNG.normal(size=d), RNG.normal(size=d)
    a = oracle.rope(q, 300, 1e4) @ oracle.rope(k, 120, 1e4)
    b = oracle.rope(q, 1300, 1e4) @ oracle.rope(k, 1120, 1e4)
    assert abs(a - b) < 1e-10 * max(1.0, abs(a))


# -------------------------------------------------------------- attention --
def test_attention_single_token_returns_its_value():
    d = 64
    q, k, v = RNG.normal(size=d), RNG.normal(size=(1, d)), RNG.normal(size=(1, d))
    o, w = oracle.attention(q, k, v)
    np.testing.assert_allclose(o, v[0], rtol=1e-15)
    np.testing.assert_array_equal(w, [1.0])


def test_attention_identical_keys_average_values():
    d, n = 32, 17
    key = RNG.normal(size=d)
    K = np.tile(key, (n, 1))
    V = RNG.normal(size=(n, d))
    o, w = oracle.attention(RNG.normal(size=d), K, V)
    np.testing.assert_allclose(w, np.full(n, 1.0 / n), rtol=1e-14)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_two_key_hand_example_fixes_scale():
    # d = 4, q = (1,1,1,1), k_0 = 0, k_1 = (1,1,1,1): s_0 = 0, s_1 = 4/sqrt(4) = 2.
    # v_0 = 0, v_1 = 1 -> o = e^2 / (1 + e^2) in every coordinate.
    q = np.ones(4)
    K = np.array([np.zeros(4), np.ones(4)])
    V = np.array([np.zeros(4), np.ones(4)])
    o, w = oracle.attention(q, K, V)
    w1 = math.exp(2.0) / (1.0 + math.exp(2.0))
    np.testing.assert_allclose(w, [1.0 - w1, w1], rtol=1e-15)
    np.testing.assert_allclose(o, np.full(4, w1), rtol=1e-15)


def test_attention_weights_sum_to_one_and_follow_score_order():
    d, n = 64, 200
    q = RNG.normal(size=d)
    K = RNG.normal(size=(n, d))
    o, w = oracle.attention(q, K, RNG.normal(size=(n, d)))
    assert abs(w.sum() - 1.0) < 1e-13
    assert np.all(w > 0)
    np.testing.assert_array_equal(np.argsort(w, kind="stable"),
                                  np.argsort(K @ q, kind="stable"))


@pytest.mark.parametrize("ends", [
    [5, 200], [1, 2, 3, 200], [0, 0, 100, 100, 200], [64, 128, 192, 200],
    list(range(1, 201))])
def test_split_kv_equals_two_pass(ends):
    d, n = 64, 200
    q = RNG.normal(size=d) * 3.0
    K = RNG.normal(size=(n, d))
    V = RNG.normal(size=(n, d))
    o, _ = oracle.attention(q, K, V)
    np.testing.assert_allclose(oracle.attention_split(q, K, V, ends), o,
                               rtol=1e-12, atol=1e-13)


# ----------------------------------------------------- whole decode block --
def _tiny(nq=4, nkv=4, d=16, H=48, S=9, theta=1e4, eps=1e-6):
    return dict(hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=d, s_max=S,
                rope_theta=theta, rms_eps=eps)


def _draw(cfg, rng):
    H, nq, nkv, d, S = (cfg[k] for k in ("hidden", "n_q_heads", "n_kv_heads",
                                         "head_dim", "s_max"))
    C = (nq + 2 * nkv) * d
    return dict(x=rng.normal(size=H), g=1 + 0.1 * rng.normal(size=H),
                wqkv=0.2 * rng.normal(size=(H, C)), wo=0.2 * rng.normal(size=(nq * d, H)),
                kc=rng.normal(size=(S, nkv, d)), vc=rng.normal(size=(S, nkv, d)))


def test_decode_zero_output_projection_returns_residual_exactly():
    cfg = _tiny()
    t = _draw(cfg, np.random.default_rng(0))
    t["wo"][:] = 0.0
    r = oracle.decode_row(cfg, t["x"], t["g"], t["wqkv"], t["wo"], t["kc"], t["vc"], 5)
    np.testing.assert_array_equal(r["out"], t["x"])


@pytest.mark.parametrize("nq,nkv", [(4, 4), (4, 2), (6, 2)])
def test_decode_zero_query_gives_uniform_attention(nq, nkv):
    # W_q = 0 makes every score 0, so o_h is the plain mean of the values at
    # positions 0..pos (the appended token included) of KV head h // (nq/nkv).
    # Expected values are built from numpy matmuls and means only.
    cfg = _tiny(nq=nq, nkv=nkv)
    H, d, pos = cfg["hidden"], cfg["head_dim"], 6
    t = _draw(cfg, np.random.default_rng(1))
    t["wqkv"][:, : nq * d] = 0.0
    kc0, vc0 = t["kc"].copy(), t["vc"].copy()
    r = oracle.decode_row(cfg, t["x"], t["g"], t["wqkv"], t["wo"], t["kc"], t["vc"], pos)
    n = oracle.rmsnorm(t["x"], t["g"], cfg["rms_eps"])
    y = n @ t["wqkv"]
    v_new = y[(nq + nkv) * d:].reshape(nkv, d)
    k_new = y[nq * d:(nq + nkv) * d].reshape(nkv, d)
    vals = vc0.copy()
    vals[pos] = v_new
    group = nq // nkv
    o_exp = np.concatenate([vals[: pos + 1, h // group].mean(axis=0) for h in range(nq)])
    np.testing.assert_allclose(r["o"], o_exp, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["proj"], o_exp @ t["wo"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(r["out"], t["x"] + o_exp @ t["wo"], rtol=1e-11, atol=1e-12)
    # Only slot pos changed; it holds v_new and RoPE(k_new, pos).
    changed = np.any(t["kc"] != kc0, axis=(1, 2)) | np.any(t["vc"] != vc0, axis=(1, 2))
    assert changed.tolist() == [s == pos for s in range(cfg["s_max"])]
    np.testing.assert_allclose(t["vc"][pos], v_new, rtol=1e-13)
    k_rot = np.stack([oracle.rope(k_new[j], pos, cfg["rope_theta"]) for j in range(nkv)])
    np.testing.assert_allclose(t["kc"][pos], k_rot, rtol=1e-12, atol=1e-13)


def test_decode_position_zero_attends_to_new_token_only():
    cfg = _tiny(nq=4, nkv=2)
    t = _draw(cfg, np.random.default_rng(2))
    r = oracle.decode_row(cfg, t["x"], t["g"], t["wqkv"], t["wo"], t["kc"], t["vc"], 0)
    n = oracle.rmsnorm(t["x"], t["g"], cfg["rms_eps"])
    y = n @ t["wqkv"]
    nq, nkv, d = 4, 2, cfg["head_dim"]
    v_new = y[(nq + nkv) * d:].reshape(nkv, d)
    np.testing.assert_allclose(r["o"].reshape(nq, d), v_new[[0, 0, 1, 1]], rtol=1e-12)
    # RoPE at position 0 is the identity, so the cached key is the raw projection.
    np.testing.assert_allclose(t["kc"][0], y[nq * d:(nq + nkv) * d].reshape(nkv, d),
                               rtol=1e-12)


def test_decode_query_heads_rotated_by_position():
    cfg = _tiny(nq=2, nkv=1, d=8, H=32, S=40)
    t = _draw(cfg, np.random.default_rng(3))
    pos = 33
    r = oracle.decode_row(cfg, t["x"], t["g"], t["wqkv"], t["wo"], t["kc"], t["vc"], pos)
    y = oracle.rmsnorm(t["x"], t["g"], cfg["rms_eps"]) @ t["wqkv"]
    q = y[: 2 * 8].reshape(2, 8)
    for h in range(2):
        np.testing.assert_allclose(r["q"][h * 8:(h + 1) * 8],
                                   oracle.rope(q[h], pos, cfg["rope_theta"]), rtol=1e-12)


def test_gqa_equals_mha_with_repeat_interleaved_kv_heads():
    # Consecutive grouping [LNA §三]: query head h reads KV head h // (nq/nkv).
    nq, nkv, d, H, S = 6, 2, 8, 32, 12
    cfg_g = _tiny(nq=nq, nkv=nkv, d=d, H=H, S=S)
    cfg_m = _tiny(nq=nq, nkv=nq, d=d, H=H, S=S)
    t = _draw(cfg_g, np.random.default_rng(4))
    grp = nq // nkv
    wq = t["wqkv"][:, : nq * d]
    wk = t["wqkv"][:, nq * d:(nq + nkv) * d].reshape(H, nkv, d)
    wv = t["wqkv"][:, (nq + nkv) * d:].reshape(H, nkv, d)
    wqkv_m = np.concatenate([wq, np.repeat(wk, grp, axis=1).reshape(H, nq * d),
                             np.repeat(wv, grp, axis=1).reshape(H, nq * d)], axis=1)
    kc_m = np.ascontiguousarray(np.repeat(t["kc"], grp, axis=1))
    vc_m = np.ascontiguousarray(np.repeat(t["vc"], grp, axis=1))
    rg = oracle.decode_row(cfg_g, t["x"], t["g"], t["wqkv"], t["wo"], t["kc"], t["vc"], 7)
    rm = oracle.decode_row(cfg_m, t["x"], t["g"], wqkv_m, t["wo"], kc_m, vc_m, 7)
    np.testing.assert_allclose(rg["out"], rm["out"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rg["o"], rm["o"], rtol=1e-13, atol=1e-14)


def test_decode_matches_brute_force_triple_loop_on_tiny_shape():
    # Brute force: every sum written as an explicit Python loop (tiny sizes).
    cfg = _tiny(nq=2, nkv=1, d=4, H=6, S=4, theta=10.0, eps=1e-3)
    t = _draw(cfg, np.random.default_rng(5))
    pos = 2
    x, g, W, Wo = t["x"], t["g"], t["wqkv"], t["wo"]
    kc, vc = t["kc"].copy(), t["vc"].copy()
    r = oracle.decode_row(cfg, x, g, W, Wo, t["kc"], t["vc"], pos)
    H, d = 6, 4
    ms = sum(x[i] * x[i] for i in range(H)) / H
    n = [x[i] / math.sqrt(ms + 1e-3) * g[i] for i in range(H)]
    y = [sum(n[i] * W[i][j] for i in range(H)) for j in range(W.shape[1])]

    def rot(u):
        out = list(u)
        for i in range(d // 2):
            ang = pos * 10.0 ** (-2.0 * i / d)
            out[i] = u[i] * math.cos(ang) - u[i + d // 2] * math.sin(ang)
            out[i + d // 2] = u[i + d // 2] * math.cos(ang) + u[i] * math.sin(ang)
        return out

    qs = [rot(y[0:4]), rot(y[4:8])]
    k_new, v_new = rot(y[8:12]), y[12:16]
    keys = [list(kc[t_, 0]) for t_ in range(pos)] + [k_new]
    vals = [list(vc[t_, 0]) for t_ in range(pos)] + [v_new]
    o = []
    for qh in qs:
        s = [sum(qh[i] * kk[i] for i in range(d)) / math.sqrt(d) for kk in keys]
        e = [math.exp(si) for si in s]
        z = sum(e)
        o += [sum(e[t_] / z * vals[t_][i] for t_ in range(pos + 1)) for i in range(d)]
    out = [x[j] + sum(o[k] * Wo[k][j] for k in range(2 * d)) for j in range(H)]
    np.testing.assert_allclose(r["o"], o, rtol=1e-12)
    np.testing.assert_allclose(r["out"], out, rtol=1e-12)


def test_decode_rejects_position_outside_cache():
    cfg = _tiny()
    t = _draw(cfg, np.random.default_rng(6))
    for bad in (-1, cfg["s_max"]):
        with pytest.raises(ValueError):
            oracle.decode_row(cfg, t["x"], t["g"], t["wqkv"], t["wo"], t["kc"], t["vc"], bad)


def test_decode_batch_rows_are_independent():
    cfg = _tiny(S=20)
    rng = np.random.default_rng(7)
    B = 3
    X = rng.normal(size=(B, cfg["hidden"]))
    t = _draw(cfg, rng)
    KC = rng.normal(size=(B, 20, 4, 16))
    VC = rng.normal(size=(B, 20, 4, 16))
    pos = [3, 19, 0]
    full = oracle.decode(cfg, X, t["g"], t["wqkv"], t["wo"], KC.copy(), VC.copy(), pos)
    perm = [2, 0, 1]
    permd = oracle.decode(cfg, X[perm], t["g"], t["wqkv"], t["wo"], KC[perm].copy(),
                          VC[perm].copy(), [pos[i] for i in perm])
    np.testing.assert_array_equal(permd["out"], full["out"][perm])


def test_oracle_regression_fixture():
    # Guards against accidental edits of the oracle (fixture written by
    # tests/golden/gen_oracle_regression.py, which calls only oracle/).
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import gen_oracle_regression as gen
    r = gen.compute()
    with open(os.path.join(here, "tiny_oracle_regression.txt")) as fh:
        rows = [ln.split() for ln in fh if not ln.startswith("#")]
    stored = {row[0]: np.array([float(v) for v in row[1:]]) for row in rows}
    np.testing.assert_allclose(r["out"][0], stored["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["o"][0], stored["o"], rtol=1e-12, atol=1e-13)


def test_ffn_oracle_regression_fixture():
    # The same guard for the FFN oracle (tiny FFN workload, seed 0).
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import gen_oracle_regression as gen
    r = gen.compute_ffn()
    with open(os.path.join(here, "tiny_ffn_oracle_regression.txt")) as fh:
        rows = [ln.split() for ln in fh if not ln.startswith("#")]
    stored = {row[0]: np.array([float(v) for v in row[1:]]) for row in rows}
    np.testing.assert_allclose(r["out"][0], stored["out"], rtol=1e-12, atol=1e-13)


def test_mla_oracle_regression_fixture():
    # The same guard for the MLA oracle (tiny MLA workload, seed 0).
    import os
    import sys
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, here)
    import gen_oracle_regression as gen
    r = gen.compute_mla()
    with open(os.path.join(here, "tiny_mla_oracle_regression.txt")) as fh:
        rows = [ln.split() for ln in fh if not ln.startswith("#")]
    stored = {row[0]: np.array([float(v) for v in row[1:]]) for row in rows}
    np.testing.assert_allclose(r["out"], stored["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["o"], stored["o"], rtol=1e-12, atol=1e-13)


# --------------------------------------------- second RMSNorm + SwiGLU FFN --
# [LNA §一] puts "第二个 RMS Norm、FFN" after the residual of the attention block
# of the LLaMA architecture; the FFN is read as LLaMA's gated form
# out = h + (silu(n Wg^T) * (n Wu^T)) Wd, with Wg, Wu, Wd [I, H].
def test_silu_closed_forms():
    # silu(z) = z * sigmoid(z): silu(0) = 0, silu(z) - silu(-z) = z exactly in
    # real arithmetic (sigmoid(z) + sigmoid(-z) = 1), silu(1) = 1/(1 + 1/e),
    # silu(z) -> z for large z, slope 1/2 at 0.
    assert oracle.silu(0.0) == 0.0
    for z in (0.3, -1.7, 4.0, 11.0):
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14 * max(1.0, abs(z))
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(1e-6) / 1e-6 - 0.5) < 1e-6


def _ffn_inputs(H, I, seed=0):
    r = np.random.default_rng(seed)
    return (r.normal(size=H), 1.0 + 0.1 * r.normal(size=H), 0.2 * r.normal(size=(I, H)),
            0.2 * r.normal(size=(I, H)), 0.2 * r.normal(size=(I, H)))


def test_ffn_hand_example_gate_and_up_roles():
    # h = 1, g2 = 1, eps = 0 gives n = 1.  Unit i's gate row sums to 1 and its
    # up row to 2, so a_i = silu(1) * 2 = 1.4621171572600098; swapping the two
    # matrices gives silu(2) * 1 = 1.7615941559557649 instead (the activation
    # belongs to the gate).  Wd = [[0,1,2,3],[4,5,6,7]] then sums the units.
    H = 4
    wg = np.array([[1.0, 0, 0, 0], [0, 0.5, 0.5, 0]])
    wu = np.array([[2.0, 0, 0, 0], [0, 0, 1.0, 1.0]])
    wd = np.arange(8.0).reshape(2, 4)
    r = oracle.ffn_row(np.ones(H), np.ones(H), wg, wu, wd, 0.0)
    a = 1.4621171572600098
    np.testing.assert_allclose(r["a"], [a, a], rtol=1e-15)
    np.testing.assert_allclose(r["out"], 1.0 + a * np.array([4.0, 6.0, 8.0, 10.0]), rtol=1e-15)
    r2 = oracle.ffn_row(np.ones(H), np.ones(H), wu, wg, wd, 0.0)
    np.testing.assert_allclose(r2["a"], [1.7615941559557649] * 2, rtol=1e-15)


def test_ffn_zero_matrices_give_the_residual_exactly():
    h, g2, wg, wu, wd = _ffn_inputs(16, 24)
    for k in range(3):
        mats = [wg, wu, wd]
        mats[k] = np.zeros_like(mats[k])
        r = oracle.ffn_row(h, g2, *mats, 1e-6)
        assert np.array_equal(r["out"], h), k


def test_ffn_second_norm_is_the_block_rmsnorm():
    # The FFN input is RMSNorm(h; g2) with eps inside the sqrt: compare with the
    # constant-vector closed form through a one-unit FFN whose gate and up rows
    # pick coordinate 3 (n_3 = g2_3 * c / sqrt(c^2 + eps)).
    H, c, eps = 8, 2.5, 0.5
    g2 = np.linspace(0.5, 1.5, H)
    e3 = np.zeros((1, H))
    e3[0, 3] = 1.0
    r = oracle.ffn_row(np.full(H, c), g2, e3, e3, np.ones((1, H)), eps)
    n3 = g2[3] * c / math.sqrt(c * c + eps)
    assert abs(r["a"][0] - (n3 / (1.0 + math.exp(-n3))) * n3) < 1e-14


def test_ffn_invariant_under_permuting_the_intermediate_units():
    # Reordering the units (the same rows of Wg, Wu and Wd) cannot change the
    # output; a mixed-up row index between the three matrices would.
    h, g2, wg, wu, wd = _ffn_inputs(12, 20, seed=3)
    perm = np.random.default_rng(5).permutation(20)
    r0 = oracle.ffn_row(h, g2, wg, wu, wd, 1e-6)
    r1 = oracle.ffn_row(h, g2, wg[perm], wu[perm], wd[perm], 1e-6)
    np.testing.assert_allclose(r1["out"], r0["out"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(r1["a"], r0["a"][perm], rtol=1e-12, atol=1e-15)


def test_ffn_is_linear_in_down_and_up_and_separable_over_units():
    # out - h is linear in Wd and in Wu, and a sum over the units: splitting the
    # I units into two halves adds the two halves' contributions.
    h, g2, wg, wu, wd = _ffn_inputs(10, 16, seed=7)
    base = oracle.ffn_row(h, g2, wg, wu, wd, 1e-6)["out"] - h
    np.testing.assert_allclose(oracle.ffn_row(h, g2, wg, wu, 3.0 * wd, 1e-6)["out"] - h,
                               3.0 * base, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(oracle.ffn_row(h, g2, wg, -2.0 * wu, wd, 1e-6)["out"] - h,
                               -2.0 * base, rtol=1e-12, atol=1e-13)
    lo = oracle.ffn_row(h, g2, wg[:7], wu[:7], wd[:7], 1e-6)["out"] - h
    hi = oracle.ffn_row(h, g2, wg[7:], wu[7:], wd[7:], 1e-6)["out"] - h
    np.testing.assert_allclose(lo + hi, base, rtol=1e-12, atol=1e-13)


def test_ffn_single_unit_one_hot_weights_transpose_check():
    # Unit 0 reads coordinate 1 of n through both gate and up and writes only
    # output coordinate 4 with weight 2: a transposed Wd (read as [H, I]) or a
    # gate row read as a column moves or drops the contribution.
    H, I = 6, 3
    h = np.linspace(-1.0, 1.5, H)
    g2 = np.ones(H)
    wg = np.zeros((I, H))
    wu = np.zeros((I, H))
    wd = np.zeros((I, H))
    wg[0, 1] = 1.0
    wu[0, 1] = 1.0
    wd[0, 4] = 2.0
    r = oracle.ffn_row(h, g2, wg, wu, wd, 0.0)
    n1 = h[1] / math.sqrt(np.mean(h * h))
    expect = h.copy()
    expect[4] += 2.0 * (n1 / (1.0 + math.exp(-n1))) * n1
    np.testing.assert_allclose(r["out"], expect, rtol=1e-14, atol=1e-15)


# -------------------------------------------------------- MLA variant --
# [CF §5.2 DeepSeek-MLA特殊处理]; projections read as DeepSeek's MLA with an
# uncompressed query (oracle.h).  Pins: pure-Python brute force of the
# definition, the weight-absorbed form (a different association of the same
# products, as the GPU computes it), one cached token, uniform attention,
# a closed form of the latent RMSNorm, RoPE on the position parts only, and
# the cache write.
def _mla_cfg(H=16, nh=3, dn=4, dr=4, dv=3, dc=6, S=7, theta=1e4, eps=1e-6):
    return dict(hidden=H, n_heads=nh, d_nope=dn, d_rope=dr, d_v=dv, d_latent=dc, s_max=S,
                rope_theta=theta, rms_eps=eps)


def _mla_inputs(cfg, seed=5, std=0.3):
    r = np.random.default_rng(seed)
    H, nh, dn, dr, dv, dc, S = (cfg[k] for k in ("hidden", "n_heads", "d_nope", "d_rope", "d_v",
                                                 "d_latent", "s_max"))
    return dict(x=r.normal(size=H), g=1 + 0.1 * r.normal(size=H),
                wq=std * r.normal(size=(H, nh * (dn + dr))),
                wdkv=std * r.normal(size=(H, dc + dr)), g_kv=1 + 0.1 * r.normal(size=dc),
                wukv=std * r.normal(size=(dc, nh * (dn + dv))),
                wo=std * r.normal(size=(nh * dv, H)), lc=r.normal(size=(S, dc + dr)))


def _mla(cfg, t, pos, lc=None):
    lc = t["lc"].copy() if lc is None else lc
    res = oracle.mla_row(cfg, t["x"], t["g"], t["wq"], t["wdkv"], t["g_kv"], t["wukv"],
                         t["wo"], lc, pos)
    return res, lc


def test_mla_brute_force_python_loops():
    cfg = _mla_cfg(H=6, nh=2, dn=2, dr=2, dv=3, dc=3, S=4, theta=100.0, eps=1e-3)
    t = _mla_inputs(cfg, seed=8, std=0.5)
    pos = 2
    res, lc = _mla(cfg, t, pos)
    H, nh, dn, dr, dv, dc = 6, 2, 2, 2, 3, 3
    x, g = list(t["x"]), list(t["g"])
    ms = sum(v * v for v in x) / H
    n = [x[i] / math.sqrt(ms + 1e-3) * g[i] for i in range(H)]
    q = [sum(n[i] * t["wq"][i][j] for i in range(H)) for j in range(nh * (dn + dr))]
    a = [sum(n[i] * t["wdkv"][i][j] for i in range(H)) for j in range(dc + dr)]
    msc = sum(a[i] * a[i] for i in range(dc)) / dc
    lat = [a[i] / math.sqrt(msc + 1e-3) * t["g_kv"][i] for i in range(dc)]
    # rotate-half over dr = 2: one pair (0, 1), angle pos * 100^0 = pos
    ang = float(pos)

    def rot(u0, u1):
        return u0 * math.cos(ang) - u1 * math.sin(ang), u1 * math.cos(ang) + u0 * math.sin(ang)

    lat += list(rot(a[dc], a[dc + 1]))
    for h in range(nh):
        b = h * (dn + dr) + dn
        q[b], q[b + 1] = rot(q[b], q[b + 1])
    rows = [list(t["lc"][s]) for s in range(pos)] + [lat]
    o = []
    for h in range(nh):
        qh = q[h * (dn + dr):(h + 1) * (dn + dr)]
        scores, vals = [], []
        for row in rows:
            k = [sum(row[i] * t["wukv"][i][h * (dn + dv) + j] for i in range(dc))
                 for j in range(dn)] + row[dc:]
            v = [sum(row[i] * t["wukv"][i][h * (dn + dv) + dn + j] for i in range(dc))
                 for j in range(dv)]
            scores.append(sum(qh[j] * k[j] for j in range(dn + dr)) / math.sqrt(dn + dr))
            vals.append(v)
        mx = max(scores)
        e = [math.exp(s - mx) for s in scores]
        o += [sum(e[t_] * vals[t_][j] for t_ in range(len(rows))) / sum(e) for j in range(dv)]
    out = [x[i] + sum(o[k] * t["wo"][k][i] for k in range(nh * dv)) for i in range(H)]
    np.testing.assert_allclose(res["lat"], lat, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["q"], q, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["o"], o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["out"], out, rtol=1e-12, atol=1e-13)


def test_mla_weight_absorbed_form_matches():
    # The GPU's association: q_lat_h = Wuk_h q_nope_h (dc values), scores
    # against the latent rows directly, o_lat_h = sum_t w_t L[t,:dc], then
    # o_h = o_lat_h . Wuv_h.  Same products, different order.
    cfg = _mla_cfg(H=24, nh=4, dn=8, dr=6, dv=5, dc=10, S=9)
    t = _mla_inputs(cfg)
    pos = 7
    res, lc = _mla(cfg, t, pos)
    nh, dn, dr, dv, dc = 4, 8, 6, 5, 10
    W = t["wukv"].reshape(dc, nh, dn + dv)
    L = lc[:pos + 1]
    o = np.empty((nh, dv))
    for h in range(nh):
        qh = res["q"][h * (dn + dr):(h + 1) * (dn + dr)]
        q_lat = W[:, h, :dn] @ qh[:dn]
        s = (L[:, :dc] @ q_lat + L[:, dc:] @ qh[dn:]) / math.sqrt(dn + dr)
        w = np.exp(s - s.max())
        w /= w.sum()
        o[h] = (w @ L[:, :dc]) @ W[:, h, dn:]
    np.testing.assert_allclose(res["o"], o.reshape(-1), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(res["proj"], o.reshape(-1) @ t["wo"], rtol=1e-11, atol=1e-13)


def test_mla_one_token_attends_to_its_own_value():
    cfg = _mla_cfg()
    t = _mla_inputs(cfg, seed=9)
    res, lc = _mla(cfg, t, 0)
    nh, dn, dv, dc = 3, 4, 3, 6
    W = t["wukv"].reshape(dc, nh, dn + dv)
    v0 = np.concatenate([res["lat"][:dc] @ W[:, h, dn:] for h in range(nh)])
    np.testing.assert_allclose(res["o"], v0, rtol=1e-12, atol=1e-14)


def test_mla_zero_query_gives_uniform_attention():
    cfg = _mla_cfg()
    t = _mla_inputs(cfg, seed=10)
    t["wq"][:] = 0.0
    pos = 5
    res, lc = _mla(cfg, t, pos)
    nh, dn, dv, dc = 3, 4, 3, 6
    W = t["wukv"].reshape(dc, nh, dn + dv)
    mean_lat = lc[:pos + 1, :dc].mean(axis=0)  # includes the new row
    want = np.concatenate([mean_lat @ W[:, h, dn:] for h in range(nh)])
    np.testing.assert_allclose(res["o"], want, rtol=1e-12, atol=1e-14)


def test_mla_latent_norm_closed_form():
    # Every compressed column of Wdkv the same vector w: c_i = n . w = kappa
    # for all i, so RMSNorm gives c'_i = g_kv_i kappa / sqrt(kappa^2 + eps).
    cfg = _mla_cfg(eps=0.04)
    t = _mla_inputs(cfg, seed=11)
    dc = 6
    t["wdkv"][:, :dc] = t["wdkv"][:, :1]
    res, _ = _mla(cfg, t, 3)
    n = oracle.rmsnorm(t["x"], t["g"], 0.04)
    kappa = n @ t["wdkv"][:, 0]
    np.testing.assert_allclose(res["lat"][:dc], t["g_kv"] * kappa / math.sqrt(kappa ** 2 + 0.04),
                               rtol=1e-12)


def test_mla_rope_only_on_position_parts_and_only_slot_pos_written():
    cfg = _mla_cfg()
    t = _mla_inputs(cfg, seed=12)
    nh, dn, dr, dc = 3, 4, 4, 6
    n = oracle.rmsnorm(t["x"], t["g"], 1e-6)
    q_lin = (n @ t["wq"]).reshape(nh, dn + dr)
    a_lin = n @ t["wdkv"]
    for pos in (0, 4):
        res, lc = _mla(cfg, t, pos)
        q = res["q"].reshape(nh, dn + dr)
        np.testing.assert_allclose(q[:, :dn], q_lin[:, :dn], rtol=1e-13)  # never rotated
        for h in range(nh):
            np.testing.assert_allclose(q[h, dn:], oracle.rope(q_lin[h, dn:], pos, 1e4),
                                       rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(res["lat"][dc:], oracle.rope(a_lin[dc:], pos, 1e4),
                                   rtol=1e-12, atol=1e-14)
        if pos == 0:
            np.testing.assert_allclose(q, q_lin, rtol=1e-13)  # RoPE at 0 is the identity
        changed = np.any(lc != t["lc"], axis=1)
        assert list(np.nonzero(changed)[0]) == [pos]
        np.testing.assert_array_equal(lc[pos], res["lat"])


def test_mla_rejects_bad_position():
    cfg = _mla_cfg()
    t = _mla_inputs(cfg)
    for pos in (-1, cfg["s_max"]):
        with pytest.raises(ValueError):
            _mla(cfg, t, pos)
