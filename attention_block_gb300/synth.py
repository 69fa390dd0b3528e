"""Seeded synthetic inputs for the decode attention block.

This module is the one piece shared by the CUDA path's tests/bench and the
float64 oracle's tests: it draws random tensors and holds none of the
method's arithmetic.  Draw order per layer is fixed: hidden, ln_weight,
W_qkv, W_o, k_cache, v_cache, positions.

Value laws (the same for every workload): hidden ~ N(0,1), ln_weight ~
1 + N(0, 0.1), W_qkv and W_o ~ N(0, 0.02), KV cache ~ N(0,1) everywhere
(including the slot the new token will overwrite, so an append is visible).

The FFN that follows the attention block (second RMSNorm, gated FFN,
residual) draws, in this order, hidden ~ N(0,1) (unless the attention
block's output is passed in), its norm weight ~ 1 + N(0, 0.1) and W_gate,
W_up, W_down ~ N(0, 0.02), each [I, H]: the same laws as the attention
block's, since no workload states others.
"""
from __future__ import annotations

import dataclasses

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    batch: int
    s_max: int          # cache capacity per sequence
    dtype: str          # storage dtype: f32 | f16 | bf16
    rope_theta: float
    rms_eps: float
    positions: str      # "fixed:P" or "distinct:LO:HI" (inclusive)
    layers: int = 1

    @property
    def qkv_cols(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def oracle_cfg(self) -> dict:
        return dict(hidden=self.hidden, n_q_heads=self.n_q_heads,
                    n_kv_heads=self.n_kv_heads, head_dim=self.head_dim,
                    s_max=self.s_max, rope_theta=self.rope_theta,
                    rms_eps=self.rms_eps)


# The five workloads of the benchmark set, named by what they are.
WORKLOADS = {w.name: w for w in [
    Workload("tiny_h256_mha4x64_b1_p128_f32", 256, 4, 4, 64, 1, 129, "f32",
             1e4, 1e-6, "fixed:128"),
    Workload("llama2_7b_layer_b1_p1024_f16", 4096, 32, 32, 128, 1, 1025, "f16",
             1e4, 1e-6, "fixed:1024"),
    Workload("h2048_mha32x64_b64_p1024to2048_f16", 2048, 32, 32, 64, 64, 2049,
             "f16", 1e4, 1e-6, "distinct:1024:2048"),
    Workload("llama3_8b_gqa32x8_b16_p4096_bf16", 4096, 32, 8, 128, 16, 4097,
             "bf16", 5e5, 1e-6, "fixed:4096"),
    Workload("llama2_7b_layer_b1_p16384_f16_x32", 4096, 32, 32, 128, 1, 16385,
             "f16", 1e4, 1e-6, "fixed:16384", layers=32),
]}

TINY = "tiny_h256_mha4x64_b1_p128_f32"
LLAMA2_1K = "llama2_7b_layer_b1_p1024_f16"
SMALL_HEAD_B64 = "h2048_mha32x64_b64_p1024to2048_f16"
LLAMA3_GQA = "llama3_8b_gqa32x8_b16_p4096_bf16"
LLAMA2_16K_X32 = "llama2_7b_layer_b1_p16384_f16_x32"


def custom(name: str = "custom", **kw) -> Workload:
    base = dict(hidden=256, n_q_heads=4, n_kv_heads=4, head_dim=64, batch=1,
                s_max=129, dtype="f32", rope_theta=1e4, rms_eps=1e-6,
                positions="fixed:128", layers=1)
    base.update(kw)
    return Workload(name=name, **base)


def _positions(w: Workload, gen: torch.Generator, device) -> torch.Tensor:
    kind, *args = w.positions.split(":")
    if kind == "fixed":
        p = int(args[0])
        return torch.full((w.batch,), p, dtype=torch.int32, device=device)
    if kind == "distinct":
        lo, hi = int(args[0]), int(args[1])
        perm = torch.randperm(hi - lo + 1, generator=gen, device=device)
        return (perm[: w.batch] + lo).to(torch.int32)
    if kind == "list":
        vals = [int(v) for v in args[0].split(",")]
        assert len(vals) == w.batch
        return torch.tensor(vals, dtype=torch.int32, device=device)
    raise ValueError(w.positions)


def make_layer(w: Workload, seed: int = 0, device="cpu") -> dict:
    """Draw one layer's tensors (storage dtype) on ``device``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    dt = DTYPES[w.dtype]
    B, H, S = w.batch, w.hidden, w.s_max
    nq, nkv, d = w.n_q_heads, w.n_kv_heads, w.head_dim

    def randn(*shape, std=1.0, mean=0.0):
        t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        if mean != 0.0:
            t.add_(mean)
        return t.to(dt)

    out = {}
    out["hidden"] = randn(B, H)
    out["ln_weight"] = randn(H, std=0.1, mean=1.0)
    out["w_qkv"] = randn(H, w.qkv_cols, std=0.02)
    out["w_o"] = randn(nq * d, H, std=0.02)
    out["k_cache"] = randn(B, S, nkv, d)
    out["v_cache"] = randn(B, S, nkv, d)
    out["positions"] = _positions(w, gen, device)
    return out


@dataclasses.dataclass(frozen=True)
class FfnWorkload:
    name: str
    hidden: int
    intermediate: int
    batch: int
    dtype: str
    rms_eps: float


# FFN shapes of the two model families the attention workloads stand in for
# (Llama-2-7B: I = 11008; Llama-3-8B: I = 14336), plus a small fp32 case.
FFN_WORKLOADS = {w.name: w for w in [
    FfnWorkload("llama2_7b_ffn_i11008_b1_f16", 4096, 11008, 1, "f16", 1e-6),
    FfnWorkload("llama3_8b_ffn_i14336_b2_bf16", 4096, 14336, 2, "bf16", 1e-6),
    FfnWorkload("tiny_ffn_h256_i688_b1_f32", 256, 688, 1, "f32", 1e-6),
    # batched decode: the FFNs that follow the 64-row, 2048-hidden layer
    # (intermediate 5632 = 8/3 * 2048 rounded up to a multiple of 256, the
    # LLaMA sizing rule) and the 16-row Llama-3 GQA layer
    FfnWorkload("h2048_ffn_i5632_b64_f16", 2048, 5632, 64, "f16", 1e-6),
    FfnWorkload("llama3_8b_ffn_i14336_b16_bf16", 4096, 14336, 16, "bf16", 1e-6),
]}
LLAMA2_FFN = "llama2_7b_ffn_i11008_b1_f16"
LLAMA3_FFN = "llama3_8b_ffn_i14336_b2_bf16"
TINY_FFN = "tiny_ffn_h256_i688_b1_f32"
B64_FFN = "h2048_ffn_i5632_b64_f16"
LLAMA3_FFN_B16 = "llama3_8b_ffn_i14336_b16_bf16"


def custom_ffn(name: str = "custom_ffn", **kw) -> FfnWorkload:
    base = dict(hidden=256, intermediate=688, batch=1, dtype="f32", rms_eps=1e-6)
    base.update(kw)
    return FfnWorkload(name=name, **base)


def make_ffn(w: FfnWorkload, seed: int = 0, device="cpu", hidden=None) -> dict:
    """Draw one FFN's tensors (storage dtype) on ``device``; ``hidden`` [B, H]
    (e.g. the attention block's output) replaces the drawn input rows."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    dt = DTYPES[w.dtype]
    B, H, I = w.batch, w.hidden, w.intermediate

    def randn(*shape, std=1.0, mean=0.0):
        t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        if mean != 0.0:
            t.add_(mean)
        return t.to(dt)

    out = {"hidden": randn(B, H)}
    if hidden is not None:
        out["hidden"] = hidden.to(device=device, dtype=dt).contiguous()
    out["ln_weight"] = randn(H, std=0.1, mean=1.0)
    out["w_gate"] = randn(I, H, std=0.02)
    out["w_up"] = randn(I, H, std=0.02)
    out["w_down"] = randn(I, H, std=0.02)
    return out


def to_f64(t: torch.Tensor):
    """Exact conversion of storage values to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
