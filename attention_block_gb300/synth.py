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


def workload(spec: str) -> Workload:
    """A named workload, or an ad-hoc one written as
    ``custom:hidden=H,q=NQ,kv=NKV,d=D,batch=B,pos=P[,dtype=T][,theta=X][,layers=L]``
    (every row at position P, cache capacity P + 1; dtype f16 by default)."""
    if not spec.startswith("custom:"):
        return WORKLOADS[spec]
    kv = dict(item.split("=", 1) for item in spec[len("custom:"):].split(",") if item)
    known = {"hidden", "q", "kv", "d", "batch", "pos", "dtype", "theta", "layers"}
    unknown = set(kv) - known
    if unknown:
        raise ValueError(f"unknown workload keys {sorted(unknown)} in {spec!r}")
    pos = int(kv["pos"])
    return Workload(spec, int(kv["hidden"]), int(kv["q"]), int(kv["kv"]), int(kv["d"]),
                    int(kv["batch"]), pos + 1, kv.get("dtype", "f16"),
                    float(kv.get("theta", 1e4)), 1e-6, f"fixed:{pos}",
                    layers=int(kv.get("layers", 1)))


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


@dataclasses.dataclass(frozen=True)
class MlaWorkload:
    """The DeepSeek multi-head latent attention (MLA) variant of the block."""
    name: str
    hidden: int
    n_heads: int
    d_nope: int
    d_rope: int
    d_v: int
    d_latent: int
    batch: int
    s_max: int
    dtype: str
    rope_theta: float
    rms_eps: float
    positions: str

    def oracle_cfg(self) -> dict:
        return dict(hidden=self.hidden, n_heads=self.n_heads, d_nope=self.d_nope,
                    d_rope=self.d_rope, d_v=self.d_v, d_latent=self.d_latent, s_max=self.s_max,
                    rope_theta=self.rope_theta, rms_eps=self.rms_eps)


# MLA layers shaped like DeepSeek-V2-Lite's attention (hidden 2048, 16 heads,
# 128 + 64 query/key dims, 128 value dims, a 512-dim latent), at the two
# sequence lengths the pages measure MLA at (4K and 16K), and a tiny layer
# with the same head dims.
MLA_WORKLOADS = {w.name: w for w in [
    MlaWorkload("deepseek_v2_lite_mla_b1_p4096_bf16", 2048, 16, 128, 64, 128, 512, 1, 4097,
                "bf16", 1e4, 1e-6, "fixed:4096"),
    MlaWorkload("deepseek_v2_lite_mla_b1_p16384_bf16", 2048, 16, 128, 64, 128, 512, 1, 16385,
                "bf16", 1e4, 1e-6, "fixed:16384"),
    MlaWorkload("tiny_mla_h512_h8_b1_p128_bf16", 512, 8, 128, 64, 128, 512, 1, 129, "bf16",
                1e4, 1e-6, "fixed:128"),
]}
MLA_4K = "deepseek_v2_lite_mla_b1_p4096_bf16"
MLA_16K = "deepseek_v2_lite_mla_b1_p16384_bf16"
MLA_TINY = "tiny_mla_h512_h8_b1_p128_bf16"


def custom_mla(name: str = "custom_mla", **kw) -> MlaWorkload:
    base = dict(hidden=512, n_heads=8, d_nope=128, d_rope=64, d_v=128, d_latent=512, batch=1,
                s_max=129, dtype="bf16", rope_theta=1e4, rms_eps=1e-6, positions="fixed:128")
    base.update(kw)
    return MlaWorkload(name=name, **base)


def make_mla_layer(w: MlaWorkload, seed: int = 0, device="cpu") -> dict:
    """Draw one MLA layer's tensors (storage dtype) on ``device``, in the order
    hidden, ln_weight, w_q, w_dkv, kv_norm_weight, w_ukv, w_o, latent cache,
    positions.  Laws as for the attention block: hidden ~ N(0,1), norm
    weights ~ 1 + N(0, 0.1), weights ~ N(0, 0.02), the latent cache ~ N(0,1)
    over its whole capacity."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    dt = DTYPES[w.dtype]
    B, H, S, nh = w.batch, w.hidden, w.s_max, w.n_heads
    dn, dr, dv, dc = w.d_nope, w.d_rope, w.d_v, w.d_latent

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
    out["w_q"] = randn(H, nh * (dn + dr), std=0.02)
    out["w_dkv"] = randn(H, dc + dr, std=0.02)
    out["kv_norm_weight"] = randn(dc, std=0.1, mean=1.0)
    out["w_ukv"] = randn(dc, nh * (dn + dv), std=0.02)
    out["w_o"] = randn(nh * dv, H, std=0.02)
    out["latent_cache"] = randn(B, S, dc + dr)
    out["positions"] = _positions(w, gen, device)
    return out


def to_f64(t: torch.Tensor):
    """Exact conversion of storage values to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()
