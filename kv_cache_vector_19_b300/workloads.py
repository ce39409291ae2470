"""Seeded synthetic inputs for the TurboQuant KV-cache quantize + decode path.

This module only draws random tensors.  It contains none of the method's arithmetic and
is the single piece of code shared by the library's tests, the benchmark and the oracle.

There is no model, checkpoint or dataset here: the K/V/Q tensors are synthetic stand-ins
with the shapes of the layers the pages talk about (Llama-3.1-8B: 32 query / 8 KV heads,
head_dim 128; Llama-3-70B: 64 / 8 / 128) and the value distributions named per workload:

  tiny        1 x 1 KV head, 16 queries, 4096 tokens, d=128, b=3; N(0,1) with 4 outlier
              channels x20 (the same 4 channels in K and V)
  llama8b     batch 1, 8 KV / 32 Q heads, 32768 tokens, d=128, b=4; N(0,1) times a
              per-(kv head, channel) log-normal scale exp(N(0,1)), drawn separately for K, V
  longctx     batch 4, 8 KV / 32 Q heads, 131072 tokens, d=128, b=3, N(0,1); then 64 decode
              steps, each appending one N(0,1) token per (batch, kv head) with a new query
  llama70b    batch 16, 8 KV / 64 Q heads, 32768 tokens, d=128, b=3; K = N(0,1) times
              log-normal channel scales, and 1% of the tokens of every (batch, kv head)
              scaled x10; V plain N(0,1)
  sweep       1 KV head, 65536 tokens, d in {64,128,256}, b in {2,3,4,5}, N(0,1); 16 queries

Every draw comes from one numpy Generator(PCG64(seed)) in a fixed order: K, V, K channel
scales, V channel scales, outlier channel picks, outlier token picks, Q, then the appended
tokens and queries of each decode step.  fp32 draws are rounded to bf16 (round to nearest
even) after scaling; queries stay fp32.
"""
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    batch: int
    kv_heads: int
    q_heads: int
    tokens: int
    d: int
    b: int
    m: int
    seed: int = 0
    kind: str = "normal"          # normal | outlier_channels | lognormal | lognormal_outlier_tokens
    decode_steps: int = 1         # queries drawn per run; >1 means one appended token per step
    extra: dict = field(default_factory=dict)

    @property
    def group(self):
        return self.q_heads // self.kv_heads

    @property
    def max_tokens(self):
        return self.tokens + (self.decode_steps if self.decode_steps > 1 else 0)


PRESETS = {
    "tiny": dict(batch=1, kv_heads=1, q_heads=16, tokens=4096, d=128, b=3, kind="outlier_channels"),
    "llama8b": dict(batch=1, kv_heads=8, q_heads=32, tokens=32768, d=128, b=4, kind="lognormal"),
    "longctx": dict(batch=4, kv_heads=8, q_heads=32, tokens=131072, d=128, b=3, kind="normal",
                    decode_steps=64),
    "llama70b": dict(batch=16, kv_heads=8, q_heads=64, tokens=32768, d=128, b=3,
                     kind="lognormal_outlier_tokens"),
}


def preset(name, **override):
    cfg = dict(PRESETS[name])
    cfg.update(override)
    cfg.setdefault("m", cfg["d"])
    return Workload(name=name, **cfg)


def sweep_point(d, b, tokens=65536, seed=0):
    return Workload(name=f"sweep_d{d}_b{b}", batch=1, kv_heads=1, q_heads=1, tokens=tokens,
                    d=d, b=b, m=d, seed=seed, kind="normal", extra=dict(n_queries=16))


def to_bf16(x_f32):
    """fp32 numpy array -> torch bf16 tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)


def generate(w: Workload):
    """Returns dict(k, v: bf16 [B, Hkv, T, d] CPU tensors; q: fp32 [steps, B, Hq, d];
    k_new, v_new: bf16 [steps, B, Hkv, 1, d] (present when decode_steps > 1))."""
    rng = np.random.default_rng(w.seed)
    shape = (w.batch, w.kv_heads, w.tokens, w.d)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if w.kind in ("lognormal", "lognormal_outlier_tokens"):
        sk = np.exp(rng.standard_normal((w.kv_heads, w.d))).astype(np.float32)
        sv = np.exp(rng.standard_normal((w.kv_heads, w.d))).astype(np.float32)
        k *= sk[None, :, None, :]
        if w.kind == "lognormal":
            v *= sv[None, :, None, :]
    if w.kind == "outlier_channels":
        ch = rng.choice(w.d, 4, replace=False)
        k[..., ch] *= 20.0
        v[..., ch] *= 20.0
    if w.kind == "lognormal_outlier_tokens":
        n_out = int(0.01 * w.tokens)
        for bb in range(w.batch):
            for hh in range(w.kv_heads):
                toks = rng.choice(w.tokens, n_out, replace=False)
                k[bb, hh, toks, :] *= 10.0
    n_q = w.extra.get("n_queries", 1)
    steps = w.decode_steps
    q = rng.standard_normal((steps, w.batch, w.q_heads * n_q, w.d), dtype=np.float32)
    out = dict(k=to_bf16(k), v=to_bf16(v), q=torch.from_numpy(q))
    del k, v
    if steps > 1:
        kn = rng.standard_normal((steps, w.batch, w.kv_heads, 1, w.d), dtype=np.float32)
        vn = rng.standard_normal((steps, w.batch, w.kv_heads, 1, w.d), dtype=np.float32)
        out["k_new"] = to_bf16(kn)
        out["v_new"] = to_bf16(vn)
    return out
