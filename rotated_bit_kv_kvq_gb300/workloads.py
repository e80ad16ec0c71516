"""Seeded synthetic workloads (inputs only -- no rotation, quantization or attention here).

Five workload shapes, named by what they are:

  decode_d64_ctx256      1 seq, 1 q head / 1 KV head, head_dim 64, 256 tokens, fp32
                         Q/K/V ~ N(0,1) with 2 of 64 channels x20; q4_0/q4_0, no tail
  decode_gqa16x8_ctx4k   1 seq, 16 q / 8 KV heads, head_dim 128, 4096 tokens, fp32;
                         K,V 4 outlier channels per head x20; q8_0/q8_0, tail 256
  decode_b32_ragged8k    32 seqs of 1024..8192 tokens (uniform), 32 q / 8 KV heads,
                         head_dim 128, bf16; q5_0/q5_0, tail 512
  decode_b4_ctx64k       4 seqs x 65536 tokens, 24 q / 4 KV heads, head_dim 256, bf16;
                         K q8_0 / V q4_0, tail 1024, one appended token per seq per step
  prefill_b2_4k          2 prompts x 4096 tokens, 32 q / 8 KV heads, head_dim 128, bf16,
                         causal, chunk 512; q4_0/q4_0, tail 256

The outlier channels are "specific channels" of a head (the pages' description
of KV activations): per KV head a seeded choice of channels, fixed across
tokens, multiplied by 20.  K and V draw their channel sets independently; in
the first workload Q shares the K set of its KV head.

Random numbers come from numpy's PCG64 with the given seed (0 by default).
bf16 workloads round their inputs with torch's bf16 conversion, so both the
CUDA path and the oracle receive the same bf16 values.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx: int                      # tokens per sequence (max for ragged)
    k_type: str
    v_type: str
    tail_len: int
    dtype: str                    # "f32" or "bf16" for Q/K/V inputs
    n_outliers: int
    outlier_in_q: bool = False
    ragged_min: Optional[int] = None  # ragged lengths ~ U[ragged_min, ctx]
    prefill: bool = False
    chunk: int = 512
    append_per_step: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def max_ctx(self, extra: int = 0) -> int:
        """Cache capacity: ctx plus `extra` appended tokens, rounded up to 64."""
        n = self.ctx + extra
        return (n + 63) // 64 * 64

    def scaled(self, ctx: Optional[int] = None, batch: Optional[int] = None,
               ragged_min: Optional[int] = None, tail_len: Optional[int] = None) -> "Workload":
        """A reduced variant (same formats and head layout) for quick tests."""
        kw = {}
        if ctx is not None:
            kw["ctx"] = ctx
        if batch is not None:
            kw["batch"] = batch
        if ragged_min is not None:
            kw["ragged_min"] = ragged_min
        if tail_len is not None:
            kw["tail_len"] = tail_len
        return dataclasses.replace(self, name=self.name + "_reduced", **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("decode_d64_ctx256", 1, 1, 1, 64, 256, "q4_0", "q4_0", 0, "f32", 2,
                 outlier_in_q=True),
        Workload("decode_gqa16x8_ctx4k", 1, 16, 8, 128, 4096, "q8_0", "q8_0", 256, "f32", 4),
        Workload("decode_b32_ragged8k", 32, 32, 8, 128, 8192, "q5_0", "q5_0", 512, "bf16", 4,
                 ragged_min=1024),
        Workload("decode_b4_ctx64k", 4, 24, 4, 256, 65536, "q8_0", "q4_0", 1024, "bf16", 4,
                 append_per_step=1),
        Workload("prefill_b2_4k", 2, 32, 8, 128, 4096, "q4_0", "q4_0", 256, "bf16", 4,
                 prefill=True, chunk=512),
    ]
}

# The decode workload the headline throughput is quoted on (64k context).
HEADLINE = "decode_b4_ctx64k"


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (torch's conversion) and return them as float32."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def _as_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32)
    return round_bf16(x) if dtype == "bf16" else x


@dataclasses.dataclass
class DecodeInputs:
    lengths: np.ndarray           # [B] int64, tokens already in the cache
    k_hist: np.ndarray            # [B][ctx][Hkv][d] float32 (bf16-valued for bf16 workloads)
    v_hist: np.ndarray
    q: np.ndarray                 # [B][Hq][d] (decode) or [B][n][Hq][d] (prefill)
    k_chan: np.ndarray            # [Hkv][n_outliers] outlier channels of K
    v_chan: np.ndarray


def outlier_channels(rng: np.random.Generator, n_kv_heads: int, head_dim: int, n: int) -> np.ndarray:
    return np.stack([np.sort(rng.choice(head_dim, n, replace=False)) for _ in range(n_kv_heads)])


def _apply_outliers(x: np.ndarray, chans: np.ndarray, factor: float = 20.0) -> None:
    """x [..., Hkv, d] in place: multiply the chosen channels of each head."""
    for h in range(chans.shape[0]):
        x[..., h, chans[h]] *= factor


def make_inputs(w: Workload, seed: int = 0, batches: Optional[range] = None) -> DecodeInputs:
    """Seeded inputs of workload `w`.  `batches` optionally restricts the
    returned K/V history to some sequences (the draws stay the same)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, Hkv, d, n = w.batch, w.n_kv_heads, w.head_dim, w.ctx
    k_chan = outlier_channels(rng, Hkv, d, w.n_outliers)
    v_chan = outlier_channels(rng, Hkv, d, w.n_outliers)
    if w.ragged_min is not None:
        lengths = rng.integers(w.ragged_min, n + 1, size=B).astype(np.int64)
    else:
        lengths = np.full(B, n, dtype=np.int64)
    ks, vs = [], []
    sel = range(B) if batches is None else batches
    for b in range(B):
        kb = rng.standard_normal((n, Hkv, d), dtype=np.float32)
        vb = rng.standard_normal((n, Hkv, d), dtype=np.float32)
        if b in sel:
            _apply_outliers(kb, k_chan)
            _apply_outliers(vb, v_chan)
            kb[lengths[b]:] = 0.0
            vb[lengths[b]:] = 0.0
            ks.append(_as_dtype(kb, w.dtype))
            vs.append(_as_dtype(vb, w.dtype))
    if w.prefill:
        q = rng.standard_normal((B, n, w.n_q_heads, d), dtype=np.float32)
    else:
        q = rng.standard_normal((B, w.n_q_heads, d), dtype=np.float32)
    if w.outlier_in_q:
        g = w.group
        for h in range(w.n_q_heads):
            q[..., h, k_chan[h // g]] *= 20.0
    return DecodeInputs(lengths, np.stack(ks), np.stack(vs), _as_dtype(q, w.dtype), k_chan, v_chan)


def make_step_tokens(w: Workload, step: int, seed: int = 0):
    """K, V for the tokens appended at one decode step: [B][append][Hkv][d],
    with the workload's outlier channels, plus a fresh Q [B][Hq][d]."""
    rng = np.random.Generator(np.random.PCG64([seed, 1 + step]))
    base = np.random.Generator(np.random.PCG64(seed))
    k_chan = outlier_channels(base, w.n_kv_heads, w.head_dim, w.n_outliers)
    v_chan = outlier_channels(base, w.n_kv_heads, w.head_dim, w.n_outliers)
    n = max(1, w.append_per_step)
    k = rng.standard_normal((w.batch, n, w.n_kv_heads, w.head_dim), dtype=np.float32)
    v = rng.standard_normal((w.batch, n, w.n_kv_heads, w.head_dim), dtype=np.float32)
    _apply_outliers(k, k_chan)
    _apply_outliers(v, v_chan)
    q = rng.standard_normal((w.batch, w.n_q_heads, w.head_dim), dtype=np.float32)
    return _as_dtype(k, w.dtype), _as_dtype(v, w.dtype), _as_dtype(q, w.dtype)
