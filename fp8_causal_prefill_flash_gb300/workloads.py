"""Seeded synthetic inputs for causal prefill attention.

This module only draws random numbers and encodes them into the input formats
(per-tensor e4m3 with an fp32 descale, or bf16).  It holds none of the
attention arithmetic and serves the CUDA path, the oracle and the benchmark
alike.

The shapes and value distributions follow the workloads the articles measure
("How fast is ZYFA?": Gaussian inputs at 32K tokens, head dim 128, and the
DeepSeek-style MLA shape QK 192 / V 128).  Captured model activations are not
available, so Gaussian inputs with a few scaled "outlier" channels stand in
for them.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass
class Fp8Case:
    """One FP8 problem: e4m3 codes (uint8, BSHD) and fp32 per-tensor descales."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dq: float
    dk: float
    dv: float

    @property
    def shape(self):
        B, S, Hq, Dqk = self.q.shape
        return B, Hq, self.k.shape[2], S, Dqk, self.v.shape[3]


@dataclasses.dataclass
class Bf16Case:
    """One BF16 problem: bf16 bit patterns (uint16, BSHD)."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray

    @property
    def shape(self):
        B, S, Hq, Dqk = self.q.shape
        return B, Hq, self.k.shape[2], S, Dqk, self.v.shape[3]


def gaussian(shape, seed: int) -> np.ndarray:
    """Standard normal fp32 array from numpy's PCG64 stream for ``seed``."""
    return np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)


def quantize_e4m3(x: np.ndarray) -> tuple[np.ndarray, float]:
    """Per-tensor e4m3 quantisation: descale = amax/448 (1 when amax = 0).

    Encoding uses torch's float8_e4m3fn conversion (round to nearest even) after
    clamping to +-448.  Returns (uint8 codes, descale).
    """
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    descale = amax / E4M3_MAX if amax > 0.0 else 1.0
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = torch.clamp(t / np.float32(descale), -E4M3_MAX, E4M3_MAX)
    codes = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, float(np.float32(descale))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even, torch conversion) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def fp8_gaussian_case(B, Hq, Hkv, S, Dqk, Dv, seeds=(0, 1, 2), outlier_seed: Optional[int] = None,
                      outliers_qk: int = 0, outliers_v: bool = True, factor: float = 1.0,
                      shared_qkv_channels: bool = True) -> Fp8Case:
    """Gaussian Q, K, V with optional scaled channels, quantised per tensor.

    ``outliers_qk`` channels per kv head (chosen from ``outlier_seed``) are
    multiplied by ``factor`` in K and in the Q heads of that kv head's group;
    when ``outliers_v`` the same channels of V are scaled too (only where
    Dv == Dqk).
    """
    q = gaussian((B, S, Hq, Dqk), seeds[0])
    k = gaussian((B, S, Hkv, Dqk), seeds[1])
    v = gaussian((B, S, Hkv, Dv), seeds[2])
    if outliers_qk:
        rng = np.random.default_rng(outlier_seed)
        group = Hq // Hkv
        for g in range(Hkv):
            ch = rng.choice(Dqk, size=outliers_qk, replace=False)
            k[:, :, g, ch] *= factor
            q[:, :, g * group:(g + 1) * group, ch] *= factor
            if outliers_v and Dv == Dqk:
                v[:, :, g, ch] *= factor
    qc, dq = quantize_e4m3(q)
    del q
    kc, dk = quantize_e4m3(k)
    del k
    vc, dv = quantize_e4m3(v)
    return Fp8Case(qc, kc, vc, dq, dk, dv)


def fp8_sink_case(B, Hq, Hkv, S, Dqk, Dv, seeds=(50, 51, 52), sink_logits=(15.0, 25.0),
                  v_mean=1.0, sink_channel=0, scale=None) -> Fp8Case:
    """Gaussian Q, K, V plus an attention sink: key 0 of every kv head gets a
    large value in one channel, and every query row a per-row weight in that
    channel, so that row i's logit for key 0 exceeds the others by a value
    drawn uniformly from ``sink_logits`` (natural-log units, softmax scale
    ``scale``, default 1/sqrt(Dqk)).  The row maxima thus differ row by row
    and dwarf the rest of the row; V has mean ``v_mean``."""
    scale = 1.0 / np.sqrt(Dqk) if scale is None else scale
    q = gaussian((B, S, Hq, Dqk), seeds[0])
    k = gaussian((B, S, Hkv, Dqk), seeds[1])
    v = gaussian((B, S, Hkv, Dv), seeds[2]) + np.float32(v_mean)
    rng = np.random.default_rng(seeds[0] + 1000)
    amp = np.float32(32.0)
    k[:, 0, :, sink_channel] = amp
    target = rng.uniform(sink_logits[0], sink_logits[1], size=(B, S, Hq)).astype(np.float32)
    q[:, :, :, sink_channel] = target / np.float32(scale * amp)
    qc, dq = quantize_e4m3(q)
    del q
    kc, dk = quantize_e4m3(k)
    del k
    vc, dv = quantize_e4m3(v)
    return Fp8Case(qc, kc, vc, dq, dk, dv)


def bf16_gaussian_case(B, Hq, Hkv, S, Dqk, Dv, seeds=(20, 21, 22)) -> Bf16Case:
    """Gaussian Q, K, V rounded to bf16."""
    return Bf16Case(to_bf16_bits(gaussian((B, S, Hq, Dqk), seeds[0])),
                    to_bf16_bits(gaussian((B, S, Hkv, Dqk), seeds[1])),
                    to_bf16_bits(gaussian((B, S, Hkv, Dv), seeds[2])))


#: The measured configurations, by name.  ``kind`` selects the generator and path.
CONFIGS = {
    "fp8_h2_s256_d128": dict(kind="fp8", B=1, Hq=2, Hkv=2, S=256, Dqk=128, Dv=128,
                             seeds=(0, 1, 2)),
    "fp8_gqa_h32_8_s16k_d128_outliers": dict(kind="fp8", B=1, Hq=32, Hkv=8, S=16384, Dqk=128,
                                             Dv=128, seeds=(10, 11, 12), outlier_seed=13,
                                             outliers_qk=1, factor=8.0),
    "bf16_gqa_h32_8_s16k_d128": dict(kind="bf16", B=1, Hq=32, Hkv=8, S=16384, Dqk=128, Dv=128,
                                     seeds=(20, 21, 22)),
    "fp8_h32_s32k_d128": dict(kind="fp8", B=1, Hq=32, Hkv=32, S=32768, Dqk=128, Dv=128,
                              seeds=(30, 31, 32)),
    "fp8_mla_h16_s32k_dqk192_dv128_outliers": dict(kind="fp8", B=1, Hq=16, Hkv=16, S=32768,
                                                   Dqk=192, Dv=128, seeds=(40, 41, 42),
                                                   outlier_seed=43, outliers_qk=4, factor=20.0,
                                                   outliers_v=False),
    # few heads: one tensor-parallel shard of a larger model (fewer work items than SMs)
    "fp8_h4_s8k_d128": dict(kind="fp8", B=1, Hq=4, Hkv=4, S=8192, Dqk=128, Dv=128,
                            seeds=(60, 61, 62)),
    "bf16_h4_s8k_d128": dict(kind="bf16", B=1, Hq=4, Hkv=4, S=8192, Dqk=128, Dv=128,
                             seeds=(63, 64, 65)),
    # stress input: an attention sink at key 0 (+15..25 nats, varying per row), V mean 1
    "fp8_sink_h8_s8k_d128": dict(kind="fp8_sink", B=1, Hq=8, Hkv=8, S=8192, Dqk=128, Dv=128,
                                 seeds=(50, 51, 52)),
}


def make_case(name: str, S: Optional[int] = None, **overrides):
    """Build the named configuration (optionally with another S or shape)."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    if S is not None:
        cfg["S"] = S
    kind = cfg.pop("kind")
    if kind == "fp8_sink":
        return fp8_sink_case(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["Dqk"], cfg["Dv"],
                             seeds=cfg["seeds"])
    if kind == "bf16":
        return bf16_gaussian_case(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["Dqk"],
                                  cfg["Dv"], seeds=cfg["seeds"])
    return fp8_gaussian_case(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["S"], cfg["Dqk"], cfg["Dv"],
                             seeds=cfg["seeds"], outlier_seed=cfg.get("outlier_seed"),
                             outliers_qk=cfg.get("outliers_qk", 0),
                             outliers_v=cfg.get("outliers_v", True),
                             factor=cfg.get("factor", 1.0))


def stratified_rows(B: int, Hq: int, S: int, short: int = 512, n_long: int = 2048,
                    seed: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Rows (b, h, i) and weights for estimating a whole-output error sum.

    Causal rows with few keys have large outputs (row 0 is one value row;
    row i has about |v| / sqrt(i)), so a few hundred short rows hold about
    half of the output's sum of squares on long sequences, and a uniform
    sample of rows rarely contains them.  This sample takes every row
    i < ``short`` of every (b, h) with weight 1, and ``n_long`` rows drawn
    uniformly from the others with weight (number of other rows) / n_long,
    so that sum_r w_r f(row r) estimates the sum of f over all B*Hq*S rows.
    """
    short = min(short, S)
    b, h, i = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(short), indexing="ij")
    rows = [np.stack([b.ravel(), h.ravel(), i.ravel()], 1)]
    weights = [np.ones(B * Hq * short)]
    if S > short and n_long > 0:
        rng = np.random.default_rng(seed)
        rows.append(np.stack([rng.integers(0, B, n_long), rng.integers(0, Hq, n_long),
                              rng.integers(short, S, n_long)], 1))
        weights.append(np.full(n_long, B * Hq * (S - short) / n_long))
    return np.concatenate(rows).astype(np.int64), np.concatenate(weights)
