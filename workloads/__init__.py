"""Seeded synthetic inputs for the DSpark draft/verify hot path.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It only draws random numbers and shapes them into the workloads
below; it holds none of the method's arithmetic (no Markov bias, no Gumbel
noise, no acceptance test, no survival chain, no sort).  Random numbers that
the method itself draws (Gumbel noise, acceptance uniforms, resample
uniforms) are NOT produced here: both the CUDA path and the oracle derive
them from the counter-based Philox4x32-10 generator named by (seed, offset).

All generation runs on the host with numpy.  Large arrays are generated in
fixed-size row blocks, each block from its own generator seeded by
(seed, tensor tag, block index), so that the values do not depend on how
many threads generate them and any subset of rows can be regenerated alone.

Workloads (sizes follow the draft-step and verify descriptions of the pages
"DSpark implementation and evaluation" §2.2-§4 and "Speculative decoding:
from zero to DSpark" §2, §5-§7):

  tiny               B=1,    N=8,  H=256,  V=4096,   r=64,  fp32
  qwen3_8b_single    B=1,    N=8,  H=4096, V=151936, r=64,  bf16
  batched_draft      B=64,   N=16, H=4096, V=151936, r=256, bf16, T=0.8
  verify             B=256,  gamma=8,     V=151936,  fp32 probabilities
  verify (logits)    B=256,  gamma=8,     V=151936,  r=256, bf16 Markov weights,
                     fp32 target / draft base logits
  schedule           B=1024, N=16, SPS table over batch sizes 1..16384
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "DraftConfig", "VerifyConfig", "ScheduleConfig", "DRAFT_CONFIGS",
    "VERIFY_CONFIGS", "SCHEDULE_CONFIGS", "VerifyLogitsConfig", "VERIFY_LOGITS_CONFIGS",
    "verify_logits_inputs", "normal_rows", "draft_inputs",
    "markov_logits", "zipf_offsets", "verify_inputs", "schedule_inputs", "sps_table",
    "to_bf16_values",
]

_BLOCK_ROWS = 2048

# tensor tags used in the per-block seeds
_TAG = {"hidden": 1, "lm_head": 2, "w1": 3, "w2": 4, "anchor": 5,
        "spike_pos": 6, "base": 7, "zipf_perm": 8, "tgt": 9, "noise": 10,
        "sigma": 11, "draft_tok": 12, "mix": 13, "conf": 14, "temp": 15, "vl_len": 16}


@dataclass(frozen=True)
class DraftConfig:
    name: str
    B: int
    N: int
    H: int
    V: int
    r: int
    dtype: str                 # "f32" or "bf16": storage type of X, lm_head, w1, w2
    temperatures: tuple        # temperatures that are run (one value for all requests)
    data_seed: int
    philox_seed: int = 0
    spike: bool = False        # w1 rows get 8 coordinates multiplied by 4
    zipf: float = 0.0          # Zipf exponent of the per-row rank offset on base logits (0 = none)
    rms_norm_hidden: bool = False


@dataclass(frozen=True)
class VerifyConfig:
    name: str
    B: int
    gamma: int
    V: int
    target_std: float
    draft_sigmas: tuple        # per-request draft-noise std, drawn uniformly from this set
    independent_draft: bool    # draft logits drawn independently instead of target + noise
    data_seed: int
    draft_seed: int = 1        # seeds the categorical draw of the draft tokens from p_d
    verify_seed: int = 2       # Philox seed of the verification uniforms


@dataclass(frozen=True)
class VerifyLogitsConfig:
    name: str
    B: int
    gamma: int
    V: int
    r: int
    dtype: str                 # storage type of markov_w1 / markov_w2
    target_std: float
    draft_sigmas: tuple        # per-request std of the draft's deviation from the target logits
    draft_temps: tuple         # per-request draft temperature, drawn from this set (0 = greedy draft)
    target_temp: float
    data_seed: int
    spike: bool = True
    ragged_lengths: bool = False   # lengths drawn uniformly in [0, gamma] instead of all gamma
    draft_seed: int = 1
    verify_seed: int = 2


@dataclass(frozen=True)
class ScheduleConfig:
    name: str
    B: int
    N: int
    K_in: int                  # <0: choose K
    beta_mix: tuple            # (a, b) pairs, one drawn per request
    sps_len: int
    data_seed: int


DRAFT_CONFIGS = {
    "tiny": DraftConfig("tiny", B=1, N=8, H=256, V=4096, r=64, dtype="f32",
                        temperatures=(1.0,), data_seed=1000),
    "qwen3_8b_single": DraftConfig("qwen3_8b_single", B=1, N=8, H=4096, V=151936, r=64,
                                   dtype="bf16", temperatures=(0.0, 1.0), data_seed=2000,
                                   rms_norm_hidden=True),
    "batched_draft": DraftConfig("batched_draft", B=64, N=16, H=4096, V=151936, r=256,
                                 dtype="bf16", temperatures=(0.8,), data_seed=3000,
                                 spike=True, zipf=1.1, rms_norm_hidden=True),
}

VERIFY_CONFIGS = {
    "tiny": VerifyConfig("tiny", B=1, gamma=8, V=4096, target_std=2.0, draft_sigmas=(2.0,),
                         independent_draft=True, data_seed=1000),
    "verify": VerifyConfig("verify", B=256, gamma=8, V=151936, target_std=3.0,
                           draft_sigmas=(0.3, 1.0, 3.0), independent_draft=False,
                           data_seed=4000),
}

VERIFY_LOGITS_CONFIGS = {
    "verify": VerifyLogitsConfig("verify", B=256, gamma=8, V=151936, r=256, dtype="bf16", target_std=3.0,
                                 draft_sigmas=(0.3, 1.0, 3.0), draft_temps=(1.0,), target_temp=1.0,
                                 data_seed=4000),
}

SCHEDULE_CONFIGS = {
    "tiny": ScheduleConfig("tiny", B=1, N=8, K_in=6, beta_mix=((5, 2),), sps_len=8,
                           data_seed=1000),
    "schedule": ScheduleConfig("schedule", B=1024, N=16, K_in=-1,
                               beta_mix=((9, 1), (5, 2), (2, 3)), sps_len=16384,
                               data_seed=5000),
}


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_rows(rows: int, cols: int, std: float, seed: int, tag: str,
                row_start: int = 0, row_count: int | None = None) -> np.ndarray:
    """Rows [row_start, row_start+row_count) of a [rows, cols] N(0, std^2) float32 matrix.

    Block b of _BLOCK_ROWS rows always comes from default_rng((seed, tag, b)),
    so a sub-range reproduces exactly the rows of the full matrix.
    """
    if row_count is None:
        row_count = rows - row_start
    out = np.empty((row_count, cols), dtype=np.float32)
    b0 = row_start // _BLOCK_ROWS
    b1 = (row_start + row_count + _BLOCK_ROWS - 1) // _BLOCK_ROWS

    def work(b):
        lo, hi = b * _BLOCK_ROWS, min(rows, (b + 1) * _BLOCK_ROWS)
        rng = np.random.default_rng((seed, _TAG[tag], b))
        blk = rng.standard_normal((hi - lo, cols), dtype=np.float32)
        if std != 1.0:
            blk *= np.float32(std)
        s, e = max(lo, row_start), min(hi, row_start + row_count)
        if s < e:
            out[s - row_start:e - row_start] = blk[s - lo:e - lo]

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(b0, b1)))
    return out


def to_bf16_values(a: np.ndarray):
    """Round float32 values to bfloat16 (round to nearest even).

    Returns (torch bf16 tensor, float32 numpy array holding the exact bf16 values).
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)
    return t, t.float().numpy()


def _store(a: np.ndarray, dtype: str):
    """Return (torch CPU tensor in the storage dtype, float32 numpy array of its exact values)."""
    import torch
    if dtype == "bf16":
        return to_bf16_values(a)
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t, t.numpy()


def draft_inputs(cfg: DraftConfig, rows: slice | None = None):
    """Inputs of the draft step: hidden [B*N,H], lm_head [V,H], w1 [V,r], w2 [V,r], anchor [B].

    Readings (variance 1/fan_in): lm_head ~ N(0, 1/H); w2 ~ N(0, 1/r) (a bias-free
    r->V linear); w1 ~ N(0, 1) (an embedding, whose one-hot input has fan-in 1);
    hidden states ~ N(0, 1), optionally divided by their row RMS (no gain).
    With cfg.spike, each w1 row gets 8 distinct random coordinates multiplied by 4.
    Returns a dict of torch CPU tensors in storage dtype plus '<name>_f32' numpy
    arrays holding the exact stored values.
    """
    M = cfg.B * cfg.N
    s = cfg.data_seed
    X = normal_rows(M, cfg.H, 1.0, s, "hidden")
    if cfg.rms_norm_hidden:
        rms = np.sqrt(np.mean(X.astype(np.float64) ** 2, axis=1, keepdims=True))
        X = (X / rms).astype(np.float32)
    W = normal_rows(cfg.V, cfg.H, 1.0 / math.sqrt(cfg.H), s, "lm_head")
    out = draft_inputs_markov(cfg)
    for name, a in (("hidden", X), ("lm_head", W)):
        t, f = _store(a, cfg.dtype)
        out[name] = t
        out[name + "_f32"] = f
    return out


def markov_logits(cfg: DraftConfig, scale: float = 1.0) -> np.ndarray:
    """Synthetic base logits [B, N, V] float32 for the Markov sampler alone.

    N(0, scale^2) per element, plus (if cfg.zipf > 0) the per-(b, i) Zipf offset of
    ``zipf_offsets``.
    """
    B, N, V = cfg.B, cfg.N, cfg.V
    L = normal_rows(B * N, V, scale, cfg.data_seed, "base").reshape(B, N, V)
    if cfg.zipf > 0:
        L.reshape(B * N, V)[:] += zipf_offsets(cfg)
    return L


def zipf_offsets(cfg: DraftConfig, rows=None) -> np.ndarray:
    """Per-row Zipf rank offsets [len(rows), V] float32 (rows of the [B*N, V] logits, default all):
    entry v of row m is -zipf * ln(rank_m(v)), rank_m a seeded random permutation of 1..V for
    that row (row m's permutation depends only on (data_seed, m)), so that a few tokens of every
    row dominate as they do in real LM logits."""
    V = cfg.V
    rows = np.arange(cfg.B * cfg.N) if rows is None else np.asarray(rows)
    off = (-cfg.zipf * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    out = np.empty((len(rows), V), dtype=np.float32)

    def work(j):
        rng = np.random.default_rng((cfg.data_seed, _TAG["zipf_perm"], int(rows[j])))
        perm = rng.permutation(V)
        out[j, perm] = off

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(len(rows))))
    return out


def temperatures(cfg: DraftConfig, T: float) -> np.ndarray:
    return np.full(cfg.B, T, dtype=np.float32)


def _softmax_rows_f32(logits: np.ndarray) -> np.ndarray:
    """Row softmax computed in float64 and rounded to float32 (input shaping only)."""
    x = logits.astype(np.float64)
    x -= x.max(axis=-1, keepdims=True)
    np.exp(x, out=x)
    x /= x.sum(axis=-1, keepdims=True)
    return x.astype(np.float32)


def verify_inputs(cfg: VerifyConfig, B: int | None = None):
    """Inputs of verification: p_t [B, gamma+1, V], p_d [B, gamma, V] (float32 probabilities),
    draft tokens [B, gamma] drawn from p_d.

    Target logits ~ N(0, target_std^2).  Draft logits are target logits (first gamma
    positions) plus N(0, sigma_b^2) noise with sigma_b drawn per request from
    cfg.draft_sigmas, or independent N(0, target_std^2) draws if
    cfg.independent_draft.  Both are softmaxed per row (float64, rounded to float32).
    The draft token at each position is a categorical draw from that p_d row by
    inverse CDF with numpy's Philox bit generator seeded with cfg.draft_seed.
    """
    B = cfg.B if B is None else B
    g, V, s = cfg.gamma, cfg.V, cfg.data_seed
    tgt = normal_rows(B * (g + 1), V, cfg.target_std, s, "tgt").reshape(B, g + 1, V)
    sig_rng = np.random.default_rng((s, _TAG["sigma"]))
    sigma = np.asarray(cfg.draft_sigmas, dtype=np.float32)[
        sig_rng.integers(0, len(cfg.draft_sigmas), size=B)]
    if cfg.independent_draft:
        drf = normal_rows(B * g, V, cfg.target_std, s, "noise").reshape(B, g, V)
    else:
        drf = normal_rows(B * g, V, 1.0, s, "noise").reshape(B, g, V)
        drf *= sigma[:, None, None]
        drf += tgt[:, :g]
    p_t = np.empty_like(tgt)
    p_d = np.empty_like(drf)

    def work(b):
        p_t[b] = _softmax_rows_f32(tgt[b])
        p_d[b] = _softmax_rows_f32(drf[b])

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(B)))
    del tgt, drf
    rng = np.random.Generator(np.random.Philox(key=cfg.draft_seed))
    u = rng.random((B, g))
    tokens = np.empty((B, g), dtype=np.int32)
    for b in range(B):
        for k in range(g):
            cdf = np.cumsum(p_d[b, k], dtype=np.float64)
            v = int(np.searchsorted(cdf, u[b, k] * cdf[-1], side="right"))
            tokens[b, k] = min(v, V - 1)
    return {"p_t": p_t, "p_d": p_d, "draft_tokens": tokens, "sigma": sigma}


def verify_logits_inputs(cfg: VerifyLogitsConfig, B: int | None = None, V: int | None = None):
    """Inputs of verification from logits.

    target_logits [B, gamma+1, V] ~ N(0, target_std^2) (as ``verify_inputs``); the
    draft's base logits of the drafted positions are the target logits plus
    N(0, sigma_b^2) noise, sigma_b drawn per request from cfg.draft_sigmas; markov
    w1 / w2 [V, r] follow ``draft_inputs`` (w1 ~ N(0, 1) with 8 coordinates x4 per
    row if cfg.spike, w2 ~ N(0, 1/r)); anchors uniform; draft temperatures drawn per
    request from cfg.draft_temps; lengths all gamma or, with cfg.ragged_lengths,
    uniform in [0, gamma].  Draft tokens: for T_d > 0 a categorical draw from
    softmax(base_logits / T_d) (the Markov bias left out: input shaping only), for
    T_d = 0 the argmax of the base logits, with numpy's Philox generator seeded by
    cfg.draft_seed.
    Returns numpy arrays plus torch CPU tensors "w1" / "w2" in storage dtype
    ("w1_f32" / "w2_f32" hold their exact values).
    """
    B = cfg.B if B is None else B
    V = cfg.V if V is None else V
    g, s = cfg.gamma, cfg.data_seed
    tgt = normal_rows(B * (g + 1), V, cfg.target_std, s, "tgt").reshape(B, g + 1, V)
    sig_rng = np.random.default_rng((s, _TAG["sigma"]))
    sigma = np.asarray(cfg.draft_sigmas, dtype=np.float32)[sig_rng.integers(0, len(cfg.draft_sigmas), size=B)]
    base = normal_rows(B * g, V, 1.0, s, "noise").reshape(B, g, V)
    base *= sigma[:, None, None]
    base += tgt[:, :g]
    dc = DraftConfig("verify_logits", B=B, N=g, H=16, V=V, r=cfg.r, dtype=cfg.dtype, temperatures=(1.0,),
                     data_seed=s, spike=cfg.spike)
    w = draft_inputs_markov(dc)
    t_rng = np.random.default_rng((s, _TAG["temp"]))
    T_d = np.asarray(cfg.draft_temps, dtype=np.float32)[t_rng.integers(0, len(cfg.draft_temps), size=B)]
    T_t = np.full(B, cfg.target_temp, dtype=np.float32)
    if cfg.ragged_lengths:
        lengths = np.random.default_rng((s, _TAG["vl_len"])).integers(0, g + 1, size=B).astype(np.int32)
    else:
        lengths = None
    rng = np.random.Generator(np.random.Philox(key=cfg.draft_seed))
    u = rng.random((B, g))
    tokens = np.empty((B, g), dtype=np.int32)
    for b in range(B):
        for k in range(g):
            if T_d[b] == 0:
                tokens[b, k] = int(np.argmax(base[b, k]))
                continue
            p = _softmax_rows_f32(base[b, k] / np.float32(T_d[b]))
            cdf = np.cumsum(p, dtype=np.float64)
            tokens[b, k] = min(int(np.searchsorted(cdf, u[b, k] * cdf[-1], side="right")), V - 1)
    return {"target_logits": tgt, "base_logits": base, "anchor": w["anchor"], "w1": w["w1"], "w2": w["w2"],
            "w1_f32": w["w1_f32"], "w2_f32": w["w2_f32"], "T_t": T_t, "T_d": T_d, "lengths": lengths,
            "draft_tokens": tokens, "sigma": sigma}


def draft_inputs_markov(cfg: DraftConfig):
    """markov_w1, markov_w2 and the anchors of ``draft_inputs`` alone (no hidden states or LM head)."""
    s = cfg.data_seed
    w1 = normal_rows(cfg.V, cfg.r, 1.0, s, "w1")
    if cfg.spike:
        rng = np.random.default_rng((s, _TAG["spike_pos"]))
        keys = rng.random((cfg.V, cfg.r), dtype=np.float32)
        pos = np.argpartition(keys, 8, axis=1)[:, :8]
        np.multiply.at(w1, (np.arange(cfg.V)[:, None], pos), np.float32(4.0))
    w2 = normal_rows(cfg.V, cfg.r, 1.0 / math.sqrt(cfg.r), s, "w2")
    anchor = np.random.default_rng((s, _TAG["anchor"])).integers(
        0, cfg.V, size=cfg.B, dtype=np.int64).astype(np.int32)
    out = {"anchor": anchor}
    for name, a in (("w1", w1), ("w2", w2)):
        t, f = _store(a, cfg.dtype)
        out[name] = t
        out[name + "_f32"] = f
    return out


def sps_table(n: int) -> np.ndarray:
    """Synthetic steps-per-second curve over batch sizes 1..n (entry j is batch size j+1).

    Flat at 100 up to batch size 2048, then decaying as 100*2048/size, times a
    +-5% sawtooth that restarts every 128 batch sizes (the tile-boundary
    staircase of "Speculative decoding: from zero to DSpark" §7).
    """
    size = np.arange(1, n + 1, dtype=np.float64)
    base = np.where(size <= 2048, 100.0, 100.0 * 2048.0 / size)
    saw = 1.0 + 0.05 * (1.0 - 2.0 * ((size - 1) % 128) / 127.0)
    return base * saw


def schedule_inputs(cfg: ScheduleConfig, B: int | None = None):
    """Conditional acceptance probabilities c [B, N] (float32 in [0, 1]) and the SPS table."""
    B = cfg.B if B is None else B
    rng = np.random.default_rng((cfg.data_seed, _TAG["mix"]))
    mix = np.asarray(cfg.beta_mix, dtype=np.float64)[rng.integers(0, len(cfg.beta_mix), size=B)]
    crng = np.random.default_rng((cfg.data_seed, _TAG["conf"]))
    c = crng.beta(mix[:, 0:1], mix[:, 1:2], size=(B, cfg.N)).astype(np.float32)
    return {"cond_accept": c, "sps": sps_table(cfg.sps_len), "K_in": cfg.K_in}
