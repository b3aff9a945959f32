"""Seeded synthetic inputs for the delayed mHC seam.

This module only draws random numbers and lays them out in the shapes the seam
takes; it holds none of the seam's arithmetic.  The oracle and the CUDA path
both receive exactly the arrays built here.

Generator: a counter-based SplitMix64 stream per (seed, tensor id).  Output i
of stream s is ``mix64(key_s + (i + 1) * 0x9E3779B97F4A7C15)`` where ``mix64``
is the SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).  Uniforms take the top 53 bits;
normals use the Box-Muller transform in float64.  Everything is vectorised
numpy on uint64, so the same seed gives the same bits on x86 and Arm up to the
last-ulp behaviour of libm ``log``/``cos`` in Box-Muller.

Workload recipe (the mHC seam pages, all configurations): residual streams
``R[T,4,H]`` and sub-layer output ``Y[T,H]`` are bf16 draws of N(0,1);
the gate weight ``fn[4H,24]`` is fp32 N(0, 1/(4H)); ``gamma[H]`` is
bf16(1 + 0.1 N(0,1)); ``alpha = 1``, ``bias = 0``, ``eps = 1e-6``.  The carried
gates are built from U(-1,1) logits; turning those logits into
``sigmoid``/``2 sigmoid``/``Sinkhorn20(exp)`` form is left to the caller,
because it is the seam's own arithmetic.
"""
from __future__ import annotations

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Stream ids: one independent stream per tensor of a workload.
STREAM_R, STREAM_Y, STREAM_FN, STREAM_GAMMA = 1, 2, 3, 4
STREAM_PRE, STREAM_POST, STREAM_COMB = 5, 6, 7
STREAM_CRAFT = 8


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_bits(seed: int, stream: int, n: int) -> np.ndarray:
    """n raw 64-bit outputs of stream ``stream`` under ``seed``."""
    with np.errstate(over="ignore"):
        key = _mix64(np.array([(seed * 1_000_003 + stream) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
        ctr = np.arange(1, n + 1, dtype=np.uint64) * _GOLDEN + key
        return _mix64(ctr)


def uniform(seed: int, stream: int, n: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    """n float64 draws of U[lo, hi) from the top 53 bits of the stream."""
    u = (stream_bits(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return lo + (hi - lo) * u


def normal(seed: int, stream: int, n: int, std: float = 1.0) -> np.ndarray:
    """n float64 draws of N(0, std^2) by Box-Muller on pairs of uniforms."""
    m = (n + 1) // 2
    bits = stream_bits(seed, stream, 2 * m)
    u1 = ((bits[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)  # (0, 1]
    u2 = (bits[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.concatenate([r * np.cos(2.0 * np.pi * u2), r * np.sin(2.0 * np.pi * u2)])
    return std * z[:n]


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Store float64 draws as a bf16 tensor (torch's round-to-nearest-even cast)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.float32).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a bf16 tensor, as a numpy array."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


N_HC = 4
N_LOGITS = 24


def seam_draws(T: int, H: int, seed: int, post: bool = True, unique_tokens: int | None = None,
               token_offset: int = 0) -> dict:
    """All random inputs of one seam call (CPU tensors).

    Returns bf16 ``R [T,4,H]``, ``Y [T,H]`` (absent when ``post`` is False),
    fp32 ``fn [4H,24]``, ``bias [24]``, ``alpha [3]``, bf16 ``gamma [H]``, and
    float64 U(-1,1) logits ``pre_logits [T,4]``, ``post_logits [T,4]``,
    ``comb_logits [T,4,4]`` for the carried gates.

    ``unique_tokens``: draw only that many tokens and repeat them along T (the
    per-token inputs of token t are those of token t mod unique_tokens).  Large
    workloads use this to keep the CPU draw short; the device still streams
    every byte of the full T.  ``token_offset`` (with ``unique_tokens``): the
    T rows returned are rows token_offset .. token_offset + T - 1 of that
    repeated sequence, i.e. one shard of a larger batch.
    """
    if unique_tokens is not None and 0 < unique_tokens and (unique_tokens != T or token_offset):
        d = seam_draws(unique_tokens, H, seed, post=post)
        rows = (token_offset + np.arange(T, dtype=np.int64)) % unique_tokens
        idx = torch.from_numpy(rows)
        for k in ("R", "Y"):
            if d[k] is not None:
                d[k] = d[k][idx].contiguous()
        for k in ("pre_logits", "post_logits", "comb_logits"):
            d[k] = d[k][rows]
        d["T"] = T
        return d
    if token_offset:
        raise ValueError("token_offset needs unique_tokens")
    K = N_HC * H
    d = {
        "T": T,
        "H": H,
        "eps": 1e-6,
        "R": to_bf16(normal(seed, STREAM_R, T * N_HC * H)).reshape(T, N_HC, H),
        "fn": torch.from_numpy(normal(seed, STREAM_FN, K * N_LOGITS, std=(1.0 / K) ** 0.5)).to(torch.float32).reshape(K, N_LOGITS),
        "bias": torch.zeros(N_LOGITS, dtype=torch.float32),
        "alpha": torch.ones(3, dtype=torch.float32),
        "gamma": to_bf16(1.0 + 0.1 * normal(seed, STREAM_GAMMA, H)),
        "pre_logits": uniform(seed, STREAM_PRE, T * N_HC, -1.0, 1.0).reshape(T, N_HC),
        "post_logits": uniform(seed, STREAM_POST, T * N_HC, -1.0, 1.0).reshape(T, N_HC),
        "comb_logits": uniform(seed, STREAM_COMB, T * N_HC * N_HC, -1.0, 1.0).reshape(T, N_HC, N_HC),
    }
    d["Y"] = to_bf16(normal(seed, STREAM_Y, T * H)).reshape(T, H) if post else None
    return d


def _crafted_group(kind: int, k: int, u: np.ndarray) -> np.ndarray:
    """32 float64 values of one crafted quantiser group.

    kind 0: all zeros (signs mixed); 1: bf16 subnormals only; 2: amax exactly
    448 * 2^k with the rest below it; 3: amax just below 448 * 2^k (the bf16
    neighbour 446 * 2^k).  ``u`` is 32 uniforms in [0, 1) for the filler.
    """
    sign = np.where(u < 0.5, -1.0, 1.0)
    if kind == 0:
        return sign * 0.0
    if kind == 1:
        # bf16 subnormals are m * 2^-133 for m in 1..127
        return sign * np.floor(1.0 + u * 126.0) * 2.0 ** -133
    top = 448.0 * 2.0 ** k if kind == 2 else 446.0 * 2.0 ** k
    g = sign * top * (0.05 + 0.9 * u)
    g[int(u[0] * 32) % 32] = top
    return g


def craft_mxfp8(d: dict, seed: int, token_frac: float = 0.01, group_frac: float = 0.1) -> dict:
    """Plant crafted quantiser groups in a seam workload (in place; returns d).

    Reading of "1% of groups replaced by crafted edge groups" for the fused
    seam, where the quantiser sees the kernel's own norm: ``token_frac`` of the
    tokens get constant residual streams (R = 1, Y = 0), so their x is constant
    along H and x * rstd_x is 1 to within eps; their norm row is then gamma.
    ``group_frac`` of gamma's 32-groups are replaced by crafted groups (zeros,
    subnormals, amax = 448 * 2^k for k in [-20, 20], just below 448 * 2^k), so
    those tokens carry the crafted groups exactly and every other token carries
    scaled versions of them.
    """
    T, H = d["T"], d["H"]
    n_groups = H // 32
    n_rows = max(1, int(round(token_frac * T))) if T > 0 else 0
    n_g = max(1, int(round(group_frac * n_groups)))
    bits = stream_bits(seed, STREAM_CRAFT, n_rows + 3 * n_g)
    rows = np.unique((bits[:n_rows] % np.uint64(max(T, 1))).astype(np.int64)) if T > 0 else np.zeros(0, np.int64)
    groups = np.unique((bits[n_rows:n_rows + n_g] % np.uint64(n_groups)).astype(np.int64))
    kinds = (bits[n_rows + n_g:n_rows + 2 * n_g] % np.uint64(4)).astype(np.int64)
    ks = (bits[n_rows + 2 * n_g:n_rows + 3 * n_g] % np.uint64(41)).astype(np.int64) - 20
    fill = uniform(seed, STREAM_CRAFT + 100, 32 * len(groups)).reshape(len(groups), 32)
    gamma = d["gamma"].to(torch.float64).numpy().copy()
    for j, g in enumerate(groups):
        gamma[32 * g:32 * g + 32] = _crafted_group(int(kinds[j]), int(ks[j]), fill[j])
    d["gamma"] = to_bf16(gamma)
    if len(rows):
        R = d["R"].clone()
        R[torch.from_numpy(rows)] = 1.0
        d["R"] = R
        if d.get("Y") is not None:
            Y = d["Y"].clone()
            Y[torch.from_numpy(rows)] = 0.0
            d["Y"] = Y
    d["crafted_rows"] = rows
    d["crafted_groups"] = groups
    return d


def crafted_quant_tensor(rows: int, H: int, seed: int, frac: float = 0.01) -> tuple[torch.Tensor, np.ndarray]:
    """A bf16 [rows, H] tensor of N(0,1) draws with ``frac`` of its 32-groups
    replaced by crafted groups; returns the tensor and the flat indices of the
    crafted groups."""
    n_groups = rows * (H // 32)
    x = normal(seed, STREAM_R, rows * H).reshape(n_groups, 32)
    n_c = max(1, int(round(frac * n_groups)))
    bits = stream_bits(seed, STREAM_CRAFT, 3 * n_c)
    pick = np.unique((bits[:n_c] % np.uint64(n_groups)).astype(np.int64))
    kinds = (bits[n_c:2 * n_c] % np.uint64(4)).astype(np.int64)
    ks = (bits[2 * n_c:3 * n_c] % np.uint64(41)).astype(np.int64) - 20
    fill = uniform(seed, STREAM_CRAFT + 200, 32 * len(pick)).reshape(len(pick), 32)
    for j, g in enumerate(pick):
        x[g] = _crafted_group(int(kinds[j]), int(ks[j]), fill[j])
    return to_bf16(x.reshape(rows, H)), pick
