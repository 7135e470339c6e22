"""Seeded synthetic inputs for the Parallax attention layer.

This module only draws random numbers and rounds them to the storage type.  It
holds none of the layer's arithmetic: the oracle (under ``oracle/``) and the
CUDA library both consume what it returns, and neither shares any other code.

Workloads are synthetic stand-ins for the attention shapes of the 0.6B / 1.7B
Qwen-3-style models that "Parallax: Parameterized Local Linear Attention for
Language Modeling" pretrains at context 4096 (encorp.ai write-up, "Pretraining
gains").  No dataset, tokenizer or trained weight is involved.

Recipe (every array is drawn in float64 with ``numpy.random.default_rng(seed)``
(PCG64), then rounded to the storage dtype with round-to-nearest-even):

* draw order: q, k (including any key-covariance draws), v, P, dO, multipliers;
* q, k, v, dO ~ N(0, 1) unless the workload says otherwise;
* P_h ~ N(0, p_std^2) i.i.d. per head, stored float32, row-major, u = P_h @ delta;
* ``key_cov``: per head, Sigma_h = Q diag(lam) Q^T with Q Haar-orthogonal (QR of
  a Gaussian, column signs fixed by diag(R) > 0) and lam log-uniform in
  [0.1, 10]; k = z * sqrt(lam) @ Q^T with z ~ N(0, 1); P_h = 0.5 (Sigma_h + 0.1 I)^-1;
* ``norm_mult``: one multiplier per (b, t), shared over heads, log-uniform in
  [0.5, 2], drawn independently for q and for k and multiplied into the rows.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Workload", "WORKLOADS", "generate", "to_bf16_bits", "bf16_bits_to_f32",
           "widen", "causal_pairs"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dtype: str          # "fp32" or "bf16"
    seed: int
    p_std: float        # std of the i.i.d. Gaussian P_h entries (ignored with key_cov)
    backward: bool = False
    key_cov: bool = False
    norm_mult: bool = False
    describe: str = ""


WORKLOADS = {
    "pr1": Workload("pr1", 1, 2, 256, 64, "fp32", 0, 0.02,
                    describe="causal Parallax forward, fp32, B1 H2 T256 d64"),
    "c2": Workload("c2", 8, 16, 2048, 64, "bf16", 1, 0.1 / math.sqrt(64),
                   describe="causal Parallax forward, bf16, B8 H16 T2048 d64"),
    "c3": Workload("c3", 4, 16, 4096, 128, "bf16", 2, 0.0, key_cov=True,
                   describe="causal Parallax forward, bf16, B4 H16 T4096 d128, "
                            "correlated keys, P_h = 0.5 (Sigma_h + 0.1 I)^-1"),
    "c4": Workload("c4", 8, 16, 4096, 64, "bf16", 3, 0.1 / math.sqrt(64), backward=True,
                   describe="causal Parallax forward+backward, bf16, B8 H16 T4096 d64"),
    "c5": Workload("c5", 1, 16, 16384, 128, "bf16", 4, 0.1 / math.sqrt(128), norm_mult=True,
                   describe="long-context causal Parallax forward, bf16, B1 H16 T16384 d128"),
}


def causal_pairs(B: int, H: int, T: int) -> int:
    """Number of (query, key) pairs with key index <= query index."""
    return B * H * T * (T + 1) // 2


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64/float32 to bfloat16 (RNE) and return the raw uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    r = ((u + bias) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r[nan] = 0x7FC0
    return r.reshape(f.shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def widen(x: np.ndarray) -> np.ndarray:
    """Exact float64 copy of a stored array (uint16 = bfloat16 bits, else float)."""
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return to_bf16_bits(x)
    if dtype == "fp32":
        return x.astype(np.float32)
    raise ValueError(dtype)


def _haar_orthogonal(rng, d):
    g = rng.standard_normal((d, d))
    q, r = np.linalg.qr(g)
    return q * np.sign(np.diag(r))[None, :]


def generate(B: int, H: int, T: int, d: int, dtype: str = "bf16", seed: int = 0,
             p_std: float = 0.02, backward: bool = False, key_cov: bool = False,
             norm_mult: bool = False, zero_P: bool = False) -> dict:
    """Draw one seeded input set.  Tensors are [B, H, T, d]; P is [H, d, d] fp32.

    Returns a dict with q, k, v (and dout when ``backward``) in storage form
    (uint16 bf16 bits or float32) plus P (float32) and the shape fields.
    """
    rng = np.random.default_rng(seed)
    shape = (B, H, T, d)
    q = rng.standard_normal(shape)
    sigma = None
    if key_cov:
        sigma = np.empty((H, d, d))
        k = rng.standard_normal(shape)
        for h in range(H):
            Q = _haar_orthogonal(rng, d)
            lam = np.exp(rng.uniform(math.log(0.1), math.log(10.0), size=d))
            sigma[h] = (Q * lam[None, :]) @ Q.T
            k[:, h] = (k[:, h] * np.sqrt(lam)[None, None, :]) @ Q.T
    else:
        k = rng.standard_normal(shape)
    v = rng.standard_normal(shape)
    if key_cov:
        P = np.stack([0.5 * np.linalg.inv(sigma[h] + 0.1 * np.eye(d)) for h in range(H)])
    else:
        P = rng.standard_normal((H, d, d)) * p_std
    if zero_P:
        P = np.zeros_like(P)
    out = {"B": B, "H": H, "T": T, "d": d, "dtype": dtype, "seed": seed}
    if backward:
        out["dout"] = _store(rng.standard_normal(shape), dtype)
    if norm_mult:
        mq = np.exp(rng.uniform(math.log(0.5), math.log(2.0), size=(B, 1, T, 1)))
        mk = np.exp(rng.uniform(math.log(0.5), math.log(2.0), size=(B, 1, T, 1)))
        q = q * mq
        k = k * mk
    out["q"] = _store(q, dtype)
    out["k"] = _store(k, dtype)
    out["v"] = _store(v, dtype)
    out["P"] = P.astype(np.float32)
    return out


def generate_workload(name: str, **override) -> dict:
    w = WORKLOADS[name]
    kw = dict(B=w.B, H=w.H, T=w.T, d=w.d, dtype=w.dtype, seed=w.seed, p_std=w.p_std,
              backward=w.backward, key_cov=w.key_cov, norm_mult=w.norm_mult)
    kw.update(override)
    return generate(**kw)
