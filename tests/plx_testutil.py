"""Shared helpers for the parity tests (no layer arithmetic here)."""
import numpy as np
import torch

import plx_synth

# Tolerances: max |gpu - oracle| / RMS(oracle), per output tensor.
TOL_FP32 = 1e-4
TOL_BF16 = 2e-2
TOL_BF16_GRAD = 3e-2

# Largest relative error of rounding a real number to the storage type with
# round-to-nearest-even (half an ulp): 2^-8 for bfloat16 (8 significant bits),
# 2^-24 for float32.  The tolerance charges the arithmetic of the path, not
# this unavoidable rounding of a stored result: the first rows of causal
# attention see one or two keys, so |o| there is many times RMS(o) and the
# bf16 rounding of those rows alone exceeds 2e-2 * RMS.
STORAGE_REL = {"bf16": 2.0 ** -8, "fp32": 2.0 ** -24}


def rel_err(got, ref, storage: str = "fp32", roundings: int = 1) -> float:
    """max_i max(0, |got_i - ref_i| - n u |ref_i|) / RMS(ref), u = STORAGE_REL[storage].

    ``roundings`` (n) is how many of the two sides were rounded to the storage
    type: 1 against the fp64 oracle, 2 when both sides are stored results.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.maximum(0.0, np.abs(got - ref) - roundings * STORAGE_REL[storage] * np.abs(ref))
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        return float(err.max())
    return float(err.max() / rms)


def to_device(x: np.ndarray, device="cuda") -> torch.Tensor:
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def to_host64(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def inputs_f64(inp: dict):
    """Exact float64 views of the stored inputs (bf16 widened exactly)."""
    out = {k: plx_synth.widen(inp[k]) for k in ("q", "k", "v") if k in inp}
    out["P"] = inp["P"].astype(np.float64)
    if "dout" in inp:
        out["dout"] = plx_synth.widen(inp["dout"])
    return out


def sample_rows(B, H, T, n, seed=0):
    """Sampled (b, h, t) rows: always the first and last query plus tile edges."""
    rng = np.random.default_rng(seed)
    rows = set()
    for t in (0, 1, T - 1, min(T - 1, 127), min(T - 1, 128), T // 2):
        rows.add((int(rng.integers(B)), int(rng.integers(H)), t))
    while len(rows) < n:
        rows.add((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(T))))
    return sorted(rows)


# Guard bands: an output is a view into a larger buffer whose leading and
# trailing GUARD elements hold a sentinel; a kernel that stores past either end
# of its output (a row past T, a ragged tail) changes a sentinel.  The sentinel
# is finite and exactly representable in bf16 and fp32, so a stray store of
# NaN, inf or any ordinary value is caught.
GUARD = 256
SENTINEL = -12288.0


def guarded_empty(shape, dtype, device="cuda"):
    """(buffer, view): `view` has `shape`, starts 16-byte aligned, and is
    surrounded by GUARD sentinel elements on each side; its own elements are
    NaN until written."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=dtype, device=device)
    view = buf[GUARD:GUARD + n].view(shape)
    view.fill_(float("nan"))
    return buf, view


def guards_intact(buf, shape) -> bool:
    n = int(np.prod(shape))
    band = torch.cat([buf[:GUARD], buf[GUARD + n:]])
    return bool((band == SENTINEL).all())
