"""GPU parity of the decode step (parallax_decode) against the fp64 oracle.

A decode step for sequence b is the layer's row lens[b] - 1 with the caches
as keys and values, so the oracle is the (pinned) forward evaluated at exactly
those rows: the query goes into row lens[b] - 1 of an otherwise unused query
array, and the oracle computes only the requested rows.
"""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import TOL_BF16, TOL_FP32, inputs_f64, rel_err, to_device, to_host64

pytestmark = pytest.mark.gpu


def _case(B, H, L, d, dtype, lens, seed):
    inp = plx_synth.generate(B, H, L, d, dtype, seed=seed, p_std=0.3 / np.sqrt(d))
    rng = np.random.default_rng(seed + 1)
    # the new queries: one per (b, h), drawn like q and rounded to the storage type
    qn = rng.standard_normal((B, H, d))
    if dtype == "bf16":
        qn_store = plx_synth.to_bf16_bits(qn)
        qn64 = plx_synth.bf16_bits_to_f32(qn_store).astype(np.float64)
    else:
        qn_store = qn.astype(np.float32)
        qn64 = qn_store.astype(np.float64)
    eff = np.full(B, L) if lens is None else np.asarray(lens)
    f = inputs_f64(inp)
    qfull = np.zeros((B, H, L, d))
    rows = []
    for b in range(B):
        for h in range(H):
            qfull[b, h, eff[b] - 1] = qn64[b, h]
            rows.append((b, h, int(eff[b]) - 1))
    ro, rl, _ = oracle.forward_rows(qfull, f["k"], f["v"], f["P"], rows)
    q = to_device(qn_store)
    k, v, P = (to_device(inp[x]) for x in ("k", "v", "P"))
    lens_t = None if lens is None else torch.tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    out, lse = plx.parallax_decode(q, k, v, P, lens=lens_t)
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    return to_host64(out).reshape(-1, d), to_host64(lse).reshape(-1), ro, rl


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_ragged_lengths(d, dtype):
    B, H, L = 5, 2, 300
    lens = [1, 128, 129, 300, 257]  # a single key, chunk edges, the full cache, a ragged tail
    go, gl, ro, rl = _case(B, H, L, d, dtype, lens, seed=40 + d)
    tol = TOL_FP32 if dtype == "fp32" else TOL_BF16
    assert rel_err(go, ro, dtype) < tol
    assert np.abs(gl - rl).max() < tol * max(1.0, float(np.sqrt(np.mean(rl * rl))))
    # lens[b] = 1: the output is that sequence's first value row
    assert np.isfinite(go).all()


@pytest.mark.parametrize("d", [64, 128])
def test_decode_lengths_across_key_blocks(d):
    # a cache of 1100 keys spans several key blocks per head, so some blocks
    # lie wholly past a short sequence and others end one key into a block
    B, H, L = 5, 2, 1100
    lens = [1, 513, 1100, 600, 257]
    go, gl, ro, rl = _case(B, H, L, d, "bf16", lens, seed=60 + d)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))


def test_decode_without_lengths_uses_the_whole_cache():
    go, gl, ro, rl = _case(2, 3, 200, 64, "bf16", None, seed=7)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))


def test_decode_full_size_c4_cache():
    # one new query per head over the B8 H16 T4096 d64 workload's keys and values
    w = plx_synth.WORKLOADS["c4"]
    go, gl, ro, rl = _case(w.B, w.H, w.T, w.d, "bf16", None, seed=w.seed)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))


def test_decode_invalid_arguments():
    q = torch.zeros(1, 1, 48, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(1, 1, 16, 48, device="cuda", dtype=torch.bfloat16)
    P = torch.zeros(1, 48, 48, device="cuda")
    with pytest.raises(plx.PlxError) as e:
        plx.parallax_decode(q, kc, kc, P)
    assert e.value.code == plx.PLX_ERR_UNSUPPORTED
    assert plx.parallax_last_device_error()[0] == plx.PLX_OK


def test_decode_full_size_d128_many_tiles_per_chunk():
    # B4 H16 with a 4096-key cache at d = 128 (the B4 H16 T4096 d128 forward's
    # shape): each head's keys split into a few chunks of many 64-key tiles,
    # so the stage ring wraps many times per chunk and the merge combines
    # several chunks; ragged lengths put chunk ends inside tiles
    B, H, L, d = 4, 16, 4096, 128
    lens = [4096, 1, 2047, 3001]
    go, gl, ro, rl = _case(B, H, L, d, "bf16", lens, seed=77)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))


def test_decode_nan_rows_past_the_lengths_are_ignored():
    # cache rows past lens[b] are not part of the sequence: even NaN there
    # must not reach the output
    B, H, L, d = 3, 2, 500, 64
    inp = plx_synth.generate(B, H, L, d, "bf16", seed=88, p_std=0.3 / np.sqrt(d))
    lens = [37, 500, 129]
    for b_, n in enumerate(lens):
        inp["k"][b_, :, n:] = 0x7FC0  # bf16 NaN
        inp["v"][b_, :, n:] = 0x7FC0
    rng = np.random.default_rng(89)
    qn_store = plx_synth.to_bf16_bits(rng.standard_normal((B, H, d)))
    f = inputs_f64(inp)
    qfull = np.zeros((B, H, L, d))
    rows = []
    for b_ in range(B):
        for h in range(H):
            qfull[b_, h, lens[b_] - 1] = plx_synth.bf16_bits_to_f32(qn_store[b_, h]).astype(np.float64)
            rows.append((b_, h, lens[b_] - 1))
    kk = np.nan_to_num(f["k"], nan=0.0)
    vv = np.nan_to_num(f["v"], nan=0.0)
    ro, rl, _ = oracle.forward_rows(qfull, kk, vv, f["P"], rows)
    q = to_device(qn_store)
    k, v, P = (to_device(inp[x]) for x in ("k", "v", "P"))
    out, lse = plx.parallax_decode(q, k, v, P, lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert plx.parallax_last_device_error()[0] == plx.PLX_OK
    go = to_host64(out).reshape(-1, d)
    assert np.isfinite(go).all()
    assert rel_err(go, ro, "bf16") < TOL_BF16


@pytest.mark.parametrize("d", [64, 128])
def test_decode_ctas_span_several_heads(d):
    # short caches and many heads: the tiles of all heads split over one wave
    # of CTAs put several heads in one CTA's range, so a CTA ends one head's
    # partial (M read out of TMEM, M started afresh) and begins the next inside
    # its range; ragged lengths leave some heads' tiles in a range empty
    B, H, L = 64, 16, 64 if d == 64 else 32
    lens = [1 + (11 * b) % L for b in range(B)]
    go, gl, ro, rl = _case(B, H, L, d, "bf16", lens, seed=230 + d)
    assert np.isfinite(go).all()
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))
    # two tiles per head: a CTA's range may end between a head's tiles
    B, H, L = 24, 16, 128 if d == 64 else 64
    lens = [(1, L // 2, L // 2 + 1, L)[b % 4] for b in range(B)]
    go, gl, ro, rl = _case(B, H, L, d, "bf16", lens, seed=240 + d)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))
