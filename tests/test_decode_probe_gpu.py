"""GPU parity of the given-probe decode step (parallax_decode_probe) against the fp64 oracle.

A decode step for sequence b is the given-probe layer's row lens[b] - 1 with
the caches as keys and values ("Parallax: Parameterized Local Linear Attention
for Language Modeling", technical summary, "Core mechanism": o = o^SA -
Sigma_KV rho).  The query and its probe go into row lens[b] - 1 of otherwise
unused query and probe arrays, and the oracle computes only those rows.
"""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import TOL_BF16, inputs_f64, rel_err, to_device, to_host64

pytestmark = pytest.mark.gpu


def _case(B, H, L, d, lens, seed, rho_scale=0.3, nan_tail=False, zero_rho=False):
    inp = plx_synth.generate(B, H, L, d, "bf16", seed=seed, p_std=0.3 / np.sqrt(d))
    eff = np.full(B, L) if lens is None else np.asarray(lens)
    if nan_tail:
        for b, n in enumerate(eff):
            inp["k"][b, :, n:] = 0x7FC0  # bf16 NaN: rows past the sequence must not be read
            inp["v"][b, :, n:] = 0x7FC0
    rng = np.random.default_rng(seed + 1)
    qn = plx_synth.to_bf16_bits(rng.standard_normal((B, H, d)))
    rn = plx_synth.to_bf16_bits((0.0 if zero_rho else rho_scale) * rng.standard_normal((B, H, d)))
    f = inputs_f64(inp)
    kk = np.nan_to_num(f["k"], nan=0.0)
    vv = np.nan_to_num(f["v"], nan=0.0)
    qfull = np.zeros((B, H, L, d))
    rfull = np.zeros((B, H, L, d))
    rows = []
    for b in range(B):
        for h in range(H):
            qfull[b, h, eff[b] - 1] = plx_synth.bf16_bits_to_f32(qn[b, h])
            rfull[b, h, eff[b] - 1] = plx_synth.bf16_bits_to_f32(rn[b, h])
            rows.append((b, h, int(eff[b]) - 1))
    ro, rl = oracle.forward_probe_rows(qfull, kk, vv, rfull, rows)
    q, rho = to_device(qn), to_device(rn)
    k, v = to_device(inp["k"]), to_device(inp["v"])
    lens_t = None if lens is None else torch.tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    out, lse = plx.parallax_decode_probe(q, k, v, rho, lens=lens_t)
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    return to_host64(out).reshape(-1, d), to_host64(lse).reshape(-1), ro, rl, inp, q, lens_t


def _check(go, gl, ro, rl):
    assert np.isfinite(go).all()
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))


@pytest.mark.parametrize("d", [64, 128])
def test_decode_probe_ragged_lengths(d):
    lens = [1, 128, 129, 300, 257]  # a single key, tile edges, the full cache, a ragged tail
    go, gl, ro, rl, *_ = _case(5, 2, 300, d, lens, seed=140 + d)
    _check(go, gl, ro, rl)


def test_decode_probe_many_tiles_per_chunk_d128():
    # B4 H16 with a 4096-key cache at d = 128: each head's keys split into a
    # few chunks of many tiles (the stage ring wraps many times per chunk) and
    # the merge combines several chunks; ragged lengths end chunks inside tiles
    go, gl, ro, rl, *_ = _case(4, 16, 4096, 128, [4096, 1, 2047, 3001], seed=177)
    _check(go, gl, ro, rl)


def test_decode_probe_full_size_c4_cache():
    # the B8 H16 T4096 d64 workload's cache, every sequence full length
    go, gl, ro, rl, *_ = _case(8, 16, 4096, 64, None, seed=178)
    _check(go, gl, ro, rl)


def test_decode_probe_nan_rows_past_the_lengths_are_ignored():
    go, gl, ro, rl, *_ = _case(3, 2, 500, 64, [37, 500, 129], seed=188, nan_tail=True)
    _check(go, gl, ro, rl)


def test_decode_probe_zero_probe_is_softmax_attention():
    # rho = 0: the correction vanishes, o = mu_v, as the committed-probe decode
    # with a zero projector gives
    B, H, L, d = 4, 3, 700, 64
    go, gl, ro, rl, inp, q, lens_t = _case(B, H, L, d, [700, 1, 350, 64], seed=190, zero_rho=True)
    _check(go, gl, ro, rl)
    k, v = to_device(inp["k"]), to_device(inp["v"])
    P0 = torch.zeros((H, d, d), dtype=torch.float32, device="cuda")
    out0, lse0 = plx.parallax_decode(q, k, v, P0, lens=lens_t)
    assert rel_err(go, to_host64(out0).reshape(-1, d), "bf16") < TOL_BF16
    assert np.abs(gl - to_host64(lse0).reshape(-1)).max() < 1e-4


def test_decode_probe_ctas_span_several_heads():
    # short caches and many heads: the tiles of all heads split over the CTAs
    # put several heads in one CTA's range, so partials start and end inside a
    # CTA, some heads' ranges hold tiles past their length (empty partials),
    # and a head's partials come from CTAs that also serve other heads
    B, H, L = 128, 16, 32
    lens = [1 + (13 * b) % L for b in range(B)]
    go, gl, ro, rl, *_ = _case(B, H, L, 64, lens, seed=211)
    _check(go, gl, ro, rl)
    B, H, L = 32, 16, 100  # two tiles per head: a CTA range may end between them
    lens = [(1, 64, 65, 100)[b % 4] for b in range(B)]
    go, gl, ro, rl, *_ = _case(B, H, L, 64, lens, seed=212)
    _check(go, gl, ro, rl)


def test_decode_probe_one_key_one_head():
    go, gl, ro, rl, *_ = _case(1, 1, 1, 64, None, seed=213)
    _check(go, gl, ro, rl)
    go, gl, ro, rl, *_ = _case(1, 1, 1, 128, None, seed=214)
    _check(go, gl, ro, rl)
