"""GPU parity of the one-pass given-probe forward (parallax_fwd_probe)
against the fp64 oracle's statement o = o^SA - Sigma_KV rho."""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import TOL_BF16, rel_err, to_device, to_host64

pytestmark = pytest.mark.gpu


def _probe_inputs(B, H, T, d, seed, rho_std):
    inp = plx_synth.generate(B, H, T, d, "bf16", seed=seed, p_std=0.0)
    rng = np.random.default_rng(seed + 1000)
    rho_bits = plx_synth.to_bf16_bits(rho_std * rng.standard_normal((B, H, T, d)))
    f = {x: plx_synth.widen(inp[x]) for x in ("q", "k", "v")}
    f["rho"] = plx_synth.widen(rho_bits)
    dev = {x: to_device(inp[x]) for x in ("q", "k", "v")}
    dev["rho"] = to_device(rho_bits)
    return f, dev


def _check(f, dev):
    ro, rl = oracle.forward_probe(f["q"], f["k"], f["v"], f["rho"])
    out, lse = plx.parallax_fwd_probe(dev["q"], dev["k"], dev["v"], dev["rho"])
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    go, gl = to_host64(out), to_host64(lse)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, float(np.sqrt(np.mean(rl * rl))))
    assert np.isfinite(go).all()


@pytest.mark.parametrize("B,H,T,d", [(1, 1, 1, 64), (1, 2, 7, 128), (2, 2, 130, 64), (1, 3, 300, 128),
                                     (2, 1, 513, 64)])
def test_probe_small_full_compare(B, H, T, d):
    f, dev = _probe_inputs(B, H, T, d, seed=T + d, rho_std=0.3 / np.sqrt(d))
    _check(f, dev)


def test_probe_zero_is_softmax_attention():
    f, dev = _probe_inputs(2, 2, 200, 64, seed=3, rho_std=0.0)
    _check(f, dev)
    out, _ = plx.parallax_fwd_probe(dev["q"], dev["k"], dev["v"], dev["rho"])
    sd = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(f["q"]), torch.from_numpy(f["k"]), torch.from_numpy(f["v"]), is_causal=True).numpy()
    assert rel_err(to_host64(out), sd, "bf16") < TOL_BF16


def test_probe_long_rows_d128():
    # one head at T = 2048, d = 128: many key tiles, lazy rescales of both accumulators
    f, dev = _probe_inputs(1, 1, 2048, 128, seed=9, rho_std=0.1 / np.sqrt(128))
    _check(f, dev)


def test_probe_fp32_is_unsupported():
    x = torch.zeros(1, 1, 16, 64, device="cuda")
    with pytest.raises(plx.PlxError) as e:
        plx.parallax_fwd_probe(x, x, x, x)
    assert e.value.code == plx.PLX_ERR_UNSUPPORTED
