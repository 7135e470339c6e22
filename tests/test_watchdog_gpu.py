"""Failure detection on the GPU without a fault: the bounded-wait watchdog.

Every mbarrier wait in the tensor-core kernels gives up after a limit.  The
test shortens that limit to 64 cycles (parallax_set_wait_limit), so waits
that would have completed time out: the kernel records (kernel id, wait site)
in the device status word, every role of each aborted CTA leaves its loop,
waits for its own copies and MMAs in flight (long bound) and releases its
TMEM.  The host then reads PLX_ERR_TIMEOUT through
parallax_last_device_error, and the context is still usable: with the default
limit restored, the next forward and backward agree with the oracle.  No
trap, assert, bad address or endless loop is involved.
"""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import TOL_BF16, TOL_BF16_GRAD, inputs_f64, rel_err, to_device, to_host64

pytestmark = pytest.mark.gpu

KERNEL_IDS = set(range(1, 8))  # KID_TC_PASS1 .. KID_TC_BWD_B2


def _fwd_bwd(t):
    out, lse, mu = plx.parallax_fwd(t["q"], t["k"], t["v"], t["P"])
    dq, dk, dv, dP = plx.parallax_bwd(t["q"], t["k"], t["v"], t["P"], lse, mu, t["dout"])
    return out, mu, dq, dk, dv, dP


@pytest.mark.parametrize("d", [64, 128])
def test_short_wait_limit_times_out_and_the_context_recovers(d):
    assert torch.cuda.is_available()
    prev = plx.parallax_set_path(plx.PLX_PATH_TC)
    try:
        inp = plx_synth.generate(1, 2, 1024, d, "bf16", seed=70 + d, p_std=0.3 / np.sqrt(d), backward=True)
        t = {n: to_device(inp[n]) for n in ("q", "k", "v", "P", "dout")}
        _fwd_bwd(t)
        assert plx.parallax_last_device_error() == (plx.PLX_OK, 0)

        plx.parallax_set_wait_limit(64)
        try:
            _fwd_bwd(t)
            code, detail = plx.parallax_last_device_error()
        finally:
            plx.parallax_set_wait_limit(0)
        assert code == plx.PLX_ERR_TIMEOUT, (code, hex(detail))
        assert (detail >> 16) in KERNEL_IDS and (detail & 0xFFFF) > 0, hex(detail)
        # reading the status cleared it
        assert plx.parallax_last_device_error() == (plx.PLX_OK, 0)

        out, mu, dq, dk, dv, dP = _fwd_bwd(t)
        assert plx.parallax_last_device_error() == (plx.PLX_OK, 0)
        f = inputs_f64(inp)
        ro, _, rm = oracle.forward(f["q"], f["k"], f["v"], f["P"])
        rg = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"])
        assert rel_err(to_host64(out), ro, "bf16") < TOL_BF16
        assert rel_err(to_host64(mu), rm) < TOL_BF16
        for name, g, r in zip(("dq", "dk", "dv", "dP"), (dq, dk, dv, dP), rg):
            assert rel_err(to_host64(g), r, "bf16" if name != "dP" else "fp32") < TOL_BF16_GRAD, name
    finally:
        plx.parallax_set_path(prev)
        plx.parallax_set_wait_limit(0)
