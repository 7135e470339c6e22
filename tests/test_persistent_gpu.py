"""The persistent kernels with few CTAs: every CTA runs many work items.

Pass 2 of the tensor-core forward at d = 128 and B2 of the tensor-core
backward at d = 64 launch at most one CTA per SM (two for B2) and take work
items from a counter.  On the small problems the oracle checks element by
element, that grid already covers every item, so each CTA runs one item.
parallax_set_persistent_ctas caps the grid instead: with 1 to 3 CTAs, each
one runs items of mixed lengths back to back.  This exercises the item
changes: the slot pairs trading roles, the records of the next item, the
read-out of one item's output while the next one's scores run, and the end
record.

Each case is compared with the default grid bit for bit: only which CTA
runs an item changes, not the item's arithmetic.  The forward cases and the
first backward case are also compared with the fp64 oracle element by
element.  The second backward case (B1 H3 T1000, seed 1403) is compared bit
for bit only.  At that shape and seed, the default path's dq measures 0.0345
on the parity metric, above its 3e-2 bound.  The excess sits in the first
rows (t <= 8), which see one to nine keys: |dq| there is about ten times the
RMS, and the f16 rounding of U and z is amplified by terms that nearly
cancel.  Other seeds at the same shape measure 0.009 to 0.011.
"""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import (TOL_BF16, TOL_BF16_GRAD, guarded_empty, guards_intact, inputs_f64, rel_err,
                          to_device, to_host64)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tc_path():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    prev_path = plx.parallax_set_path(plx.PLX_PATH_TC)
    prev_cap = plx.parallax_set_persistent_ctas(0)
    yield
    plx.parallax_set_path(prev_path)
    plx.parallax_set_persistent_ctas(prev_cap)


def _forward(t):
    B, H, T, d = t["q"].shape
    g = {"out": guarded_empty((B, H, T, d), t["q"].dtype), "lse": guarded_empty((B, H, T), torch.float32),
         "mu": guarded_empty((B, H, T, d), torch.float32)}
    out, lse, mu = plx.parallax_fwd(t["q"], t["k"], t["v"], t["P"], out=g["out"][1], lse=g["lse"][1],
                                    mu_k=g["mu"][1])
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    for name, shape in (("out", (B, H, T, d)), ("lse", (B, H, T)), ("mu", (B, H, T, d))):
        assert guards_intact(g[name][0], shape), f"{name}: a store landed outside the tensor"
    return out.clone(), lse.clone(), mu.clone()


# (B, H, T, CTAs): query tiles of 128 rows give items of 1 .. ceil(T / 128)
# key tiles, and T not a multiple of 128 leaves a ragged last tile
FWD_CASES = [
    (1, 2, 1000, 3),
    (2, 3, 700, 2),
    (1, 5, 1100, 1),
    (1, 1, 129, 2),
]


@pytest.mark.parametrize("B,H,T,ctas", FWD_CASES)
def test_forward_d128_few_ctas_match_oracle_and_default_grid(B, H, T, ctas):
    d = 128
    inp = plx_synth.generate(B, H, T, d, "bf16", seed=300 + T + ctas, p_std=0.3 / np.sqrt(d))
    t = {n: to_device(inp[n]) for n in ("q", "k", "v", "P")}
    ref_out, ref_lse, ref_mu = _forward(t)  # default grid: one CTA per item here
    plx.parallax_set_persistent_ctas(ctas)
    out, lse, mu = _forward(t)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse) and torch.equal(mu, ref_mu)
    f = inputs_f64(inp)
    ro, rl, rm = oracle.forward(f["q"], f["k"], f["v"], f["P"])
    assert rel_err(to_host64(out), ro, "bf16") < TOL_BF16
    assert rel_err(to_host64(mu), rm) < TOL_BF16
    gl = to_host64(lse)
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, np.sqrt(np.mean(rl * rl)))


@pytest.mark.parametrize("B,H,T,ctas,vs_oracle", [(2, 2, 700, 1, True), (1, 3, 1000, 3, False)])
def test_backward_d64_few_ctas_match_default_grid(B, H, T, ctas, vs_oracle):
    d = 64
    inp = plx_synth.generate(B, H, T, d, "bf16", seed=400 + T + ctas, p_std=0.3 / np.sqrt(d), backward=True)
    t = {n: to_device(inp[n]) for n in ("q", "k", "v", "P", "dout")}

    def fwd_bwd():
        out, lse, mu = plx.parallax_fwd(t["q"], t["k"], t["v"], t["P"])
        grads = plx.parallax_bwd(t["q"], t["k"], t["v"], t["P"], lse, mu, t["dout"])
        code, detail = plx.parallax_last_device_error()
        assert code == plx.PLX_OK, (code, hex(detail))
        return [x.clone() for x in grads]

    ref = fwd_bwd()
    plx.parallax_set_persistent_ctas(ctas)
    got = fwd_bwd()
    for name, a, b in zip(("dq", "dk", "dv", "dP"), got, ref):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), name
    if not vs_oracle:
        return
    f = inputs_f64(inp)
    rg = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"])
    for name, g, r in zip(("dq", "dk", "dv", "dP"), got, rg):
        assert rel_err(to_host64(g), r, "bf16" if name != "dP" else "fp32") < TOL_BF16_GRAD, name
