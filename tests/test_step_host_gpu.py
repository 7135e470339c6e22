"""parallax_step_host (host buffers, head groups with copies overlapped) against
the device entry points on the same inputs, and against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import TOL_BF16, TOL_BF16_GRAD, inputs_f64, rel_err, to_host64

pytestmark = pytest.mark.gpu


def _host_inputs(B, H, T, d, dtype, seed):
    inp = plx_synth.generate(B, H, T, d, dtype, seed=seed, p_std=0.3 / np.sqrt(d), backward=True)

    def host(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
        return torch.from_numpy(x).pin_memory()

    return inp, {n: host(inp[n]) for n in ("q", "k", "v", "P", "dout")}


def _device_reference(h):
    d_ = {n: t.cuda() for n, t in h.items()}
    out, lse, mu = plx.parallax_fwd(d_["q"], d_["k"], d_["v"], d_["P"])
    dq, dk, dv, dP = plx.parallax_bwd(d_["q"], d_["k"], d_["v"], d_["P"], lse, mu, d_["dout"])
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in dict(out=out, lse=lse, mu_k=mu, dq=dq, dk=dk, dv=dv, dP=dP).items()}


def _host_step(h, chunks, want_stats=True):
    B, H, T, d = h["q"].shape
    lse = torch.empty((B, H, T), dtype=torch.float32).pin_memory() if want_stats else None
    mu = torch.empty((B, H, T, d), dtype=torch.float32).pin_memory() if want_stats else None
    out, dq, dk, dv, dP, lse, mu = plx.parallax_step_host(h["q"], h["k"], h["v"], h["P"], h["dout"],
                                                          lse=lse, mu_k=mu, chunks=chunks)
    torch.cuda.synchronize()
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    return dict(out=out, lse=lse, mu_k=mu, dq=dq, dk=dk, dv=dv, dP=dP)


def _same_dq(a, b):
    # one unit of the storage rounding: the fp32 reduce-add order differs between runs
    a, b = a.double(), b.double()
    ulp = 2.0 ** -7 if a.dtype == torch.bfloat16 else 2.0 ** -22
    return bool(((a - b).abs() <= ulp * b.abs() + 1e-6 * b.pow(2).mean().sqrt()).all())


@pytest.mark.parametrize("B,H,T,d,dtype,chunks", [
    (2, 5, 300, 64, "bf16", 0),     # default grouping: 5 groups of one head
    (2, 5, 300, 64, "bf16", 2),     # uneven groups: 3 + 2 heads
    (1, 3, 129, 128, "bf16", 3),
    (2, 4, 100, 64, "fp32", 1),     # one group, SIMT family
    (1, 3, 70, 64, "fp32", 2),
])
def test_host_step_matches_device_entry_points(B, H, T, d, dtype, chunks):
    _, h = _host_inputs(B, H, T, d, dtype, seed=100 + T)
    ref = _device_reference(h)
    got = _host_step(h, chunks)
    for name in ("out", "lse", "mu_k", "dk", "dv", "dP"):
        assert torch.equal(got[name], ref[name]), name
    assert _same_dq(got["dq"], ref["dq"])


def test_host_step_against_the_oracle():
    B, H, T, d = 1, 2, 96, 64
    inp, h = _host_inputs(B, H, T, d, "bf16", seed=5)
    got = _host_step(h, chunks=2, want_stats=False)
    assert got["lse"] is None and got["mu_k"] is None
    f = inputs_f64(inp)
    ro, rl, rm = oracle.forward(f["q"], f["k"], f["v"], f["P"])
    assert rel_err(to_host64(got["out"]), ro, "bf16") < TOL_BF16
    rdq, rdk, rdv, rdP = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"])
    for g, r in ((got["dq"], rdq), (got["dk"], rdk), (got["dv"], rdv)):
        assert rel_err(to_host64(g), r, "bf16") < TOL_BF16_GRAD
    assert rel_err(got["dP"].double().numpy(), rdP, "fp32") < TOL_BF16_GRAD


def test_host_step_rejects_device_pointers():
    q = torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    P = torch.zeros(1, 64, 64, device="cuda")
    L = plx.lib()
    ptr = ctypes.c_void_p
    args = [ptr(q.data_ptr())] * 3 + [ptr(P.data_ptr()), ptr(q.data_ptr())] + [ptr(q.data_ptr()), None, None] + \
        [ptr(q.data_ptr())] * 3 + [ptr(P.data_ptr())]
    rc = L.parallax_step_host(*args, 0, 1, 1, 16, 64, plx.PLX_BF16, None)
    assert rc == plx.PLX_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        plx.parallax_step_host(q, q, q, P, q)
    assert plx.parallax_last_device_error()[0] == plx.PLX_OK
