"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every output; the full-size
workloads are compared on sampled rows (forward) and on a subset of heads
(backward) that the oracle computes directly.  Tolerances are
max |gpu - oracle| / RMS(oracle): 1e-4 for fp32, 2e-2 for bf16 outputs,
3e-2 for bf16 gradients.
"""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import (TOL_BF16, TOL_BF16_GRAD, TOL_FP32, inputs_f64, rel_err, sample_rows,
                          to_device, to_host64)

pytestmark = pytest.mark.gpu

PATHS = {"simt": plx.PLX_PATH_SIMT, "tc": plx.PLX_PATH_TC}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    plx.lib()
    yield
    plx.parallax_set_path(plx.PLX_PATH_AUTO)


def _tc_available():
    prev = plx.parallax_set_path(plx.PLX_PATH_TC)
    try:
        return plx.parallax_fwd_workspace_bytes(1, 1, 128, 64, plx.PLX_BF16) > 0
    finally:
        plx.parallax_set_path(prev)


def _use_path(name, dtype):
    if name == "tc":
        if dtype != "bf16":
            pytest.skip("tensor-core path is bf16 only")
        if not _tc_available():
            pytest.skip("tensor-core path not built yet")
    plx.parallax_set_path(PATHS[name])


def _run_fwd(inp):
    q, k, v, P = (to_device(inp[x]) for x in ("q", "k", "v", "P"))
    out, lse, mu = plx.parallax_fwd(q, k, v, P)
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    return to_host64(out), to_host64(lse), to_host64(mu)


def _tol(dtype):
    return TOL_FP32 if dtype == "fp32" else TOL_BF16


SMALL = [
    # (B, H, T, d, dtype)
    (1, 2, 256, 64, "fp32"),
    (1, 1, 1, 64, "fp32"),
    (2, 3, 77, 128, "fp32"),
    (1, 1, 1, 64, "bf16"),
    (1, 2, 7, 128, "bf16"),
    (2, 2, 130, 64, "bf16"),
    (1, 3, 300, 128, "bf16"),
    (2, 1, 513, 64, "bf16"),
]


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("B,H,T,d,dtype", SMALL)
def test_forward_small_full_compare(path, B, H, T, d, dtype):
    _use_path(path, dtype)
    inp = plx_synth.generate(B, H, T, d, dtype, seed=T + d, p_std=0.3 / np.sqrt(d))
    f = inputs_f64(inp)
    ro, rl, rm = oracle.forward(f["q"], f["k"], f["v"], f["P"])
    go, gl, gm = _run_fwd(inp)
    tol = _tol(dtype)
    assert rel_err(go, ro, dtype) < tol
    assert rel_err(gm, rm) < tol
    assert np.abs(gl - rl).max() < tol * max(1.0, np.sqrt(np.mean(rl * rl)))


@pytest.mark.parametrize("path", ["simt", "tc"])
def test_pr1_workload_and_zero_projector(path):
    _use_path(path, "fp32" if path == "simt" else "bf16")
    w = plx_synth.WORKLOADS["pr1"]
    dtype = w.dtype if path == "simt" else "bf16"
    for zero in (False, True):
        inp = plx_synth.generate(w.B, w.H, w.T, w.d, dtype, seed=w.seed, p_std=w.p_std, zero_P=zero)
        f = inputs_f64(inp)
        ro, rl, rm = oracle.forward(f["q"], f["k"], f["v"], f["P"])
        go, gl, gm = _run_fwd(inp)
        tol = _tol(dtype)
        assert rel_err(go, ro, dtype) < tol
        assert rel_err(gm, rm) < tol
        if zero:
            # P = 0 must give softmax attention (library routine, fp64)
            sd = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(f["q"]), torch.from_numpy(f["k"]), torch.from_numpy(f["v"]),
                is_causal=True).numpy()
            assert rel_err(go, sd, dtype) < tol


@pytest.mark.parametrize("name", ["c2", "c3", "c5"])
def test_forward_full_size_sampled_rows(name):
    plx.parallax_set_path(plx.PLX_PATH_AUTO)
    inp = plx_synth.generate_workload(name)
    B, H, T, d = inp["B"], inp["H"], inp["T"], inp["d"]
    go, gl, gm = _run_fwd(inp)
    rows = sample_rows(B, H, T, 48, seed=len(name))
    f = inputs_f64(inp)
    ro, rl, rm = oracle.forward_rows(f["q"], f["k"], f["v"], f["P"], rows)
    idx = tuple(np.array(rows).T)
    assert rel_err(go[idx], ro, "bf16") < TOL_BF16
    assert rel_err(gm[idx], rm) < TOL_BF16
    assert np.abs(gl[idx] - rl).max() < TOL_BF16 * max(1.0, np.sqrt(np.mean(rl * rl)))
    # properties at every row: finite outputs, lse >= the diagonal score
    assert np.isfinite(go).all() and np.isfinite(gl).all() and np.isfinite(gm).all()


def _run_bwd(inp, out_dev=None):
    q, k, v, P, do = (to_device(inp[x]) for x in ("q", "k", "v", "P", "dout"))
    out, lse, mu = plx.parallax_fwd(q, k, v, P)
    dq, dk, dv, dP = plx.parallax_bwd(q, k, v, P, lse, mu, do)
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    return [to_host64(x) for x in (dq, dk, dv, dP)]


BWD_SMALL = [
    (1, 2, 64, 64, "fp32"),
    (2, 2, 100, 128, "fp32"),
    (1, 1, 1, 64, "bf16"),
    (2, 1, 33, 64, "bf16"),
    (1, 1, 96, 64, "bf16"),
    (2, 2, 130, 64, "bf16"),
    (1, 2, 260, 64, "bf16"),
    (1, 2, 257, 128, "bf16"),
]


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("B,H,T,d,dtype", BWD_SMALL)
def test_backward_small_full_compare(path, B, H, T, d, dtype):
    _use_path(path, dtype)
    inp = plx_synth.generate(B, H, T, d, dtype, seed=3 * T + d, p_std=0.3 / np.sqrt(d), backward=True)
    f = inputs_f64(inp)
    ref = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"])
    got = _run_bwd(inp)
    tol = TOL_FP32 if dtype == "fp32" else TOL_BF16_GRAD
    for name, g, r in zip(("dq", "dk", "dv", "dP"), got, ref):
        assert rel_err(g, r, dtype if name != "dP" else "fp32") < tol, name


def test_backward_full_size_c4_head_subset():
    plx.parallax_set_path(plx.PLX_PATH_AUTO)
    inp = plx_synth.generate_workload("c4")
    B, H = inp["B"], inp["H"]
    got = _run_bwd(inp)
    h = 3
    heads = [(b, h) for b in range(B)]  # all batches of one head: the full dP_h
    f = inputs_f64(inp)
    ref = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"], heads=heads)
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        assert rel_err(g[:, h], r[:, h], "bf16") < TOL_BF16_GRAD, name
    assert rel_err(got[3][h], ref[3][h]) < TOL_BF16_GRAD, "dP"
    for g in got:
        assert np.isfinite(g).all()


def test_dp_is_bitwise_reproducible():
    plx.parallax_set_path(plx.PLX_PATH_AUTO)
    inp = plx_synth.generate(2, 2, 300, 64, "bf16", seed=5, p_std=0.05, backward=True)
    a = _run_bwd(inp)
    b = _run_bwd(inp)
    np.testing.assert_array_equal(a[3], b[3])


def test_invalid_arguments_return_codes():
    x = torch.zeros(1, 1, 16, 64, device="cuda", dtype=torch.bfloat16)
    P = torch.zeros(1, 64, 64, device="cuda")
    with pytest.raises(plx.PlxError) as e:
        plx.parallax_fwd(x[..., :48].contiguous(), x[..., :48].contiguous(), x[..., :48].contiguous(),
                         P[:, :48, :48].contiguous())
    assert e.value.code == plx.PLX_ERR_UNSUPPORTED
    raw = torch.zeros(1 * 16 * 64 + 1, device="cuda", dtype=torch.bfloat16)
    mis = raw[1:].view(1, 1, 16, 64)  # 2-byte offset: misaligned
    with pytest.raises(plx.PlxError) as e:
        plx.parallax_fwd(mis, x, x, P)
    assert e.value.code == plx.PLX_ERR_INVALID_ARG
    assert plx.parallax_last_device_error()[0] == plx.PLX_OK
