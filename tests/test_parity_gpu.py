"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every output, with every
output surrounded by guard bands that must come back untouched.  The
full-size workloads are compared element by element on one complete head
(every query row of it) plus rows sampled from every head (forward), and on
all batches of one head (backward), which the oracle computes directly.
Tolerances are max |gpu - oracle| / RMS(oracle): 1e-4 for fp32, 2e-2 for
bf16 outputs, 3e-2 for bf16 gradients.
"""
import numpy as np
import pytest
import torch

import oracle
import parallax_local_linear_fwd_b300 as plx
import plx_synth
from plx_testutil import (TOL_BF16, TOL_BF16_GRAD, TOL_FP32, guarded_empty, guards_intact, inputs_f64,
                          rel_err, sample_rows, to_device, to_host64)

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


def _run_fwd(inp, guard=False):
    q, k, v, P = (to_device(inp[x]) for x in ("q", "k", "v", "P"))
    if guard:
        B, H, T, d = q.shape
        shapes = {"out": ((B, H, T, d), q.dtype), "lse": ((B, H, T), torch.float32),
                  "mu": ((B, H, T, d), torch.float32)}
        g = {n: guarded_empty(sh, dt) for n, (sh, dt) in shapes.items()}
        out, lse, mu = plx.parallax_fwd(q, k, v, P, out=g["out"][1], lse=g["lse"][1], mu_k=g["mu"][1])
    else:
        out, lse, mu = plx.parallax_fwd(q, k, v, P)
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    if guard:
        for n, (sh, _) in shapes.items():
            assert guards_intact(g[n][0], sh), f"{n}: a store landed outside the tensor"
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
    (1, 2, 33, 64, "bf16"),
    (2, 2, 130, 64, "bf16"),
    (1, 1, 257, 128, "bf16"),
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
    go, gl, gm = _run_fwd(inp, guard=True)
    tol = _tol(dtype)
    assert rel_err(go, ro, dtype) < tol
    assert rel_err(gm, rm) < tol
    assert np.abs(gl - rl).max() < tol * max(1.0, np.sqrt(np.mean(rl * rl)))


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("qk_scale,v_scale,p_scale,d", [(30.0, 100.0, 1.0, 64), (100.0, 1.0e4, 1.0e-4, 128)])
def test_forward_large_magnitude_inputs(path, qk_scale, v_scale, p_scale, d):
    # q, k and v far from unit scale but inside f16's range (|x| < 65504): the
    # tensor-core path converts every operand to f16 exactly there.  In the
    # second case P shrinks by 1/qk_scale^2, so that g = k . P (q - mu_k) keeps
    # its usual size: with P unscaled, g reaches ~1e5 there, and the output
    # then depends on P's last bits (f16 weights, relative 2^-11) -- a
    # conditioning limit of the problem stated in the header, not a range one.
    _use_path(path, "bf16")
    B, H, T = 1, 2, 300
    inp = plx_synth.generate(B, H, T, d, "bf16", seed=90 + d, p_std=0.3 / np.sqrt(d))
    for name, sc in (("q", qk_scale), ("k", qk_scale), ("v", v_scale)):
        inp[name] = plx_synth.to_bf16_bits(plx_synth.widen(inp[name]) * sc)
    inp["P"] = (inp["P"].astype(np.float64) * p_scale).astype(np.float32)
    assert np.abs(plx_synth.widen(inp["v"])).max() < 65504
    f = inputs_f64(inp)
    ro, rl, rm = oracle.forward(f["q"], f["k"], f["v"], f["P"])
    go, gl, gm = _run_fwd(inp, guard=True)
    assert rel_err(go, ro, "bf16") < TOL_BF16
    assert rel_err(gm, rm) < TOL_BF16
    assert np.abs(gl - rl).max() < TOL_BF16 * max(1.0, np.sqrt(np.mean(rl * rl)))


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


# One complete head per full-size workload: (b, h) of the head compared over
# every query row.
FULL_HEAD = {"c2": (7, 5), "c3": (3, 15), "c4": (5, 9), "c5": (0, 11)}


@pytest.mark.parametrize("name", ["c2", "c3", "c5", "c4"])
def test_forward_full_size(name):
    """The forward at full size, in the launch configuration the benchmark
    times: one complete head element by element against the oracle, rows
    sampled from every head, and at every row of every head the bound
    lse_t >= c q_t . k_t (the log-sum-exp is at least its diagonal term)."""
    plx.parallax_set_path(plx.PLX_PATH_AUTO)
    inp = plx_synth.generate_workload(name)
    B, H, T, d = inp["B"], inp["H"], inp["T"], inp["d"]
    go, gl, gm = _run_fwd(inp)
    f = inputs_f64(inp)
    b, h = FULL_HEAD[name]
    rows = sorted(set(sample_rows(B, H, T, 48, seed=len(name))) | {(b, h, t) for t in range(T)})
    ro, rl, rm = oracle.forward_rows(f["q"], f["k"], f["v"], f["P"], rows)
    idx = tuple(np.array(rows).T)
    assert rel_err(go[idx], ro, "bf16") < TOL_BF16
    assert rel_err(gm[idx], rm) < TOL_BF16
    assert np.abs(gl[idx] - rl).max() < TOL_BF16 * max(1.0, np.sqrt(np.mean(rl * rl)))
    head = np.array([r[0] == b and r[1] == h for r in rows])
    assert head.sum() == T
    assert rel_err(go[idx][head], ro[head], "bf16") < TOL_BF16
    assert rel_err(gm[idx][head], rm[head]) < TOL_BF16
    # properties at every row: finite outputs, lse >= the diagonal score
    assert np.isfinite(go).all() and np.isfinite(gl).all() and np.isfinite(gm).all()
    diag = np.einsum("bhtd,bhtd->bht", f["q"], f["k"]) / np.sqrt(d)
    assert (gl >= diag - 1e-5 * np.maximum(1.0, np.abs(diag))).all()


def _run_bwd(inp, guard=False):
    q, k, v, P, do = (to_device(inp[x]) for x in ("q", "k", "v", "P", "dout"))
    out, lse, mu = plx.parallax_fwd(q, k, v, P)
    if guard:
        B, H, T, d = q.shape
        shapes = {"dq": ((B, H, T, d), q.dtype), "dk": ((B, H, T, d), q.dtype), "dv": ((B, H, T, d), q.dtype),
                  "dP": ((H, d, d), torch.float32)}
        g = {n: guarded_empty(sh, dt) for n, (sh, dt) in shapes.items()}
        dq, dk, dv, dP = plx.parallax_bwd(q, k, v, P, lse, mu, do, dq=g["dq"][1], dk=g["dk"][1], dv=g["dv"][1],
                                          dP=g["dP"][1])
    else:
        dq, dk, dv, dP = plx.parallax_bwd(q, k, v, P, lse, mu, do)
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    if guard:
        for n, (sh, _) in shapes.items():
            assert guards_intact(g[n][0], sh), f"{n}: a store landed outside the tensor"
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
    got = _run_bwd(inp, guard=True)
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


@pytest.mark.parametrize("path", ["simt", "tc"])
@pytest.mark.parametrize("B,H,T,d,dtype", [(2, 2, 130, 64, "bf16"), (1, 2, 257, 128, "bf16"), (1, 2, 100, 64, "fp32")])
def test_fused_step_equals_separate_calls(path, B, H, T, d, dtype):
    # parallax_fwd_bwd shares one workspace between the passes (the backward
    # reads the forward's f16 copies): every output equals parallax_fwd then
    # parallax_bwd bit for bit, and stays inside its tensor
    _use_path(path, dtype)
    inp = plx_synth.generate(B, H, T, d, dtype, seed=11 * T + d, p_std=0.3 / np.sqrt(d), backward=True)
    q, k, v, P, do = (to_device(inp[x]) for x in ("q", "k", "v", "P", "dout"))
    out, lse, mu = plx.parallax_fwd(q, k, v, P)
    sep = (out, lse, mu) + tuple(plx.parallax_bwd(q, k, v, P, lse, mu, do))
    shapes = {"out": ((B, H, T, d), q.dtype), "lse": ((B, H, T), torch.float32), "mu": ((B, H, T, d), torch.float32),
              "dq": ((B, H, T, d), q.dtype), "dk": ((B, H, T, d), q.dtype), "dv": ((B, H, T, d), q.dtype),
              "dP": ((H, d, d), torch.float32)}
    g = {n: guarded_empty(sh, dt) for n, (sh, dt) in shapes.items()}
    fused = plx.parallax_fwd_bwd(q, k, v, P, do, out=g["out"][1], lse=g["lse"][1], mu_k=g["mu"][1], dq=g["dq"][1],
                                 dk=g["dk"][1], dv=g["dv"][1], dP=g["dP"][1])
    code, detail = plx.parallax_last_device_error()
    assert code == plx.PLX_OK, (code, hex(detail))
    for n, a_, b_ in zip(shapes, sep, fused):
        assert torch.equal(a_, b_), n
        assert guards_intact(g[n][0], shapes[n][0]), f"{n}: a store landed outside the tensor"
    # and the fused step agrees with the oracle
    f = inputs_f64(inp)
    ref = oracle.backward(f["q"], f["k"], f["v"], f["P"], f["dout"])
    tol = TOL_FP32 if dtype == "fp32" else TOL_BF16_GRAD
    for name, got, r in zip(("dq", "dk", "dv", "dP"), fused[3:], ref):
        assert rel_err(to_host64(got), r, dtype if name != "dP" else "fp32") < tol, name


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
