"""The Python binding checks every tensor against q (shape, dtype, device,
contiguity) before any pointer reaches the C ABI, which cannot check them: a
smaller k or P would otherwise make a kernel read or write out of bounds.
These checks run on the host, so they are tested here without a GPU."""
import pytest
import torch

import parallax_local_linear_fwd_b300 as plx


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _fwd_args(B=1, H=2, T=16, d=64):
    return dict(q=_t(B, H, T, d), k=_t(B, H, T, d), v=_t(B, H, T, d), P=_t(H, d, d, dtype=torch.float32))


@pytest.mark.parametrize("name,bad,msg", [
    ("k", _t(1, 2, 8, 64), "k: expected shape"),
    ("v", _t(1, 2, 16, 64, dtype=torch.float32), "v: expected dtype"),
    ("P", _t(2, 64, 64), "P: expected dtype"),
    ("P", _t(1, 64, 64, dtype=torch.float32), "P: expected shape"),
    ("k", _t(1, 2, 64, 16).transpose(2, 3), "k must be contiguous"),
])
def test_forward_rejects_mismatched_tensors(name, bad, msg):
    a = _fwd_args()
    a[name] = bad
    for fn in (plx.parallax_fwd, plx.parallax_fwd_noalloc):
        with pytest.raises(ValueError, match=msg):
            fn(a["q"], a["k"], a["v"], a["P"])


def test_forward_rejects_mismatched_outputs():
    a = _fwd_args()
    with pytest.raises(ValueError, match="out: expected shape"):
        plx.parallax_fwd(a["q"], a["k"], a["v"], a["P"], out=_t(1, 2, 15, 64))
    with pytest.raises(ValueError, match="lse: expected dtype"):
        plx.parallax_fwd(a["q"], a["k"], a["v"], a["P"], lse=_t(1, 2, 16))
    with pytest.raises(ValueError, match="mu_k: expected shape"):
        plx.parallax_fwd(a["q"], a["k"], a["v"], a["P"], mu_k=_t(1, 2, 16, 32, dtype=torch.float32))
    with pytest.raises(ValueError, match="workspace is required"):
        plx.parallax_fwd_ws(a["q"], a["k"], a["v"], a["P"], _t(1, 2, 16, 64), _t(1, 2, 16, dtype=torch.float32),
                            _t(1, 2, 16, 64, dtype=torch.float32), None)


def test_host_tensors_are_refused_by_device_entry_points():
    a = _fwd_args()
    with pytest.raises(ValueError, match="CUDA device"):
        plx.parallax_fwd(a["q"], a["k"], a["v"], a["P"])


def test_backward_rejects_mismatched_tensors():
    a = _fwd_args()
    lse, mu = _t(1, 2, 16, dtype=torch.float32), _t(1, 2, 16, 64, dtype=torch.float32)
    do = _t(1, 2, 16, 64)
    with pytest.raises(ValueError, match="dout: expected shape"):
        plx.parallax_bwd(a["q"], a["k"], a["v"], a["P"], lse, mu, _t(1, 2, 16, 32))
    with pytest.raises(ValueError, match="mu_k: expected dtype"):
        plx.parallax_bwd(a["q"], a["k"], a["v"], a["P"], lse, _t(1, 2, 16, 64), do)
    with pytest.raises(ValueError, match="dP: expected shape"):
        plx.parallax_bwd(a["q"], a["k"], a["v"], a["P"], lse, mu, do, dP=_t(2, 64, 32, dtype=torch.float32))
    with pytest.raises(ValueError, match="dk: expected dtype"):
        plx.parallax_bwd(a["q"], a["k"], a["v"], a["P"], lse, mu, do, dk=_t(1, 2, 16, 64, dtype=torch.float32))


def test_probe_and_decode_reject_mismatched_tensors():
    a = _fwd_args()
    with pytest.raises(ValueError, match="rho: expected shape"):
        plx.parallax_fwd_probe(a["q"], a["k"], a["v"], _t(1, 2, 16, 128))
    kc, vc = _t(2, 2, 32, 64), _t(2, 2, 32, 64)
    P = _t(2, 64, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="q: expected shape"):
        plx.parallax_decode(_t(2, 1, 64), kc, vc, P)
    with pytest.raises(ValueError, match="v_cache: expected shape"):
        plx.parallax_decode(_t(2, 2, 64), kc, _t(2, 2, 31, 64), P)
    with pytest.raises(ValueError, match="lens: expected dtype"):
        plx.parallax_decode(_t(2, 2, 64), kc, vc, P, lens=torch.zeros(2, dtype=torch.int64))


def test_step_host_rejects_mismatched_tensors():
    a = _fwd_args()
    with pytest.raises(ValueError, match="dout: expected shape"):
        plx.parallax_step_host(a["q"], a["k"], a["v"], a["P"], _t(1, 2, 16, 32))
    with pytest.raises(ValueError, match="P: expected shape"):
        plx.parallax_step_host(a["q"], a["k"], a["v"], _t(3, 64, 64, dtype=torch.float32), _t(1, 2, 16, 64))
