"""CPU-only checks of the C ABI: the library builds, loads, and exports every
symbol include/parallax.h declares; host-side argument checks return the
documented codes without touching a GPU."""
import ctypes
import os
import re

import pytest

import parallax_local_linear_fwd_b300 as plx
from parallax_local_linear_fwd_b300 import build as plx_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(parallax_\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def L():
    plx_build.build()
    return plx.lib()


def test_every_declared_symbol_is_exported(L):
    declared = _declared_symbols()
    assert "parallax_fwd" in declared and "parallax_bwd" in declared
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(declared) == sorted(plx.exported_symbols())


def test_hidden_internals(L):
    # only the C ABI is exported; kernel-side C++ symbols stay hidden
    with pytest.raises(AttributeError):
        getattr(L, "_ZN3plx8simt_fwdERKNS_7FwdArgsE")


def test_strerror_and_path(L):
    for code in range(5):
        assert plx.parallax_strerror(code)
    assert "unknown" in plx.parallax_strerror(99)
    prev = plx.parallax_set_path(plx.PLX_PATH_SIMT)
    assert plx.parallax_set_path(prev) == plx.PLX_PATH_SIMT
    assert plx.parallax_set_path(7) == -1


def test_persistent_ctas_cap_needs_no_gpu(L):
    assert L.parallax_set_persistent_ctas(-1) == -1
    with pytest.raises(ValueError):
        plx.parallax_set_persistent_ctas(-1)
    prev = plx.parallax_set_persistent_ctas(5)
    assert plx.parallax_set_persistent_ctas(prev) == 5


def test_host_argument_checks_need_no_gpu(L):
    p = ctypes.c_void_p(256)  # never dereferenced: the checks fail first
    assert L.parallax_fwd(p, p, p, p, p, p, p, 1, 1, 16, 96, 1, None) == plx.PLX_ERR_UNSUPPORTED
    assert L.parallax_fwd(p, p, p, p, p, p, p, 1, 1, 16, 64, 5, None) == plx.PLX_ERR_UNSUPPORTED
    assert L.parallax_fwd(p, p, p, p, p, p, p, 0, 1, 16, 64, 1, None) == plx.PLX_ERR_INVALID_ARG
    assert L.parallax_fwd(p, p, p, p, p, p, p, 1, 1, 0, 64, 1, None) == plx.PLX_ERR_INVALID_ARG
    assert L.parallax_fwd(None, p, p, p, p, p, p, 1, 1, 16, 64, 1, None) == plx.PLX_ERR_INVALID_ARG
    q = ctypes.c_void_p(258)  # misaligned
    assert L.parallax_fwd(q, p, p, p, p, p, p, 1, 1, 16, 64, 1, None) == plx.PLX_ERR_INVALID_ARG
    assert L.parallax_fwd_ws(p, p, p, p, p, p, p, ctypes.c_void_p(16), 1, 1, 16, 64, 1, None) \
        == plx.PLX_ERR_INVALID_ARG
    args = [p] * 11
    assert L.parallax_bwd(*args, None, 1, 1, 16, 48, 1, None) == plx.PLX_ERR_UNSUPPORTED
    assert L.parallax_bwd(*args, ctypes.c_void_p(272), 1, 1, 16, 64, 1, None) == plx.PLX_ERR_INVALID_ARG
    assert L.parallax_fwd_workspace_bytes(1, 1, 16, 80, 1) == 0
    assert L.parallax_bwd_workspace_bytes(-1, 1, 16, 64, 1) == 0
    # 2^31 elements overflow the supported index range
    assert L.parallax_fwd(p, p, p, p, p, p, p, 1 << 10, 1 << 10, 1 << 10, 64, 1, None) == plx.PLX_ERR_INVALID_ARG


def test_decode_probe_workspace_holds_a_partial_per_cta_and_head(L):
    # the given-probe decode splits the tiles of all heads over at most 1024
    # CTAs and writes one partial {m, l, sum p r, pad, sum p v [d], sum p r v [d]}
    # per (CTA, head) pair that overlaps, in slot cta + head
    for B, H, Lmax, d in ((1, 1, 1, 64), (8, 16, 4096, 64), (4, 16, 4096, 128), (128, 16, 32, 64)):
        need = (1024 + B * H) * (4 + 2 * d) * 4
        got = L.parallax_decode_probe_workspace_bytes(B, H, Lmax, d, plx.PLX_BF16)
        assert got >= need and got % 256 == 0, (B, H, Lmax, d, got, need)
    assert L.parallax_decode_probe_workspace_bytes(1, 1, 16, 64, plx.PLX_FP32) == 0
