"""CPU checks of the library's host-side logic and its C ABI surface: the work
split, the tiled layout, the exported symbols and host-side validation."""
import os
import re
import subprocess

import pytest

from transformer_layer_decode_gb300 import build as tld_build
from transformer_layer_decode_gb300 import dec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "transformer_layer_decode_gb300", "csrc")


def test_split_and_tiled_layout(tmp_path):
    exe = tmp_path / "host_logic_check"
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", "/usr/local/cuda/include",
                    os.path.join(ROOT, "tests", "host", "host_logic_check.cpp"), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "dec.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(dec_\w+)\(", src, re.M)))


@pytest.fixture(scope="module")
def lib():
    tld_build.build()
    return dec.load_library()


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert set(names) == set(dec.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", tld_build.LIB], capture_output=True,
                         text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, re.M), n


def _create(lib, **kw):
    import ctypes
    base = dict(n_layers=1, hidden=512, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=1408,
                rms_eps=1e-6, rope_theta=1e4, max_ctx=128, weight_fmt=0, flags=0)
    base.update(kw)
    desc = dec.ModelDesc(*[base[f] for f, _ in dec.ModelDesc._fields_])
    h = ctypes.c_void_p()
    rc = lib.dec_create(ctypes.byref(desc), ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw,code", [
    ({"head_dim": 96}, dec.DEC_ERR_SHAPE),
    ({"n_q_heads": 6, "n_kv_heads": 4}, dec.DEC_ERR_SHAPE),
    ({"n_q_heads": 48, "n_kv_heads": 3}, dec.DEC_ERR_SHAPE),
    ({"hidden": 500}, dec.DEC_ERR_SHAPE),
    ({"ffn": 1410}, dec.DEC_ERR_SHAPE),
    ({"max_ctx": 70000}, dec.DEC_ERR_SHAPE),
    ({"n_layers": 0}, dec.DEC_ERR_ARG),
    ({"weight_fmt": 7}, dec.DEC_ERR_ARG),
    ({"flags": 8192}, dec.DEC_ERR_ARG),
    ({"flags": 1 | 512}, dec.DEC_ERR_SHAPE),   # paged KV cache with the unfused plan
    ({"flags": 4096 | 32}, dec.DEC_ERR_SHAPE),  # attention + o-proj without the cluster attention
    ({"rope_theta": 0.0}, dec.DEC_ERR_ARG),
])
def test_create_rejects_bad_descs_on_the_host(lib, kw, code):
    rc, h = _create(lib, **kw)
    assert rc == code and not h.value
    assert lib.dec_last_error(None).decode()


def test_null_arguments_are_errors(lib):
    import ctypes
    assert lib.dec_create(None, None) == dec.DEC_ERR_ARG
    h = ctypes.c_void_p()
    assert lib.dec_create(None, ctypes.byref(h)) == dec.DEC_ERR_ARG
    assert lib.dec_step(None, None, 0, None, None) == dec.DEC_ERR_ARG
    assert lib.dec_load_weights(None, 0, 0, None, 0) == dec.DEC_ERR_ARG
    assert lib.dec_destroy(None) == dec.DEC_OK


def test_missing_library_fails_loudly(tmp_path):
    """A loader pointed at a missing library raises instead of falling back."""
    with pytest.raises(RuntimeError, match="not built"):
        dec.load_library(str(tmp_path / "nope.so"))


def test_quantizer_rounding_matches_ieee_division(tmp_path):
    """The int8 quantizer's quotients from the reciprocal with one FMA correction
    equal the IEEE fp32 division (scales, quotients and codes)."""
    exe = tmp_path / "quant_rounding_check"
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off",
                    os.path.join(ROOT, "tests", "host", "quant_rounding_check.cpp"), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout
