"""The C-ABI library builds for sm_103a, loads without a GPU, and exports
every entry point that include/*.h declares.  CPU only (no compute calls)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:int|void)\s+(spec_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libpath():
    from speculative_decoding_verification_round_gb300 import _build
    return _build.build()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["spec_model_create", "spec_linear_q", "spec_verify_attn", "spec_lm_head",
                     "spec_accept_greedy", "spec_accept_stochastic", "spec_verify_round"]:
        assert required in names


def test_library_exports_every_declared_symbol(libpath):
    L = ctypes.CDLL(libpath)
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_lists_the_same_symbols(libpath):
    import speculative_decoding_verification_round_gb300 as sv
    assert sorted(sv.EXPORTED) == declared_functions()
    sv.lib()  # loads and binds signatures


def test_host_side_checks_fail_closed_without_gpu(libpath):
    """Argument checks happen before any device work: errors come back as
    codes with a message, never a crash."""
    import speculative_decoding_verification_round_gb300 as sv
    L = sv.lib()
    assert L.spec_verify_round(None, 1, None, None, 0, None, None, None, None, None, None) == sv.SPEC_E_INVALID
    assert "null" in sv.last_error()
    assert L.spec_linear_q(None, None, 1, None, None) == sv.SPEC_E_INVALID
    qw = sv.spec_qweight(5, 16, 32, None, None, None)
    h = ctypes.c_void_p()
    assert L.spec_qmat_create(ctypes.byref(qw), 16, None, ctypes.byref(h)) != sv.SPEC_OK
    assert L.spec_accept_greedy(None, None, 1, 1, None, None, None) == sv.SPEC_E_INVALID


def test_binding_constants_match_the_header():
    """The binding's copies of the header's #defines (block formats, the row
    limit, error codes) are the header's values."""
    import speculative_decoding_verification_round_gb300 as sv
    text = open(os.path.join(ROOT, "include", "spec_verify.h")).read()
    defs = dict(re.findall(r"^#define\s+(SPEC_\w+)\s+\(?(-?\d+)\)?", text, flags=re.M))
    for name in ["SPEC_OK", "SPEC_E_INVALID", "SPEC_E_SHAPE", "SPEC_E_CUDA", "SPEC_E_OOM",
                 "SPEC_E_UNSUPPORTED", "SPEC_E_TIMEOUT", "SPEC_Q4", "SPEC_Q6", "SPEC_Q8",
                 "SPEC_MAX_NT"]:
        assert name in defs, name
        assert getattr(sv, name) == int(defs[name]), name


def test_q8_weight_without_its_plane_fails_closed(libpath):
    import speculative_decoding_verification_round_gb300 as sv
    L = sv.lib()
    h = ctypes.c_void_p()
    qw = sv.spec_qweight(sv.SPEC_Q8, 16, 64, None, None, None)
    assert L.spec_qmat_create(ctypes.byref(qw), 16, None, ctypes.byref(h)) == sv.SPEC_E_INVALID
    assert "plane" in sv.last_error()
