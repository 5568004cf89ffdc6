"""The C ABI boundary without a GPU: the library builds and loads, exports
every entry point include/specverify.h declares, and rejects bad arguments
before it touches a device."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_06_gb300 as sv
from speculative_decoding_verification_06_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def exported_symbols():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_header_declares_the_binding_names():
    assert declared_functions() == sorted(sv.EXPORTED)


def test_library_exports_every_declared_function(lib):
    syms = exported_symbols()
    missing = [f for f in declared_functions() if f not in syms]
    assert not missing, missing
    for f in declared_functions():
        assert hasattr(lib, f)


def test_status_strings_and_version(lib):
    assert sv.version() == 10000
    for code in range(6):
        assert sv.status_string(code)
    assert sv.status_string(99) == "unknown status"


def _call(lib, B=2, gamma=3, V=64, dtype=0, ptr=0x1000, ws=0x1000, ws_bytes=1 << 20):
    p = ptr
    return lib.spec_verify(p, p, dtype, B, gamma, V, p, p, p, p, p, p, ws, ws_bytes, None)


def test_bad_shapes_are_rejected_before_launch(lib):
    assert _call(lib, B=-1) == sv.SV_ERR_INVALID_ARG
    assert _call(lib, gamma=0) == sv.SV_ERR_INVALID_ARG
    assert _call(lib, gamma=sv.SV_MAX_GAMMA + 1) == sv.SV_ERR_INVALID_ARG
    assert _call(lib, V=0) == sv.SV_ERR_INVALID_ARG
    assert _call(lib, V=sv.SV_MAX_V + 1) == sv.SV_ERR_INVALID_ARG
    assert _call(lib, dtype=7) == sv.SV_ERR_INVALID_ARG
    assert _call(lib, ptr=0) == sv.SV_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    assert _call(lib, B=0, ptr=0) == sv.SV_OK
    assert sv.last_launch_count() == 0


def test_size_queries_validate_arguments(lib):
    n = ctypes.c_size_t(0)
    assert lib.spec_verify_workspace_size(1, 0, 10, 0, ctypes.byref(n)) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_host_staging_size(1, 1, 10, 5, ctypes.byref(n)) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_verify_workspace_size(1, 1, 10, 0, None) == sv.SV_ERR_INVALID_ARG


def test_no_device_is_reported_not_faked(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    n = ctypes.c_size_t(0)
    assert lib.spec_verify_workspace_size(1, 1, 10, 0, ctypes.byref(n)) == sv.SV_ERR_UNSUPPORTED
    assert _call(lib) == sv.SV_ERR_UNSUPPORTED


def test_commit_rejects_bad_arguments_before_launch(lib):
    p = 0x1000
    assert lib.spec_commit(p, p, -1, 4, p, 16, p, p, p, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_commit(p, p, 2, 0, p, 16, p, p, p, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_commit(p, p, 2, 65, p, 16, p, p, p, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_commit(p, p, 2, 4, p, 0, p, p, p, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_commit(0, p, 2, 4, p, 16, p, p, p, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_commit(p, p, 2, 4, p, 16, 0, p, p, None) == sv.SV_ERR_INVALID_ARG
    assert lib.spec_commit(p, p, 0, 4, p, 16, p, p, p, None) == sv.SV_OK


def test_ngram_rejects_bad_arguments_before_launch(lib):
    p = 0x1000
    ok = dict(B=2, max_len=16, gamma=4, n_min=2, n_max=5)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.spec_ngram_propose(kw.get("buf", p), a["B"], a["max_len"], kw.get("lens", p), a["gamma"],
                                      a["n_min"], a["n_max"], p, p, p, None)
    assert call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert call(max_len=0) == sv.SV_ERR_INVALID_ARG
    assert call(gamma=0) == sv.SV_ERR_INVALID_ARG
    assert call(n_min=0) == sv.SV_ERR_INVALID_ARG
    assert call(n_min=4, n_max=3) == sv.SV_ERR_INVALID_ARG
    assert call(n_max=17) == sv.SV_ERR_INVALID_ARG
    assert call(buf=0) == sv.SV_ERR_INVALID_ARG
    assert call(B=0) == sv.SV_OK
