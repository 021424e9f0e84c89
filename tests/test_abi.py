"""The C-ABI library builds for sm_103a, loads, and exports every symbol the
header declares (CPU only: no compute call is made)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa.h")


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^(?:csa_status_t|size_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from compressed_sparse_attention_compress_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_six_calls():
    names = _declared()
    for n in ["csa_compress", "csa_indexer_topk", "csa_sparse_attn_fwd", "hca_attn_fwd", "window_attn_fwd",
              "csa_indexer_kl"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_workspace_query(lib):
    lib.csa_status_string.restype = ctypes.c_char_p
    assert lib.csa_status_string(0) == b"CSA_OK"
    assert lib.csa_status_string(-6) == b"CSA_ERR_DEVICE_BOUNDS"
    lib.csa_indexer_kl_workspace.restype = ctypes.c_size_t
    assert lib.csa_indexer_kl_workspace(1000) >= 8000
    assert lib.csa_indexer_kl_workspace(0) == 0


def test_null_handle_is_rejected_before_any_launch(lib):
    # argument checks run on the host before anything touches the device
    lib.csa_compress.restype = ctypes.c_int
    assert lib.csa_compress(None, *([None] * 5), 0, 0, 0, 0, 0, 0, 0, None, None) == -1
    lib.csa_create.restype = ctypes.c_int
    assert lib.csa_create(0, None) == -1


def _params(name):
    text = open(HEADER).read()
    m = re.search(r"^(?:csa_status_t)\s+" + name + r"\s*\((.*?)\);", text, flags=re.M | re.S)
    return [p.strip() for p in m.group(1).replace("\n", " ").split(",")]


def _null_args(params):
    out = []
    for p in params:
        if "*" in p or p.startswith(("csa_handle_t", "cudaStream_t")):
            out.append(ctypes.c_void_p(None))
        elif p.startswith("float"):
            out.append(ctypes.c_float(0.0))
        elif p.startswith("int64_t"):
            out.append(ctypes.c_int64(0))
        elif p.startswith("size_t"):
            out.append(ctypes.c_size_t(0))
        else:  # int, csa_dtype_t
            out.append(ctypes.c_int(0))
    return out


def test_every_call_rejects_a_null_handle_on_the_host(lib):
    # the header's error rule: host-visible argument errors return CSA_ERR_INVALID_ARG
    # before any launch -- checked for every call that takes a handle, with all
    # other arguments zero or null, so nothing here touches a device
    text = open(HEADER).read()
    names = re.findall(r"^csa_status_t\s+(\w+)\s*\(\s*csa_handle_t", text, flags=re.M)
    names = [n for n in names if n != "csa_destroy"]
    assert len(names) >= 18, names
    for n in names:
        fn = getattr(lib, n)
        fn.restype = ctypes.c_int
        assert fn(*_null_args(_params(n))) == -1, n
