"""The C ABI without a GPU: the library loads, exports every entry point that
include/bra.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import vision_transformer_sparse_route_b300 as bra
from vision_transformer_sparse_route_b300 import build as bra_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bra.h")


@pytest.fixture(scope="module")
def lib():
    bra_build.build()
    return bra._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bra_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ["bra_route", "bra_attend", "bra_forward", "bra_idx_workspace_bytes",
                 "bra_device_status", "bra_status_string", "bra_abi_version"]:
        assert must in names
    assert set(names) == set(bra.SYMBOLS), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.check_output(["nm", "-D", "--defined-only", bra.library_path()]).decode()
    exported = set(re.findall(r"\bT (bra_[a-z_]+)\b", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_version_and_strings(lib):
    assert lib.bra_abi_version() == 103
    assert bra.status_string(0) == "ok"
    assert "unsupported" in bra.status_string(2)
    assert bra.status_string(99) == "unknown status"


def test_workspace_bytes(lib):
    assert lib.bra_idx_workspace_bytes(64, 7, 4) == 64 * 49 * 4 * 4
    assert lib.bra_idx_workspace_bytes(0, 7, 4) == 0
    assert lib.bra_idx_workspace_bytes(1, 0, 4) == 0


# Fake, 16-byte aligned, non-overlapping "device" addresses: argument checks
# reject these calls before any CUDA call, so nothing is dereferenced.
A, B_, C_, D_, E_, F_ = (ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(6))
NULL = None


def route(lib, q=A, k=B_, B=1, H=14, W=14, C=64, S=7, topk=4, dtype=1, idx=C_):
    return lib.bra_route(q, k, B, H, W, C, S, topk, dtype, idx, NULL, NULL)


def attend(lib, q=A, k=B_, v=C_, idx=D_, B=1, H=14, W=14, C=64, heads=2, S=7, topk=4,
           w=E_, ks=5, dtype=1, out=F_):
    return lib.bra_attend(q, k, v, idx, B, H, W, C, heads, S, topk, w, NULL, ks, dtype,
                          out, NULL)


def test_route_argument_errors(lib):
    assert route(lib, q=NULL) == bra.BRA_ERR_INVALID_ARG
    assert route(lib, idx=NULL) == bra.BRA_ERR_INVALID_ARG
    assert route(lib, H=15) == bra.BRA_ERR_INVALID_ARG          # H % S
    assert route(lib, topk=50) == bra.BRA_ERR_INVALID_ARG       # topk > S^2
    assert route(lib, topk=0) == bra.BRA_ERR_INVALID_ARG
    assert route(lib, dtype=7) == bra.BRA_ERR_INVALID_ARG
    assert route(lib, q=ctypes.c_void_p(0x10000004)) == bra.BRA_ERR_INVALID_ARG  # misaligned
    assert route(lib, C=60) == bra.BRA_ERR_UNSUPPORTED          # 16-byte channel groups
    assert route(lib, C=96) == bra.BRA_ERR_UNSUPPORTED          # 12 groups: not a power of 2
    assert route(lib, C=512) == bra.BRA_ERR_UNSUPPORTED         # 64 groups: more than 32
    assert route(lib, H=66, W=66, S=33, topk=1) == bra.BRA_ERR_UNSUPPORTED  # S^2 > 1024
    assert route(lib, B=0, q=NULL, k=NULL, idx=NULL) == bra.BRA_OK  # empty batch


def test_attend_argument_errors(lib):
    assert attend(lib, v=NULL) == bra.BRA_ERR_INVALID_ARG
    assert attend(lib, w=NULL) == bra.BRA_ERR_INVALID_ARG
    assert attend(lib, heads=3) == bra.BRA_ERR_INVALID_ARG      # C % heads
    assert attend(lib, ks=4) == bra.BRA_ERR_INVALID_ARG         # even kernel
    assert attend(lib, out=A) == bra.BRA_ERR_INVALID_ARG        # out aliases q
    assert attend(lib, ks=9) == bra.BRA_ERR_UNSUPPORTED
    assert attend(lib, heads=1) == bra.BRA_ERR_UNSUPPORTED      # bf16 needs d == 32
    assert attend(lib, C=96, heads=3) == bra.BRA_ERR_UNSUPPORTED  # bf16 needs C % 64
    assert attend(lib, dtype=0, C=256, heads=2) == bra.BRA_ERR_UNSUPPORTED  # f32 d <= 64
    assert attend(lib, B=0, q=NULL, k=NULL, v=NULL, idx=NULL, w=NULL, out=NULL) == bra.BRA_OK


def test_forward_argument_errors(lib):
    f = lib.bra_forward
    assert f(A, B_, C_, 1, 14, 14, 64, 2, 7, 4, E_, NULL, 5, 1, NULL, F_, NULL) == \
        bra.BRA_ERR_INVALID_ARG  # no workspace
    assert f(A, B_, C_, 1, 14, 14, 64, 2, 7, 4, E_, NULL, 5, 1, A, F_, NULL) == \
        bra.BRA_ERR_INVALID_ARG  # workspace overlaps q
    assert f(None, None, None, 0, 14, 14, 64, 2, 7, 4, None, None, 5, 1, None, None,
             None) == bra.BRA_OK


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(bra, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(bra, "_lib", None)
    with pytest.raises(ImportError):
        bra._load()


def test_wait_timeout_check_rejects_bad_limits(lib):
    assert lib.bra_check_wait_timeout(0, NULL) == bra.BRA_ERR_INVALID_ARG
    assert lib.bra_check_wait_timeout(999, NULL) == bra.BRA_ERR_INVALID_ARG
    assert lib.bra_check_wait_timeout(1_000_000_001, NULL) == bra.BRA_ERR_INVALID_ARG


def test_projection_argument_errors(lib):
    f = lib.bra_qkv_project
    G = ctypes.c_void_p(0x70000000)
    assert f(NULL, B_, NULL, 100, 64, 1, C_, D_, E_, NULL) == bra.BRA_ERR_INVALID_ARG
    assert f(A, B_, NULL, -1, 64, 1, C_, D_, E_, NULL) == bra.BRA_ERR_INVALID_ARG
    assert f(A, B_, NULL, 100, 64, 1, A, D_, E_, NULL) == bra.BRA_ERR_INVALID_ARG  # q aliases x
    assert f(A, B_, NULL, 100, 64, 1, C_, C_, E_, NULL) == bra.BRA_ERR_INVALID_ARG  # q == k
    assert f(A, B_, NULL, 100, 64, 1, ctypes.c_void_p(0x30000008), D_, E_, NULL) == \
        bra.BRA_ERR_INVALID_ARG  # misaligned
    assert f(A, B_, NULL, 100, 96, 1, C_, D_, E_, NULL) == bra.BRA_ERR_UNSUPPORTED
    assert f(A, B_, NULL, 100, 512, 1, C_, D_, G, NULL) == bra.BRA_ERR_UNSUPPORTED
    assert f(A, B_, NULL, 100, 64, 0, C_, D_, E_, NULL) == bra.BRA_ERR_UNSUPPORTED  # f32
    assert f(NULL, NULL, NULL, 0, 64, 1, NULL, NULL, NULL, NULL) == bra.BRA_OK  # empty


G1, G2, G3, G4, G5 = (ctypes.c_void_p(0x90000000 + 0x08000000 * i) for i in range(5))


def attend_backward(lib, q=A, k=B_, v=C_, idx=D_, B=1, H=14, W=14, C=64, heads=2, S=7,
                    topk=4, w=E_, ks=5, dout=F_, dtype=1, dq=G1, dk=G2, dv=G3, dw=G4, db=G5):
    return lib.bra_attend_backward(q, k, v, idx, B, H, W, C, heads, S, topk, w, ks, dout,
                                   dtype, dq, dk, dv, dw, db, NULL)


def test_attend_backward_argument_errors(lib):
    assert attend_backward(lib, dout=NULL) == bra.BRA_ERR_INVALID_ARG
    assert attend_backward(lib, dw=NULL) == bra.BRA_ERR_INVALID_ARG
    assert attend_backward(lib, heads=3) == bra.BRA_ERR_INVALID_ARG   # C % heads
    assert attend_backward(lib, ks=4) == bra.BRA_ERR_INVALID_ARG      # even kernel
    assert attend_backward(lib, H=15) == bra.BRA_ERR_INVALID_ARG      # H % S
    assert attend_backward(lib, dq=A) == bra.BRA_ERR_INVALID_ARG      # dq aliases q
    assert attend_backward(lib, dk=G1) == bra.BRA_ERR_INVALID_ARG     # dk aliases dq
    assert attend_backward(lib, db=G4) == bra.BRA_ERR_INVALID_ARG     # db aliases dw
    assert attend_backward(lib, ks=9) == bra.BRA_ERR_UNSUPPORTED
    assert attend_backward(lib, C=256, heads=2) == bra.BRA_ERR_UNSUPPORTED  # d = 128 > 64
    assert attend_backward(lib, B=0, q=NULL, k=NULL, v=NULL, idx=NULL, w=NULL, dout=NULL,
                           dq=NULL, dk=NULL, dv=NULL, dw=NULL, db=NULL) == bra.BRA_OK
