"""The C ABI loads and exports every function include/qrita.h declares, and its
argument checks answer without touching a GPU (no compute calls here)."""

import ctypes
import os
import re

import pytest

from top_selection_row_gb300.build import LIB_PATH, build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(LIB_PATH):
        build_library()
    import top_selection_row_gb300 as q

    return q.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qrita.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(qrita_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_function_is_exported(L):
    names = declared_functions()
    assert len(names) >= 6
    import top_selection_row_gb300._lib as bind

    assert sorted(bind.EXPORTED) == names
    for n in names:
        assert hasattr(L, n), n


def test_version_and_strerror(L):
    assert L.qrita_version() >= 100
    for code in range(4):
        assert L.qrita_strerror(code)
    assert b"unknown" in L.qrita_strerror(99)


NULL = ctypes.c_void_p(0)
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every case fails validation first


@pytest.mark.parametrize(
    "logits,dtype,B,V,mask,flags",
    [
        (FAKE, 7, 1, 10, FAKE, 0),             # unknown dtype
        (FAKE, 0, -1, 10, FAKE, 0),            # negative B
        (FAKE, 0, 1, 0, FAKE, 0),              # V = 0
        (FAKE, 0, 1, 2**31, FAKE, 0),          # V above 2^31 - 1
        (NULL, 0, 1, 10, FAKE, 0),             # null logits
        (FAKE, 0, 1, 10, NULL, 0),             # null mask
        (ctypes.c_void_p(0x1002), 0, 1, 10, FAKE, 0),  # fp32 pointer not 4-byte aligned
        (ctypes.c_void_p(0x1001), 1, 1, 10, FAKE, 0),  # bf16 pointer not 2-byte aligned
        (FAKE, 0, 1, 10, FAKE, 0x1000),        # unknown flag bit
    ],
)
def test_invalid_arguments_are_rejected(L, logits, dtype, B, V, mask, flags):
    rc = L.qrita_select_ex(logits, dtype, B, V, NULL, NULL, mask, NULL, flags, NULL, NULL)
    assert rc == 1
    if flags == 0:
        assert L.qrita_select(logits, dtype, B, V, NULL, NULL, mask, NULL) == 1


def test_empty_batch_is_ok_and_launches_nothing(L):
    assert L.qrita_select(NULL, 0, 0, 100, NULL, NULL, NULL, NULL) == 0
    assert L.qrita_select_ex(NULL, 1, 0, 5, NULL, NULL, NULL, NULL, 0, NULL, NULL) == 0


def test_host_staging_bytes(L):
    # sections: logits, k, p, mask, each rounded up to 256 bytes
    def up(x):
        return (x + 255) // 256 * 256

    for dt, s in ((0, 4), (1, 2)):
        for B, V in ((1, 1), (3, 1000), (64, 128256)):
            assert L.qrita_host_staging_bytes(dt, B, V) == up(B * V * s) + 2 * up(B * 4) + up(B * V)
    assert L.qrita_host_staging_bytes(5, 1, 1) == 0
    assert L.qrita_host_staging_bytes(0, 1, 0) == 0


def test_host_entry_rejects_short_staging(L):
    rc = L.qrita_select_host(FAKE, 0, 2, 10, NULL, NULL, FAKE, FAKE, ctypes.c_size_t(16), NULL)
    assert rc == 1
    rc = L.qrita_select_host(FAKE, 0, 2, 10, NULL, NULL, FAKE, NULL, ctypes.c_size_t(1 << 20), NULL)
    assert rc == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import top_selection_row_gb300._lib as bind

    monkeypatch.setattr(bind, "_lib", None)
    monkeypatch.setattr(bind, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        bind.lib()
