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
        (FAKE, 0, 1, 10, FAKE, 0x80000000),    # unknown flag bit
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
    # sizes whose byte count would overflow size_t are refused, not wrapped
    assert L.qrita_host_staging_bytes(0, 2**62, 2**31 - 1) == 0
    assert L.qrita_host_staging_bytes(1, 2**40, 2**30) == 0


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


def _header_probe(tmp_path):
    """Compile a C program against include/qrita.h that prints the row-info
    layout and every constant; returns {name: int}."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    fields = ["mu", "sigma", "threshold", "row_max", "survivors", "path", "rounds_k", "rounds_p", "boundary",
              "n_boundary", "kept", "status", "z", "passes", "reserved"]
    consts = ["QRITA_DTYPE_F32", "QRITA_DTYPE_BF16", "QRITA_OK", "QRITA_EINVAL", "QRITA_EUNSUPPORTED",
              "QRITA_ECUDA", "QRITA_ROW_OK", "QRITA_ROW_NONFINITE", "QRITA_ROW_SEARCH_CAP", "QRITA_ROW_TIMEOUT",
              "QRITA_FLAG_NO_TRUNCATION", "QRITA_FLAG_FORCE_FALLBACK", "QRITA_FLAG_KEY_PIVOTS",
              "QRITA_FLAG_FORCE_RETRY", "QRITA_FLAG_HIST_MISS", "QRITA_FLAG_CLUSTER_SHIFT", "QRITA_FLAG_CLUSTER_SET",
              "QRITA_FLAG_TEST_GIVE_UP", "QRITA_FLAG_NO_KEY_HIST", "QRITA_PATH_KEYHIST",
              "QRITA_FLAG_SEARCH_QUATERNARY", "QRITA_FLAG_SEARCH_BINARY",
              "QRITA_PATH_TOPK", "QRITA_PATH_TOPP", "QRITA_PATH_TRUNC", "QRITA_PATH_HIT", "QRITA_PATH_FALLBACK",
              "QRITA_PATH_OVERFLOW", "QRITA_PATH_KEEP_ALL", "QRITA_PATH_RETRY", "QRITA_PATH_HIST",
              "QRITA_PATH_SAMPLE_T"]
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "qrita.h"', "int main(void) {",
             '  printf("sizeof %zu\\n", sizeof(qrita_row_info_t));']
    lines += [f'  printf("off_{f} %zu\\n", offsetof(qrita_row_info_t, {f}));' for f in fields]
    lines += [f'  printf("size_{f} %zu\\n", sizeof(((qrita_row_info_t*)0)->{f}));' for f in fields]
    lines += [f'  printf("{c} %lld\\n", (long long)({c}));' for c in consts]
    lines += ["  return 0;", "}"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "probe"
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(root, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, timeout=120)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout
    return {k: int(v) for k, v in (ln.split() for ln in out.splitlines())}


def test_row_info_layout_matches_the_header(tmp_path):
    import top_selection_row_gb300 as q

    h = _header_probe(tmp_path)
    dt = q.ROW_INFO_DTYPE
    assert h["sizeof"] == dt.itemsize == 64
    assert list(dt.names) == [k[4:] for k in h if k.startswith("off_")]
    for name in dt.names:
        ftype, off = dt.fields[name][:2]
        assert h[f"off_{name}"] == off, name
        assert h[f"size_{name}"] == ftype.itemsize, name


def test_binding_constants_match_the_header(tmp_path):
    import top_selection_row_gb300 as q

    h = _header_probe(tmp_path)
    for name, v in h.items():
        if not name.startswith("QRITA_") or name == "QRITA_FLAG_CLUSTER_SHIFT":
            continue
        attr = name[len("QRITA_"):]
        assert getattr(q, attr) == v, name
    assert q.flag_cluster(1) == h["QRITA_FLAG_CLUSTER_SET"]
    assert q.flag_cluster(16) == h["QRITA_FLAG_CLUSTER_SET"] | (4 << h["QRITA_FLAG_CLUSTER_SHIFT"])


def test_binding_rejects_bad_host_arguments_before_any_device_work():
    torch = pytest.importorskip("torch")
    import top_selection_row_gb300 as q

    x = torch.zeros(3, 10)
    with pytest.raises(ValueError):
        q.qrita_select(x)  # device entry point: host tensors are refused
    with pytest.raises(ValueError):
        q.qrita_select_host(torch.zeros(10))  # not [B, V]
    with pytest.raises(TypeError):
        q.qrita_select_host(torch.zeros(3, 10, dtype=torch.float16))
    with pytest.raises(ValueError):
        q.qrita_select_host(torch.zeros(10, 3).t())  # not row-major
    with pytest.raises(ValueError):
        q.qrita_select_host(x, k=torch.ones(3, dtype=torch.int64))
    with pytest.raises(ValueError):
        q.qrita_select_host(x, k=torch.ones(2, dtype=torch.int32))
    with pytest.raises(ValueError):
        q.qrita_select_host(x, p=torch.ones(3, dtype=torch.float64))
