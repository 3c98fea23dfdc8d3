"""The C-ABI library builds, loads on a machine without a GPU, and exports every symbol that
include/dsa.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*DSA_API\s+(?:const\s+)?\w+\s*\*?\s*(dsa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_indexer_e4m3_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dsa_index_score", "dsa_topk", "dsa_index_topk", "dsa_topk_workspace_size",
              "dsa_index_topk_workspace_size", "dsa_get_device_error", "dsa_status_string", "dsa_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dsa.h but not exported"


def test_library_exports_nothing_else(lib):
    import subprocess

    from sparse_attention_indexer_e4m3_gb300 import library_path

    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True, text=True).stdout
    exported = sorted(set(re.findall(r"\b(dsa_\w+)\b", out)))
    assert exported == declared_functions()


def test_c_consumer_compiles_and_links(lib, tmp_path):
    """The header is plain C: a C99 program (pedantic, warnings as errors) that takes the address
    of every function dsa.h declares (as a generic function pointer) compiles against it and links
    against the built library."""
    import shutil
    import subprocess

    from sparse_attention_indexer_e4m3_gb300 import library_path

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "consumer.c"
    src.write_text('#include "dsa.h"\n#include <stdio.h>\n\ntypedef void (*fn_t)(void);\n\nint main(void) {\n'
                   "  const fn_t fns[] = {\n" +
                   "".join(f"      (fn_t)&{n},\n" for n in names) +
                   '  };\n  printf("%d %s\\n", (int)(sizeof(fns) / sizeof(fns[0])), dsa_status_string(DSA_OK));\n'
                   "  return 0;\n}\n")
    so = library_path()
    exe = tmp_path / "consumer"
    cmd = [cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-o", str(exe), "-L", os.path.dirname(so), "-l:" + os.path.basename(so),
           "-Wl,-rpath," + os.path.dirname(so), "-Wl,--allow-shlib-undefined"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_without_gpu(lib):
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    assert lib.dsa_status_string(0) == b"DSA_OK"
    assert lib.dsa_status_string(5) == b"DSA_ERR_TIMEOUT"
    assert lib.dsa_status_string(99) == b"DSA_ERR_UNKNOWN"
    assert lib.dsa_version() == 10000


def test_argument_checks_return_before_any_device_work(lib):
    """Invalid arguments are rejected synchronously (these checks need no GPU)."""
    lib.dsa_index_score.restype = ctypes.c_int
    p = ctypes.c_void_p
    # unsupported head count / head dim
    assert lib.dsa_index_score(None, None, None, None, None, None, 4, 4, 3, 128, None, None) == 2
    assert lib.dsa_index_score(None, None, None, None, None, None, 4, 4, 64, 96, None, None) == 2
    # negative sizes
    assert lib.dsa_index_score(None, None, None, None, None, None, -1, 4, 64, 128, None, None) == 1
    # null inputs with T > 0
    assert lib.dsa_index_score(None, None, None, None, None, None, 4, 4, 64, 128, None, None) == 1
    # misaligned q
    buf = ctypes.create_string_buffer(64)
    mis = p(ctypes.addressof(buf) + 1)
    ok = p(ctypes.addressof(buf))
    assert lib.dsa_index_score(mis, ok, ok, ok, ok, ok, 1, 1, 4, 64, ok, None) == 1
    # top-k limits
    lib.dsa_topk.argtypes = [p, p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p, ctypes.c_size_t, p]
    assert lib.dsa_topk(ok, ok, ok, 1, 1, 0, ok, None, 0, None) == 2
    assert lib.dsa_topk(ok, ok, ok, 1, 1, 4096, ok, None, 0, None) == 2
    # zero tokens: nothing to do, nothing launched
    assert lib.dsa_topk(None, None, None, 0, 10, 8, None, None, 0, None) == 0
    # key quantiser: head dim, negative rows, null / misaligned pointers, zero rows
    lib.dsa_quantize_k.argtypes = [p, ctypes.c_int, ctypes.c_int, p, p, p]
    lib.dsa_quantize_k.restype = ctypes.c_int
    assert lib.dsa_quantize_k(ok, 4, 96, ok, ok, None) == 2
    assert lib.dsa_quantize_k(ok, -1, 128, ok, ok, None) == 1
    assert lib.dsa_quantize_k(None, 4, 128, ok, ok, None) == 1
    assert lib.dsa_quantize_k(mis, 4, 128, ok, ok, None) == 1
    assert lib.dsa_quantize_k(ok, 4, 64, mis, ok, None) == 1
    assert lib.dsa_quantize_k(None, 0, 64, None, None, None) == 0
    # sparse attention: head dim, negative sizes, null / misaligned pointers, zero tokens
    i = ctypes.c_int
    lib.dsa_sparse_attn.argtypes = [p, p, p, p, i, i, i, i, i, ctypes.c_float, p, p, p]
    lib.dsa_sparse_attn.restype = i
    assert lib.dsa_sparse_attn(ok, ok, None, ok, 2, 4, 1, 96, 4, 1.0, ok, None, None) == 2
    assert lib.dsa_sparse_attn(ok, ok, None, ok, -1, 4, 1, 64, 4, 1.0, ok, None, None) == 1
    assert lib.dsa_sparse_attn(ok, ok, None, ok, 2, 4, 0, 64, 4, 1.0, ok, None, None) == 1
    assert lib.dsa_sparse_attn(ok, ok, None, None, 2, 4, 1, 64, 4, 1.0, ok, None, None) == 1
    assert lib.dsa_sparse_attn(ok, p(ctypes.addressof(buf) + 2), None, ok, 2, 4, 1, 64, 4, 1.0, ok, None, None) == 1
    assert lib.dsa_sparse_attn(ok, ok, mis, ok, 2, 4, 1, 64, 4, 1.0, ok, None, None) == 1
    assert lib.dsa_sparse_attn(ok, ok, None, ok, 2, 4, 1, 64, 4, 1.0, ok, mis, None) == 1  # misaligned lse
    assert lib.dsa_sparse_attn(None, None, None, None, 0, 4, 1, 64, 4, 1.0, None, None, None) == 0
    # attention backward: head dims without a kernel, negative sizes, null pointers
    lib.dsa_sparse_attn_bwd.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, ctypes.c_float, p, p, p, p]
    lib.dsa_sparse_attn_bwd.restype = i
    bwd = lib.dsa_sparse_attn_bwd
    assert bwd(ok, ok, None, ok, ok, ok, ok, 2, 4, 4, 64, 4, 1.0, ok, ok, None, None) == 2
    assert bwd(ok, ok, None, ok, ok, ok, ok, 2, 4, 4, 512, 4, 1.0, ok, ok, None, None) == 2
    assert bwd(ok, ok, None, ok, ok, ok, ok, -1, 4, 4, 128, 4, 1.0, ok, ok, None, None) == 1
    assert bwd(ok, ok, None, ok, ok, None, ok, 2, 4, 4, 128, 4, 1.0, ok, ok, None, None) == 1  # no lse
    assert bwd(ok, ok, None, ok, ok, ok, ok, 2, 4, 4, 128, 4, 1.0, ok, None, None, None) == 1  # no dkv
    assert bwd(mis, ok, None, ok, ok, ok, ok, 2, 4, 4, 128, 4, 1.0, ok, ok, None, None) == 1   # q misaligned
    # K-resident scorer: unsupported shape, workspace size rule, null inputs
    lib.dsa_index_score_kres_workspace_size.argtypes = [i, i, i, i]
    lib.dsa_index_score_kres_workspace_size.restype = ctypes.c_size_t
    assert lib.dsa_index_score_kres_workspace_size(100, 1000, 3, 128) == 0
    assert lib.dsa_index_score_kres_workspace_size(100, 1000, 64, 128) == lib.dsa_index_score_kres_workspace_size(
        100, 5, 64, 64)  # depends on T and H only
    assert lib.dsa_index_score_kres_workspace_size(100, 1000, 64, 128) >= 256 + 100 * 8
    lib.dsa_index_score_kres.argtypes = [p, p, p, p, p, p, i, i, i, i, p, p, ctypes.c_size_t, p]
    lib.dsa_index_score_kres.restype = i
    assert lib.dsa_index_score_kres(None, None, None, None, None, None, 4, 4, 3, 128, None, None, 0, None) == 2
    assert lib.dsa_index_score_kres(None, None, None, None, None, None, 4, 4, 64, 128, None, None, 0, None) == 1
