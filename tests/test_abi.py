"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/qkmla.h declares, the ctypes mirror of qkmla_decode_args has
the C layout, and host-side validation rejects bad arguments before any
launch."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qkmla.h")


@pytest.fixture(scope="module")
def L():
    from qk_normed_latent_gb300 import build as B
    B.build()
    import qk_normed_latent_gb300 as Q
    return Q


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(qkmla_\w+)\s*\(", txt)))


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ["qkmla_absorb_query", "qkmla_append", "qkmla_decode", "qkmla_decode_workspace_size",
              "qkmla_get_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        getattr(L.lib(), n)


def test_decode_args_layout_matches_c(L):
    fields = [f for f, _ in L.DecodeArgs._fields_]
    src = "#include <stdio.h>\n#include <stddef.h>\n#include \"qkmla.h\"\nint main(void){\n"
    src += 'printf("%zu\\n", sizeof(qkmla_decode_args));\n'
    for f in fields:
        src += f'printf("%zu\\n", offsetof(qkmla_decode_args, {f}));\n'
    src += "return 0;}\n"
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "t")
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(L.DecodeArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(L.DecodeArgs, f).offset == off, f


def test_status_strings_and_version(L):
    assert L.status_string(0) == "ok"
    assert "workspace" in L.status_string(L.ERR_WORKSPACE)
    assert L.lib().qkmla_version() >= 100


def test_host_validation_rejects_before_launch(L):
    lib = L.lib()
    f = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # rows = 0
    assert lib.qkmla_absorb_query(f, f, f, f, 0, 16, 4, 64, 128, 1e-6, 0, f, 0, f, None) == L.ERR_INVALID
    # H % G != 0
    assert lib.qkmla_absorb_query(f, f, f, f, 1, 15, 4, 64, 128, 1e-6, 0, f, 0, f, None) == L.ERR_INVALID
    # null gammas outside plain mode
    assert lib.qkmla_absorb_query(f, None, None, f, 1, 16, 4, 64, 128, 1e-6, 0, f, 0, f, None) == L.ERR_INVALID
    # bad dtype
    assert lib.qkmla_absorb_query(f, f, f, f, 1, 16, 4, 64, 128, 1e-6, 0, f, 7, f, None) == L.ERR_UNSUPPORTED
    # append: N = 0 is a no-op, negative N invalid
    assert lib.qkmla_append(None, None, None, None, None, 0, 4, 128, 64, 32, 1e-6, 0, f, 0, f, 64, None) == L.OK
    assert lib.qkmla_append(f, f, f, None, f, -1, 4, 128, 64, 32, 1e-6, 0, f, 0, f, 64, None) == L.ERR_INVALID
    # decode: null args, zero batch, missing pointers
    assert lib.qkmla_decode(None, None) == L.ERR_INVALID
    a = L.DecodeArgs()
    assert lib.qkmla_decode(ctypes.byref(a), None) == L.ERR_INVALID
    assert lib.qkmla_decode_workspace_size(ctypes.byref(a)) == 0
    assert lib.qkmla_decode_kernel_name(ctypes.byref(a)) == b"invalid"
