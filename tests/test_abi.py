"""The C ABI without a GPU: the library builds and loads, exports exactly what
include/s2.h declares, and rejects bad arguments before touching the device.

No call here reaches a kernel: every argument error is detected on the host,
so these tests use fake (never dereferenced) pointer values.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "s2.h")


@pytest.fixture(scope="module")
def lib():
    from sketch_compressed_sparse_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^S2_API\s+[^(]*?\b(s2_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for fn in ["s2_encode", "s2_encode_batched", "s2_reduce", "s2_decode_dense", "s2_decode_compact",
               "s2_decode_workspace_size", "s2_hash", "s2_status_string"]:
        assert fn in names


def test_every_declared_symbol_is_exported(lib):
    for fn in declared_functions():
        assert hasattr(lib, fn), f"{fn} declared in s2.h but not exported"


def test_only_declared_symbols_are_exported():
    import subprocess

    from sketch_compressed_sparse_gb300 import build

    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("s2_")}
    assert exported == set(declared_functions())


class Params(ctypes.Structure):
    _fields_ = [("d", ctypes.c_uint32), ("w", ctypes.c_uint32), ("seed", ctypes.c_uint32)]


def _fn(lib, name, argtypes):
    f = getattr(lib, name)
    f.argtypes = argtypes
    f.restype = ctypes.c_int
    return f


VP, U32, U64, I32, F32, SZ = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
OK, INVALID, ALIGN, UNSUP = 0, 1, 2, 3
A = 0x10000000  # fake, 256-aligned device addresses; never dereferenced


def test_status_strings_and_version(lib):
    lib.s2_status_string.restype = ctypes.c_char_p
    lib.s2_status_string.argtypes = [I32]
    assert lib.s2_status_string(0) == b"S2_OK"
    assert lib.s2_status_string(2) == b"S2_ERR_ALIGNMENT"
    assert lib.s2_status_string(99) == b"S2_UNKNOWN_STATUS"
    lib.s2_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.s2_version()


def test_encode_argument_errors(lib):
    enc = _fn(lib, "s2_encode_batched", [VP, I32, U32, U64, Params, VP, VP, VP])
    good = Params(3, 64, 0)
    assert enc(A, 0, 2, 1024, Params(0, 64, 0), A + 2**20, A + 2**21, None) == INVALID  # d = 0
    assert enc(A, 0, 2, 1024, Params(17, 64, 0), A + 2**20, A + 2**21, None) == INVALID  # d > 16
    assert enc(A, 0, 2, 1024, Params(3, 0, 0), A + 2**20, A + 2**21, None) == INVALID  # w = 0
    assert enc(A, 0, 2, 1024, Params(3, 2**31 + 1, 0), A + 2**20, A + 2**21, None) == INVALID
    assert enc(A, 7, 2, 1024, good, A + 2**20, A + 2**21, None) == INVALID  # bad dtype
    assert enc(A, 0, 2, 2**32, good, A + 2**40, A + 2**41, None) == UNSUP  # n >= 2^32
    assert enc(None, 0, 2, 1024, good, A + 2**20, A + 2**21, None) == INVALID  # null grad
    assert enc(A + 4, 0, 2, 1024, good, A + 2**20, A + 2**21, None) == ALIGN
    assert enc(A, 0, 2, 1024, good, A + 2**20 + 8, A + 2**21, None) == ALIGN
    assert enc(A, 0, 2, 1024, good, A + 4096, A + 2**21, None) == INVALID  # bitmaps overlap grad (8 KB)
    assert enc(A, 0, 2, 1024, good, A + 2**20, A + 2**20 + 128, None) == INVALID  # sketch overlaps bitmaps
    assert enc(None, 0, 0, 1024, good, None, None, None) == OK  # W = 0: nothing to do


def test_reduce_and_decode_argument_errors(lib):
    red = _fn(lib, "s2_reduce", [VP, VP, U32, U64, Params, VP, VP, VP])
    good = Params(3, 64, 0)
    assert red(A, A + 2**20, 4, 1024, good, A + 2**21, None, None) == INVALID  # null sketch_out
    assert red(A, A + 2**20, 4, 1024, good, A + 2**21 + 4, A + 2**22, None) == ALIGN
    assert red(A, A + 2**20, 4, 1024, good, A + 16, A + 2**22, None) == INVALID  # out overlaps in
    dec = _fn(lib, "s2_decode_dense", [VP, VP, U64, Params, F32, VP, VP])
    assert dec(A, A + 2**20, 1000, good, 1.0, A + 2**21 + 4, None) == ALIGN
    assert dec(A, A + 2**20, 1000, good, 1.0, A + 64, None) == INVALID
    assert dec(A, A + 2**20, 1000, good, 1.0, None, None) == INVALID
    assert dec(A, A + 2**20, 2**32, good, 1.0, A + 2**40, None) == UNSUP
    assert dec(None, None, 0, good, 1.0, None, None) == OK  # n = 0


def test_compact_workspace_and_errors(lib):
    wsz = _fn(lib, "s2_decode_workspace_size", [U64, ctypes.POINTER(SZ)])
    b = SZ()
    assert wsz(0, ctypes.byref(b)) == OK and b.value == 0
    assert wsz(1 << 20, ctypes.byref(b)) == OK and b.value >= 2 * 4 * ((1 << 15) // 256)
    assert wsz(2**32, ctypes.byref(b)) == UNSUP
    assert wsz(10, None) == INVALID
    dc = _fn(lib, "s2_decode_compact", [VP, VP, U64, Params, F32, VP, VP, U64, VP, VP, SZ, VP])
    good = Params(3, 64, 0)
    wsz(100_000, ctypes.byref(b))
    need = b.value
    args = lambda **k: dict(dict(bm=A, sk=A + 2**20, n=100_000, idx=A + 2**21, val=A + 2**22, cap=100_000,
                                 cnt=A + 2**23, ws=A + 2**24, wsb=need), **k)
    call = lambda a: dc(a["bm"], a["sk"], a["n"], good, 1.0, a["idx"], a["val"], a["cap"], a["cnt"], a["ws"],
                        a["wsb"], None)
    assert call(args(wsb=need - 1)) == INVALID  # workspace too small
    assert call(args(cnt=None)) == INVALID
    assert call(args(cnt=A + 2**23 + 4)) == ALIGN
    assert call(args(idx=A + 2**21 + 2)) == ALIGN
    assert call(args(val=A + 2**21 + 16)) == INVALID  # idx and val overlap


def test_compact_noalloc_limits(lib):
    dc = _fn(lib, "s2_decode_compact_noalloc", [VP, VP, U64, Params, F32, VP, VP, U64, VP, VP])
    good = Params(3, 64, 0)
    big = 2**34  # fake, far-apart addresses: nothing overlaps, nothing is dereferenced
    call = lambda n, cnt=A + 4 * big: dc(A, A + big, n, good, 1.0, A + 2 * big, A + 3 * big, 16, cnt, None)
    assert call((1 << 30) + 1) == UNSUP  # beyond the library-owned scratch
    assert call(2**32) == UNSUP
    assert call(1000, cnt=None) == INVALID
    assert call(1000, cnt=A + 4 * big + 4) == ALIGN
    assert dc(A, A + big, 1000, Params(0, 64, 0), 1.0, A + 2 * big, A + 3 * big, 16, A + 4 * big, None) == INVALID


def test_hash_and_pipeline_errors(lib):
    h = _fn(lib, "s2_hash", [VP, U64, Params, VP, VP, VP])
    assert h(A, 10, Params(3, 0, 0), A + 4096, A + 8192, None) == INVALID
    assert h(A + 2, 10, Params(3, 64, 0), A + 4096, A + 8192, None) == ALIGN
    assert h(None, 0, Params(3, 64, 0), None, None, None) == OK
    pws = _fn(lib, "s2_pipeline_workspace_size", [I32, U32, U64, Params, ctypes.POINTER(SZ)])
    b = SZ()
    assert pws(0, 8, 1 << 20, Params(5, 1 << 10, 0), ctypes.byref(b)) == OK
    # grad + bitmaps + sketches + bitmap + sketch + out + the dense decode's
    # workspace (for d = 5: two arrays of n floats, a 256-byte count and one
    # 32-bit id per 512 positions), each rounded to 256 bytes
    assert b.value == (8 * (1 << 22) + 8 * (1 << 17) + 8 * 5 * (1 << 12) + (1 << 17) + 5 * (1 << 12) + (1 << 22)
                       + 2 * (1 << 22) + 256 + 4 * 2048)
    dws = _fn(lib, "s2_decode_dense_workspace_size", [U64, Params, ctypes.POINTER(SZ)])
    c = SZ()
    assert dws(1000, Params(5, 64, 0), ctypes.byref(c)) == OK and c.value == 2 * 4 * 1024 + 256 + 256
    assert dws(1000, Params(3, 64, 0), ctypes.byref(c)) == OK and c.value == 4 * 1024 + 256 + 256
    assert dws(1000, Params(4, 64, 0), ctypes.byref(c)) == OK and c.value == 0
    assert dws(1000, Params(0, 64, 0), ctypes.byref(c)) == INVALID
    dd = _fn(lib, "s2_decode_dense_ws", [VP, VP, U64, Params, F32, VP, VP, SZ, VP])
    ws_ok = 2 * 4 * 1024 + 512
    assert dd(A, A + (1 << 20), 1000, Params(5, 64, 0), 1.0, A + (2 << 20), A + (3 << 20), ws_ok - 1, None) == INVALID
    assert dd(A, A + (1 << 20), 1000, Params(5, 64, 0), 1.0, A + (2 << 20), A + (3 << 20) + 8, ws_ok, None) == ALIGN
    assert dd(A, A + (1 << 20), 1000, Params(5, 64, 0), 1.0, A + (2 << 20), A + (2 << 20) + 16, ws_ok, None) == INVALID
    assert dd(A, A + (1 << 20), 0, Params(5, 64, 0), 1.0, A + (2 << 20), None, 0, None) == OK
    p = _fn(lib, "s2_pipeline_dense_host", [VP, I32, U32, U64, Params, F32, VP, VP, SZ, VP])
    assert p(A, 0, 8, 1 << 20, Params(5, 1 << 10, 0), 1.0, A, A + 16, b.value - 1, None) == INVALID
    assert p(A, 0, 8, 1 << 20, Params(5, 1 << 10, 0), 1.0, A, A + 8, b.value, None) == ALIGN

