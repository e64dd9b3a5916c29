"""The C-ABI library builds, loads and exports every entry point declared in
include/*.h; host-side argument checks return their status codes without
touching a GPU (they run before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(spec_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    from token_tree_verification_gb300 import build, binding
    build.build()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"spec_build_tree_mask", "spec_tree_attn", "spec_tree_verify"} <= names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(-12, 1):
        s = lib.spec_status_string(code).decode()
        assert s.startswith("SPEC_")
    assert b"unknown" in lib.spec_status_string(42)


def test_bounds_checked_build_exports_the_same_entry_points(lib):
    """The -DSPEC_CHECKED debug build compiles from the same sources, exports
    every declared entry point and says which build it is."""
    from token_tree_verification_gb300 import build
    path = build.build(checked=True)
    assert os.path.basename(path) == "libspec_tree_checked.so"
    chk = ctypes.CDLL(path)
    for n in declared_symbols():
        assert hasattr(chk, n), n
    chk.spec_build_checked.restype = ctypes.c_int
    lib.spec_build_checked.restype = ctypes.c_int
    assert chk.spec_build_checked() == 1
    assert lib.spec_build_checked() == 0
    chk.spec_status_string.restype = ctypes.c_char_p
    assert chk.spec_status_string(-12).decode().startswith("SPEC_ERR_INDEX")


def test_workspace_sizes(lib):
    assert lib.spec_tree_attn_workspace_size(1, 64, 32, 32, 128, 2048) == 0  # merged on chip
    s1 = lib.spec_tree_verify_workspace_size(1, 64, 32000)
    s2 = lib.spec_tree_verify_workspace_size(16, 900, 32000)
    assert s1 > 0 and s2 > s1 and s2 % 256 == 0
    assert lib.spec_tree_verify_workspace_size(0, 1, 1) == 0


def test_host_side_validation(lib):
    P = ctypes.c_void_p
    fake = P(0x1000)   # never dereferenced: validation fails before any launch
    # null pointers
    assert lib.spec_build_tree_mask(None, fake, 1, 1, fake, fake, fake, None) == -1
    assert lib.spec_tree_attn(fake, fake, None, fake, 1, 1, 1, 1, 1, 128, 8, 8, fake, fake, fake,
                              0.0, None, 0, fake, None) == -1
    # sizes
    assert lib.spec_build_tree_mask(fake, fake, 0, 1, fake, fake, fake, None) == -2
    assert lib.spec_build_tree_mask(fake, fake, 1, 129, fake, fake, fake, None) == -2
    assert lib.spec_tree_attn(fake, fake, fake, fake, 1, 1, 1, 4, 4, 96, 8, 8, fake, fake, fake,
                              0.0, None, 0, fake, None) == -2          # D = 96 unsupported
    assert lib.spec_tree_attn(fake, fake, fake, fake, 1, 1, 1, 12, 4, 64, 8, 8, fake, fake, fake,
                              0.0, None, 0, fake, None) == -2          # G = 3 unsupported
    assert lib.spec_tree_attn(fake, fake, fake, fake, 7, 1, 1, 4, 4, 64, 8, 8, fake, fake, fake,
                              0.0, None, 0, fake, None) == -3          # dtype
    assert lib.spec_tree_attn(P(0x1004), fake, fake, fake, 1, 1, 1, 4, 4, 64, 8, 8, fake, fake,
                              fake, 0.0, None, 0, fake, None) == -11   # alignment
    # verify: workspace, temperature, missing draft rows
    V = 1000
    ws = lib.spec_tree_verify_workspace_size(1, 8, V)
    args = [fake, fake, fake, fake, fake, 1, 8, V]
    outs = [fake, fake, fake, fake, 4]
    assert lib.spec_tree_verify(*args, ctypes.c_float(0.0), 0, *outs, None, 0, fake, None) == -7
    assert lib.spec_tree_verify(*args, ctypes.c_float(0.0), 0, *outs, fake, ws - 1, fake, None) == -7
    assert lib.spec_tree_verify(*args, ctypes.c_float(-1.0), 0, *outs, fake, ws, fake, None) == -2
    assert lib.spec_tree_verify(fake, None, fake, fake, fake, 1, 8, V, ctypes.c_float(0.7), 0,
                                *outs, fake, ws, fake, None) == -1
    assert lib.spec_tree_verify(*args, ctypes.c_float(float("nan")), 0, *outs, fake, ws, fake,
                                None) == -2


def test_host_side_validation_of_the_other_entry_points(lib):
    P, F32, U64, I, SZ = ctypes.c_void_p, ctypes.c_float, ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
    fake = P(0x1000)   # never dereferenced: validation fails before any launch
    # top-p verification: top_p must be > 0 (NaN rejected); the nucleus search
    # covers V <= 131072
    V = 1000
    ws = lib.spec_tree_verify_workspace_size(1, 8, V)
    outs = [fake, fake, fake, fake, 4]
    f = lib.spec_tree_verify_top_p
    assert f(fake, fake, fake, fake, fake, 1, 8, V, F32(0.7), F32(0.0), 0, *outs, fake, ws, fake, None) == -2
    assert f(fake, fake, fake, fake, fake, 1, 8, V, F32(0.7), F32(float("nan")), 0, *outs, fake, ws, fake,
             None) == -2
    big = 131073
    wsb = lib.spec_tree_verify_workspace_size(1, 8, big)
    assert f(fake, fake, fake, fake, fake, 1, 8, big, F32(0.7), F32(0.9), 0, *outs, fake, wsb, fake, None) == -2
    assert f(fake, None, fake, fake, fake, 1, 8, V, F32(0.7), F32(0.9), 0, *outs, fake, ws, fake, None) == -1
    # KV compaction
    g = lib.spec_kv_compact
    kv = lambda k=fake, dtype=1, D=128, W=4: g(k, fake, dtype, 1, 2, D, 256, fake, fake, fake, fake, W,
                                               fake, fake, None)
    assert g(None, fake, 1, 1, 2, 128, 256, fake, fake, fake, fake, 4, fake, fake, None) == -1
    assert kv(dtype=7) == -3
    assert kv(D=4) == -2                    # D < 8
    assert kv(W=0) == -2                    # no output row
    assert kv(W=129) == -2                  # more rows than a tree has nodes
    assert kv(dtype=0, D=1024, W=128) == -2  # 127 rows of 4 KB, K and V: beyond shared memory
    assert kv(k=P(0x1008)) == -11
    # expansion
    e = lib.spec_tree_expand
    ex = lambda F=4, V=64, w=5, t=0.7: e(fake, fake, fake, fake, F, V, w, F32(t), 1, fake, fake, fake, None)
    assert e(None, fake, fake, fake, 4, 64, 5, F32(0.7), 1, fake, fake, fake, None) == -1
    assert ex(F=0) == -2 and ex(w=0) == -2 and ex(w=17) == -2 and ex(V=4, w=5) == -2
    assert ex(t=float("nan")) == -2 and ex(t=-1.0) == -2
    # pruning
    p = lib.spec_tree_prune
    pr = lambda B=1, keep=64: p(fake, fake, fake, fake, B, keep, fake, fake, fake, fake, fake, None)
    assert p(None, fake, fake, fake, 1, 64, fake, fake, fake, fake, fake, None) == -1
    assert pr(B=0) == -2 and pr(keep=0) == -2 and pr(keep=129) == -2
    # the static entry point refuses a batch beyond its fixed array before touching a device
    s = lib.spec_tree_verify_static
    s.argtypes = [P, P, P, P, P, I, I, I, F32, U64, P, P, P, P, I, P, P]
    s.restype = I
    B, T = 400, 40000
    assert lib.spec_tree_verify_workspace_size(B, T, 32000) > 256 * 1024
    assert s(fake, fake, fake, fake, fake, B, T, 32000, F32(0.7), 0, *outs, fake, None) == -7
