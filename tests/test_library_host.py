"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from speculative_decode_gated_gdn_gb300 import lib as L

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gdn_\w+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    return L.load()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"gdn_conv_verify", "gdn_commit", "gdn_flush", "gdn_prefill_chunked"} <= names
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(L.EXPORTS) <= names


def test_only_gdn_symbols_exported():
    out = os.popen(f"nm -D --defined-only {L.library_path()}").read()
    syms = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert syms and all(s.startswith("gdn_") for s in syms), sorted(syms)[:20]


def test_version(lib):
    assert "sm_103a" in L.gdn_version()


def test_workspace_sizes(lib):
    d = L.dims(8, 2, 16, 32, 128)
    rec = L.gdn_layer_workspace_bytes(d, L.GDN_COMMIT_RECOMPUTE)
    snap = L.gdn_layer_workspace_bytes(d, L.GDN_COMMIT_SNAPSHOT)
    assert rec >= 4 * 8 * 2 * (32 * 128 + 16 * 128 + 32)
    assert snap == 4 * 2 * 8 * 32 * 128 * 128
    assert L.gdn_layer_workspace_bytes(d, 7) == 0
    assert L.gdn_layer_workspace_bytes(L.dims(8, 2, 16, 32, 96), 0) == 0


BAD_DIMS = [
    (dict(B=8, T=0, H_k=16, H_v=32, d=128), L.GDN_ERR_UNSUPPORTED),
    (dict(B=8, T=3, H_k=16, H_v=32, d=128, T_max=2), L.GDN_ERR_UNSUPPORTED),
    (dict(B=8, T=9, H_k=16, H_v=32, d=128), L.GDN_ERR_UNSUPPORTED),
    (dict(B=8, T=2, H_k=3, H_v=32, d=128), L.GDN_ERR_UNSUPPORTED),
    (dict(B=8, T=2, H_k=16, H_v=32, d=96), L.GDN_ERR_UNSUPPORTED),
    (dict(B=8, T=2, H_k=16, H_v=32, d=128, width=3), L.GDN_ERR_UNSUPPORTED),
    (dict(B=8, T=2, H_k=16, H_v=32, d=128, act=5), L.GDN_ERR_INVALID_ARG),
    (dict(B=-1, T=2, H_k=16, H_v=32, d=128), L.GDN_ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("kw,code", BAD_DIMS)
def test_bad_dims_rejected_before_launch(lib, kw, code):
    d = L.dims(**kw)
    fake = 1 << 20  # never dereferenced: validation fails first
    rc = lib.gdn_conv_verify(ctypes.byref(d), 0, *([fake] * 10), 1 << 30, None)
    assert rc == code, L.gdn_last_error()
    assert L.gdn_last_error()


def test_null_and_misaligned_pointers(lib):
    d = L.dims(8, 2, 16, 32, 128)
    good = 1 << 20
    ptrs = [good] * 10
    ptrs[0] = None
    assert lib.gdn_conv_verify(ctypes.byref(d), 0, *ptrs, 1 << 30, None) == L.GDN_ERR_INVALID_ARG
    assert "x is NULL" in L.gdn_last_error()
    ptrs[0] = good + 2
    assert lib.gdn_conv_verify(ctypes.byref(d), 0, *ptrs, 1 << 30, None) == L.GDN_ERR_MISALIGNED
    ptrs[0] = good
    assert lib.gdn_conv_verify(ctypes.byref(d), 0, *ptrs, 16, None) == L.GDN_ERR_WORKSPACE
    assert lib.gdn_conv_verify(ctypes.byref(d), 3, *ptrs, 1 << 30, None) == L.GDN_ERR_INVALID_ARG


def test_commit_argument_checks(lib):
    d = L.dims(8, 2, 16, 32, 128)
    P = ctypes.c_void_p
    arr = (P * 1)(1 << 20)
    g = 1 << 20
    assert lib.gdn_commit(ctypes.byref(d), 0, 0, arr, arr, arr, g, g, g, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_commit(ctypes.byref(d), 0, L.GDN_MAX_LAYERS + 1, arr, arr, arr, g, g, g,
                          None) == L.GDN_ERR_INVALID_ARG
    bad = (P * 1)(None)
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, bad, arr, arr, g, g, g, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, arr, bad, arr, g, g, g, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, arr, None, arr, g, g, g, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, arr, arr, bad, g, g, g, None) == L.GDN_ERR_INVALID_ARG
    mis = (P * 1)((1 << 20) + 8)
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, mis, arr, arr, g, g, g, None) == L.GDN_ERR_MISALIGNED
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, arr, mis, arr, g, g, g, None) == L.GDN_ERR_MISALIGNED
    assert lib.gdn_commit(ctypes.byref(d), 5, 1, arr, arr, arr, g, g, g, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, arr, arr, arr, None, g, g, None) == L.GDN_ERR_INVALID_ARG


def test_flush_argument_checks(lib):
    d = L.dims(8, 2, 16, 32, 128)
    P = ctypes.c_void_p
    arr = (P * 1)(1 << 20)
    bad = (P * 1)(None)
    assert lib.gdn_flush(ctypes.byref(d), L.GDN_COMMIT_DEFERRED, 0, arr, arr, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_flush(ctypes.byref(d), L.GDN_COMMIT_DEFERRED, 1, bad, arr, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_flush(ctypes.byref(d), L.GDN_COMMIT_DEFERRED, 1, arr, bad, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_flush(ctypes.byref(d), 7, 1, arr, arr, None) == L.GDN_ERR_INVALID_ARG
    # the eager modes leave nothing pending: a flush launches nothing
    assert lib.gdn_flush(ctypes.byref(d), L.GDN_COMMIT_RECOMPUTE, 1, arr, arr, None) == L.GDN_OK
    assert lib.gdn_flush(ctypes.byref(d), L.GDN_COMMIT_SNAPSHOT, 1, arr, arr, None) == L.GDN_OK


def test_deferred_workspace_size(lib):
    d = L.dims(8, 2, 16, 32, 128)
    rec = lib.gdn_layer_workspace_bytes(ctypes.byref(d), L.GDN_COMMIT_RECOMPUTE)
    dfr = lib.gdn_layer_workspace_bytes(ctypes.byref(d), L.GDN_COMMIT_DEFERRED)
    # the pending keep of every (row, head), then the captures with k kept
    # per value head
    assert dfr == 8 * 32 * 4 + 2 * 8 * 32 * 2 * 128 * 4 + 8 * 32 * 8 * 4
    # captures: e per (row, value head, position), normalised k per (row, key
    # head, position), G padded to 8 positions per (row, value head)
    assert rec == 8 * 32 * 2 * 128 * 4 + 8 * 16 * 2 * 128 * 4 + 8 * 32 * 8 * 4
    assert dfr % 256 == 0


def test_accept_argument_checks(lib):
    assert lib.gdn_accept_workspace_bytes(8, 2, 151936) > 0
    assert lib.gdn_accept_workspace_bytes(8, 0, 10) == 0 and lib.gdn_accept_workspace_bytes(8, 65, 10) == 0
    g = 1 << 20
    ws = lib.gdn_accept_workspace_bytes(8, 2, 1000)
    assert lib.gdn_accept_greedy(8, 2, 1000, None, g, g, g, g, g, ws, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_accept_greedy(8, 2, 1000, g + 2, g, g, g, g, g, ws, None) == L.GDN_ERR_MISALIGNED
    assert lib.gdn_accept_greedy(8, 2, 1000, g, g, g, g, g, g, ws - 1, None) == L.GDN_ERR_WORKSPACE
    assert lib.gdn_accept_greedy(8, 65, 1000, g, g, g, g, g, g, 1 << 30, None) == L.GDN_ERR_UNSUPPORTED
    assert lib.gdn_accept_greedy(8, 0, 1000, g, g, g, g, g, g, 1 << 30, None) == L.GDN_ERR_INVALID_ARG
    assert lib.gdn_accept_greedy(0, 2, 1000, None, None, None, None, None, None, 0, None) == L.GDN_OK


def test_empty_batch_is_a_no_op(lib):
    d = L.dims(0, 2, 16, 32, 128)
    assert lib.gdn_conv_verify(ctypes.byref(d), 0, *([None] * 10), 0, None) == L.GDN_OK
    P = ctypes.c_void_p
    arr = (P * 1)(1 << 20)
    assert lib.gdn_commit(ctypes.byref(d), 0, 1, arr, arr, arr, None, None, None, None) == L.GDN_OK
    assert lib.gdn_flush(ctypes.byref(d), L.GDN_COMMIT_DEFERRED, 1, arr, arr, None) == L.GDN_OK


def declared_arity():
    """Number of parameters of every gdn_* function declared in the headers."""
    arity = {}
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(HEADER_DIR, fn)).read(), flags=re.S)
            for name, params in re.findall(r"\b(gdn_\w+)\s*\(([^)]*)\)\s*;", text):
                params = params.strip()
                arity[name] = 0 if params in ("", "void") else params.count(",") + 1
    return arity


def test_binding_argument_counts_match_header(lib):
    arity = declared_arity()
    assert arity, "no declarations parsed"
    for name, n in arity.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, f"{name}: header has {n} parameters, binding {argtypes}"


PAGES = ('"perf(qwen): full-context MTP draft prefill and replay-free rewind"',
         '"MTP inference: review and commit structure"',
         '"Add request-owned eight-way MTP serving for Qwen 35B"')


def test_every_declaration_cites_its_passage():
    """Each call of the boundary names the page passage that defines it in the
    comment before it, or says that the pages have no such call."""
    text = open(os.path.join(HEADER_DIR, "gdn.h")).read()
    body = text[text.index('extern "C" {'):]
    flat = lambda c: " ".join(c.split()).replace(" * ", " ")
    missing = []
    for m in re.finditer(r"^[a-z][\w\s\*]*?\b(gdn_\w+)\s*\(", body, flags=re.M):
        comments = re.findall(r"/\*.*?\*/", body[:m.start()], flags=re.S)
        last = flat(comments[-1]) if comments else ""
        if not (any(" ".join(pg.split()) in last for pg in PAGES) or "describe no such call" in last):
            missing.append(m.group(1))
    assert not missing, f"declarations without a page citation: {missing}"
