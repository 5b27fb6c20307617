"""The C-ABI library loads, exports every function include/art.h declares, and
rejects bad arguments on the host (no GPU, no compute call). CPU only."""
import ctypes
import os
import re

import pytest

import kv_cache_early_gb300 as K
from kv_cache_early_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "art.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("art_decode", "dense_decode", "art_workspace_bytes", "art_read_device_status", "art_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in art.h but not exported"
        assert getattr(lib, n) is not None


def test_shape_struct_matches_header():
    src = open(HEADER).read()
    body = re.search(r"typedef struct art_shape \{(.*?)\} art_shape;", src, flags=re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"int32_t\s+(\w+);", body)
    assert fields == [f[0] for f in K.ArtShape._fields_]
    assert ctypes.sizeof(K.ArtShape) == 4 * len(fields)


def good_shape(**kw):
    s = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16, block_size=64,
             max_pages_per_seq=8, max_visit=2, num_probe=32, num_pages_total=16, dtype=0)
    s.update(kw)
    return K.make_shape(**s)


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below fails a host check first


def call_art(lib, shape, q=FAKE, probe=FAKE, bu=FAKE, ws=FAKE, ws_bytes=1 << 20, patience=2, em=1e-3, ed=1e-3):
    P = ctypes.c_void_p
    return lib.art_decode(P(q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, em, ed, patience, P(probe), P(FAKE),
                          P(bu), None if shape is None else ctypes.byref(shape), P(ws), ws_bytes, None)


@pytest.mark.parametrize("case,expect", [
    (dict(shape=None), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(num_q_heads=7, num_kv_heads=2)), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(num_q_heads=6, num_kv_heads=2)), K.ART_ERR_UNSUPPORTED),  # G = 3
    (dict(shape=good_shape(head_dim=96)), K.ART_ERR_UNSUPPORTED),
    (dict(shape=good_shape(block_size=32)), K.ART_ERR_UNSUPPORTED),
    (dict(shape=good_shape(page_size=12)), K.ART_ERR_UNSUPPORTED),
    (dict(shape=good_shape(page_size=4)), K.ART_ERR_UNSUPPORTED),
    (dict(shape=good_shape(dtype=5)), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(batch=0)), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(num_probe=33, dtype=1)), K.ART_ERR_UNSUPPORTED),  # > 32 probe columns: bf16 only
    (dict(shape=good_shape(num_probe=129)), K.ART_ERR_INVALID_ARG),  # more probe columns than head dims
    (dict(shape=good_shape(num_probe=0)), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), patience=0), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), em=float("nan")), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), ed=-1.0), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), q=0), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), q=FAKE + 4), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), probe=0), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), bu=0), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), ws=FAKE + 8), K.ART_ERR_INVALID_ARG),
    (dict(shape=good_shape(), ws_bytes=16), K.ART_ERR_WORKSPACE),
])
def test_host_argument_checks(lib, case, expect):
    assert call_art(lib, **case) == expect


def test_dense_host_checks(lib):
    P = ctypes.c_void_p
    s = good_shape()
    assert lib.dense_decode(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), ctypes.byref(s), P(FAKE),
                            8, None) == K.ART_ERR_WORKSPACE
    assert lib.dense_decode(None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), ctypes.byref(s), P(FAKE),
                            1 << 20, None) == K.ART_ERR_INVALID_ARG
    # the dense twin ignores the probe and the thresholds
    s2 = good_shape(num_probe=0)
    assert lib.dense_decode(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(FAKE), ctypes.byref(s2), P(FAKE),
                            8, None) == K.ART_ERR_WORKSPACE


def test_workspace_size(lib):
    # one CTA per item: the 64-byte header, then per item {n, flags} and a claim-order slot
    s = good_shape(batch=3, num_kv_heads=4, num_q_heads=16, dtype=1)
    assert K.art_workspace_bytes(s) == 64 + 12 * 12
    # bf16: plus the unit path's area, which grows with the items and the longest possible list
    small = good_shape(batch=3, num_kv_heads=4, num_q_heads=16)
    longer = good_shape(batch=3, num_kv_heads=4, num_q_heads=16, max_pages_per_seq=8 * 64)
    assert K.art_workspace_bytes(small) > 64 + 12 * 12
    assert K.art_workspace_bytes(longer) > K.art_workspace_bytes(small)
    more = good_shape(batch=300, num_kv_heads=1, num_q_heads=1)
    assert K.art_workspace_bytes(more) > 64 + 12 * 300
    assert lib.art_workspace_bytes(None) == 0


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, 7):
        assert lib.art_status_string(code)


def test_decode_path_choice(lib, monkeypatch):
    """Which kernel path a call takes (host logic only: with ART_UNITS set the
    choice needs no device). The unit path is offered for bf16 with patience at
    most 16, at most 32 probe columns per head and a workspace that holds its
    area."""
    monkeypatch.setenv("ART_UNITS", "1")
    small = good_shape(batch=3, num_kv_heads=4, num_q_heads=16)  # bf16, 12 items
    ws = K.art_workspace_bytes(small)
    assert K.art_decode_path(small, 2, ws) == 1
    assert K.art_decode_path(small, 16, ws) == 1
    assert K.art_decode_path(small, 17, ws) == 0  # patience beyond the longest unit
    assert K.art_decode_path(small, 2, 64 + 12 * 12) == 0  # the one-CTA path's workspace only
    assert K.art_decode_path(good_shape(batch=3, num_kv_heads=4, num_q_heads=16, dtype=1), 2, 1 << 30) == 0
    big = good_shape(batch=300, num_kv_heads=1, num_q_heads=1)  # 300 items
    assert K.art_decode_path(big, 2, K.art_workspace_bytes(big)) == 1
    full = good_shape(batch=3, num_kv_heads=4, num_q_heads=16, num_probe=128)  # a probe over every head dim
    assert K.art_decode_path(full, 2, K.art_workspace_bytes(full)) == 0
    assert K.art_decode_path(good_shape(head_dim=96), 2, 1 << 30) == 0  # fails the shape checks
    monkeypatch.setenv("ART_UNITS", "0")
    assert K.art_decode_path(small, 2, ws) == 0
    assert K.dense_decode_path(small, ws) == 0


def test_dense_path_choice(lib, monkeypatch):
    """The dense twin's unit path is offered for bf16 with a workspace that holds
    its area, at any batch size and probe width (ART_UNITS=1 takes it wherever it
    is offered; the default, which compares the item count with the SM count, is
    checked on the device)."""
    monkeypatch.setenv("ART_UNITS", "1")
    for shape in (good_shape(batch=3, num_kv_heads=4, num_q_heads=16),
                  good_shape(batch=300, num_kv_heads=1, num_q_heads=1),
                  good_shape(batch=2, num_probe=128)):
        ws = K.art_workspace_bytes(shape)
        assert K.dense_decode_path(shape, ws) == 1
        assert K.dense_decode_path(shape, 64 + 12 * shape.batch * shape.num_kv_heads) == 0  # one-CTA workspace only
    fp32 = good_shape(dtype=1)
    assert K.dense_decode_path(fp32, 1 << 30) == 0
    assert K.dense_decode_path(good_shape(head_dim=96), 1 << 30) == 0
