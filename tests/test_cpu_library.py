"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point include/kvinj.h declares, and its host-side parts behave.
No kernel is launched here."""
import ctypes
import math
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from paged_kv_cache_inject_gb300 import build as kbuild
from paged_kv_cache_inject_gb300 import kvinj as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvinj.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return K.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvinj_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = _declared_functions()
    for need in ("kvinj_inject", "kvinj_append", "kvinj_paged_decode", "kvinj_slot_mapping",
                 "kvinj_rope_table_host", "kvinj_decode_workspace_size", "kvinj_strerror",
                 "kvinj_kv_bytes"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvinj_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(lib, n)
    assert sorted(K.EXPORTS) == names  # the binding covers the same entry points


def test_kv_bytes_matches_oracle_and_pages(golden_dir):
    for L, H, D, N, b in ((80, 8, 128, 8192, 2), (32, 8, 128, 1024, 2), (12, 12, 64, 1, 4),
                          (80, 64, 128, 4096, 2)):
        assert K.kvinj_kv_bytes(L, H, D, N, b) == oracle.kv_bytes(L, H, D, N, b)
    assert K.kvinj_kv_bytes(80, 8, 128, 8192, 2) == 2_684_354_560


def test_rope_table_host_against_fp64_cos_sin():
    for theta, D, P in ((1e4, 64, 300), (5e5, 128, 40000)):
        t = K.kvinj_rope_table_host(theta, D, P).astype(np.float64)
        assert t.shape == (P, D // 2, 4)
        rng = np.random.default_rng(0)
        for p in rng.integers(0, P, 200):
            for i in rng.integers(0, D // 2, 8):
                ang = p * theta ** (-2.0 * i / D)
                assert abs(t[p, i, 0] + t[p, i, 2] - math.cos(ang)) <= 2.0 ** -46
                assert abs(t[p, i, 1] + t[p, i, 3] - math.sin(ang)) <= 2.0 ** -46
                assert t[p, i, 0] == np.float32(math.cos(ang)) or \
                    abs(t[p, i, 0] - math.cos(ang)) <= 2.0 ** -24
    assert K.kvinj_rope_table_bytes(128, 10) == 10 * 64 * 16


def test_rope_table_host_rejects_bad_args(lib):
    buf = np.empty(64, np.float32)
    p = buf.ctypes.data_as(ctypes.c_void_p)
    assert lib.kvinj_rope_table_host(1e4, 3, 4, p) == K.KVINJ_EINVAL
    assert lib.kvinj_rope_table_host(1e4, 4, 0, p) == K.KVINJ_EINVAL
    assert lib.kvinj_rope_table_host(-1.0, 4, 4, p) == K.KVINJ_EINVAL
    assert lib.kvinj_rope_table_host(1e4, 4, 4, None) == K.KVINJ_EINVAL


def test_host_validation_rejects_before_launch(lib):
    # null descriptors and impossible shapes are refused on the host, no GPU needed
    assert lib.kvinj_inject(None, None, None, None, None, None, 1, 0, 1, None, None) == K.KVINJ_EINVAL
    cache = K._Cache(2, 8, 128, 16, 10, 0, 0x1000, 0x2000)
    pool = K._Pool(2, 8, 128, 16, 4, 0, 0x3000)
    rope = K._Rope(0x4000, 100, 128)
    r = ctypes.byref
    # layer range beyond the cache
    assert lib.kvinj_inject(r(pool), r(cache), r(rope), 1, 1, 1, 1, 0, 3, None, None) == K.KVINJ_EINVAL
    # pool / cache disagree on head_dim
    pool_bad = K._Pool(2, 8, 64, 16, 4, 0, 0x3000)
    assert lib.kvinj_inject(r(pool_bad), r(cache), r(rope), 1, 1, 1, 1, 0, 1, None, None) == K.KVINJ_EINVAL
    # nothing to do
    assert lib.kvinj_inject(r(pool), r(cache), r(rope), None, None, None, 0, 0, 2, None, None) == K.KVINJ_OK
    # misaligned cache pointer
    cache_mis = K._Cache(2, 8, 128, 16, 10, 0, 0x1002, 0x2000)
    assert lib.kvinj_append(r(cache_mis), None, 0, 16, 16, 16, 16, 1, None, None) == K.KVINJ_EINVAL
    # decode: block size 32 and head_dim 96 have no kernel; Hq not a multiple of Hkv
    c32 = K._Cache(2, 8, 128, 32, 10, 0, 0x1000, 0x2000)
    assert lib.kvinj_paged_decode(r(c32), None, 0, 32, 16, 16, 16, 4, 16, 1, 0.0, 16, 16, 1 << 30,
                                  None, None) == K.KVINJ_EUNSUPPORTED
    c96 = K._Cache(2, 8, 96, 16, 10, 0, 0x1000, 0x2000)
    assert lib.kvinj_paged_decode(r(c96), None, 0, 32, 16, 16, 16, 4, 16, 1, 0.0, 16, 16, 1 << 30,
                                  None, None) == K.KVINJ_EUNSUPPORTED
    assert lib.kvinj_paged_decode(r(cache), None, 0, 12, 16, 16, 16, 4, 16, 1, 0.0, 16, 16, 1 << 30,
                                  None, None) == K.KVINJ_EINVAL
    # decode: an empty batch is a no-op; batches beyond the prefix sums' shared memory and
    # windows on the other kernels are refused
    assert lib.kvinj_paged_decode(r(cache), None, 0, 32, None, None, None, 4, None, 0, 0.0, None,
                                  None, 0, None, None) == K.KVINJ_OK
    assert lib.kvinj_paged_decode(r(cache), None, 0, 32, 16, 16, 16, 4, 16, 5000, 0.0, 16, 16,
                                  1 << 40, None, None) == K.KVINJ_EUNSUPPORTED
    assert lib.kvinj_paged_decode(r(cache), None, 0, 32, 16, 16, 16, 4, 16, -1, 0.0, 16, 16,
                                  1 << 30, None, None) == K.KVINJ_EINVAL
    # decode with rope but no q_pos
    assert lib.kvinj_paged_decode(r(cache), r(rope), 0, 32, 16, None, 16, 4, 16, 1, 0.0, 16, 16,
                                  1 << 30, None, None) == K.KVINJ_EINVAL
    # slot mapping: negative n, zero n
    assert lib.kvinj_slot_mapping(16, 4, 1, 10, 16, 16, 16, -1, 16, None, None) == K.KVINJ_EINVAL
    assert lib.kvinj_slot_mapping(None, 4, 1, 10, 16, None, None, 0, None, None, None) == K.KVINJ_OK


def test_strerror_and_codes():
    assert K.kvinj_strerror(0) == "ok"
    assert "workspace" in K.kvinj_strerror(K.KVINJ_EWORKSPACE)
    assert "unknown" in K.kvinj_strerror(99)
    text = open(HEADER).read()
    for name, val in (("KVINJ_EINVAL", 1), ("KVINJ_EUNSUPPORTED", 2), ("KVINJ_EWORKSPACE", 3),
                      ("KVINJ_ECUDA", 4), ("KVINJ_ST_BAD_CHUNK", 0x01), ("KVINJ_ST_TIMEOUT", 0x40)):
        m = re.search(rf"#define {name} (0x[0-9a-fA-F]+|\d+)", text)
        assert m and int(m.group(1), 0) == val


def test_prefill_host_validation(lib):
    # no GPU needed: sizes and argument checks happen before any launch
    assert lib.kvinj_prefill_workspace_size(0, 32, 8, 128, 64) == 0
    assert lib.kvinj_prefill_workspace_size(10, 30, 8, 128, 64) == 0  # Hq not a multiple of Hkv
    assert lib.kvinj_prefill_workspace_size(10, 32, 0, 128, 64) == 0  # no kv heads
    assert lib.kvinj_prefill_workspace_size(10, 0, 8, 128, 64) == 0  # no query heads
    assert lib.kvinj_prefill_workspace_size(10, 32, 8, 128, 0) == 0  # no table columns
    r = lambda x: (x + 255) // 256 * 256
    # tensor-core path (D = 128, G in {1, 2, 4, 8}): a header, 16 bytes of tile and 4 of
    # unit prefix per query token, per-CTA entries that do not depend on the tokens, and
    # the prepared query rows (hi and lo 16-bit parts: 512 bytes per query head)
    small = lib.kvinj_prefill_workspace_size(10, 32, 8, 128, 64)
    big = lib.kvinj_prefill_workspace_size(5000, 32, 8, 128, 64)
    assert small > 0
    assert big - small == (r(5000 * 16) - r(10 * 16)) + (r(5001 * 4) - r(11 * 4)) + \
        (r(5000 * 32 * 512) - r(10 * 32 * 512))
    assert lib.kvinj_prefill_workspace_size(10, 32, 8, 128, 4096) == small  # no table copies
    # decode rows (other shapes): the decode's workspace, then the rows' tables, context
    # lengths and q positions (at most 1024 rows per launch), each 256-byte aligned
    dec = lib.kvinj_decode_workspace_size(1, 8, 4, 64)
    assert lib.kvinj_prefill_workspace_size(10, 8, 4, 64, 64) == \
        r(dec) + r(10 * 64 * 4) + 2 * r(10 * 4)
    assert lib.kvinj_prefill_workspace_size(5000, 8, 4, 64, 64) == \
        r(dec) + r(1024 * 64 * 4) + 2 * r(1024 * 4)
    cache = K._Cache(2, 8, 128, 16, 10, 0, 0x1000, 0x2000)
    rr = ctypes.byref
    # nothing to do
    assert lib.kvinj_paged_prefill(rr(cache), None, 0, 32, None, None, None, 0, None, 4, 1, 0.0,
                                   None, None, 0, None, None) == K.KVINJ_OK
    # missing arrays, a workspace too small
    assert lib.kvinj_paged_prefill(rr(cache), None, 0, 32, None, 16, 16, 3, 16, 4, 1, 0.0, 16, 16,
                                   1 << 20, None, None) == K.KVINJ_EINVAL
    need = lib.kvinj_prefill_workspace_size(3, 32, 8, 128, 4)
    assert lib.kvinj_paged_prefill(rr(cache), None, 0, 32, 16, 16, 16, 3, 16, 4, 1, 0.0, 16, 16,
                                   need - 1, None, None) == K.KVINJ_EWORKSPACE


def test_static_scratch_size_of_the_binding_is_the_headers():
    text = open(HEADER).read()
    m = re.search(r"#define KVINJ_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m, "KVINJ_STATIC_SCRATCH_BYTES not found in the header"
    assert K.KVINJ_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_decode_flags_host_validation(lib):
    # an unknown flag bit is refused on the host before anything else runs; the one
    # defined bit is the header's
    text = open(HEADER).read()
    m = re.search(r"#define KVINJ_DECODE_KV_READY (\d+)", text)
    assert m and int(m.group(1)) == K.KVINJ_DECODE_KV_READY == 1
    cache = K._Cache(2, 8, 128, 16, 10, 0, 0x1000, 0x2000)
    r = ctypes.byref
    assert lib.kvinj_paged_decode_ex(r(cache), None, 0, 32, 16, 16, 16, 4, 16, 1, 0.0, 16, 16,
                                     1 << 30, None, None, 0, 0, 2) == K.KVINJ_EINVAL
    assert lib.kvinj_append_paged_decode_ex(r(cache), None, 0, 32, 16, 16, 16, 16, 16, 4, 16, 1,
                                            0.0, 16, 16, 1 << 30, None, None, 0, 0,
                                            4) == K.KVINJ_EINVAL
    assert lib.kvinj_paged_decode_window(r(cache), None, 0, 32, 16, None, None, 16, 16, 4, 16, 1,
                                         0, 0.0, 16, 16, 1 << 30, None, None,
                                         -1) == K.KVINJ_EINVAL
