"""fp64 CPU oracle for the paged KV-injection path -- TEST INFRASTRUCTURE.

A plain, slow statement of what the path computes (RoPE, slot mapping,
inject, append, block copies, paged decode attention, paged prefill of query tokens, int8
rows and decode over them), written in C in ``kvinj_oracle.c``
and wrapped here with ctypes over numpy arrays. It shares no code with the
CUDA library in ``paged_kv_cache_inject_gb300``, and neither imports the
other. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may use it; no product code path calls it.

Sources are cited in the C file; every function here only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvinj_oracle.c")
_LIB = os.path.join(_HERE, "libkvinj_oracle.so")
_lock = threading.Lock()
_lib = None
_SIGS: dict = {}

BF16, FP16 = 0, 1

# oracle status bits (its own numbering)
ST_CHUNK, ST_SLOT, ST_BLOCK, ST_POS, ST_CTX, ST_SEQ = 1, 2, 4, 8, 16, 32


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            sig = {
                "orc_encode": (ctypes.c_uint16, [f64, ctypes.c_int]),
                "orc_decode": (f64, [ctypes.c_uint16, ctypes.c_int]),
                "orc_encode_array": (None, [P, i64, ctypes.c_int, P]),
                "orc_decode_array": (None, [P, i64, ctypes.c_int, P]),
                "orc_rope": (None, [P, ctypes.c_int, f64, f64, P]),
                "orc_rope_round_rows": (None, [P, i64, ctypes.c_int, P, f64, ctypes.c_int, P]),
                "orc_kv_bytes": (i64, [i64, i64, i64, i64, i64]),
                "orc_slot_mapping": (i32, [P, ctypes.c_int, ctypes.c_int, i64, P, P, i64,
                                           ctypes.c_int, P]),
                "orc_inject": (i32, [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     i64, ctypes.c_int, P, P, P, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, f64, P, P, i64, ctypes.c_int, ctypes.c_int]),
                "orc_append": (i32, [P, P, ctypes.c_int, ctypes.c_int, i64, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, P, P, P, P, i64, ctypes.c_int,
                                     f64]),
                "orc_copy_blocks": (i32, [P, P, ctypes.c_int, ctypes.c_int, i64, ctypes.c_int,
                                          P, P, i64, ctypes.c_int, ctypes.c_int]),
                "orc_attention": (f64, [P, P, P, i64, ctypes.c_int, f64, P]),
                "orc_attention_bits": (None, [P, ctypes.c_int, f64, f64, P, P, i64, ctypes.c_int,
                                              ctypes.c_int, f64, P]),
                "orc_paged_decode": (i32, [P, P, ctypes.c_int, ctypes.c_int, i64, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                           ctypes.c_int, f64, P, ctypes.c_int, P, ctypes.c_int,
                                           f64, P, ctypes.c_int, ctypes.c_int]),
                "orc_paged_prefill": (i32, [P, P, ctypes.c_int, ctypes.c_int, i64, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, i64,
                                            f64, P, ctypes.c_int, ctypes.c_int, f64, P,
                                            ctypes.c_int]),
                "orc_quantize_rows_i8": (None, [P, i64, ctypes.c_int, ctypes.c_int, P, P]),
                "orc_paged_decode_i8": (i32, [P, P, P, P, ctypes.c_int, ctypes.c_int, i64,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                              ctypes.c_int, P, ctypes.c_int, f64, P, ctypes.c_int,
                                              P, ctypes.c_int, f64, P]),
                "orc_has_openmp": (ctypes.c_int, []),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
                _SIGS[name] = (res, args)
            _lib = lib
    return _lib


class use_library:
    """Context manager that points this wrapper at another build of the oracle
    source (the mutation tests compile deliberately broken copies)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        lib = ctypes.CDLL(self.path)
        for name, fn in _SIGS.items():
            f = getattr(lib, name)
            f.restype, f.argtypes = fn
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def has_openmp() -> bool:
    return bool(_load().orc_has_openmp())


# ---- 16-bit float formats -------------------------------------------------
def encode(x, dtype: int) -> np.ndarray:
    """fp64 -> nearest 16-bit value (ties to even), as uint16 bit patterns."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_encode_array(_p(x), x.size, dtype, _p(out))
    return out


def decode(bits, dtype: int) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().orc_decode_array(_p(bits), bits.size, dtype, _p(out))
    return out


# ---- RoPE -----------------------------------------------------------------
def rope(x, pos: float, theta: float) -> np.ndarray:
    """Rotate one vector x[D] (fp64) to absolute position `pos`."""
    x = _c(x, np.float64)
    y = np.empty_like(x)
    _load().orc_rope(_p(x), x.shape[-1], float(pos), float(theta), _p(y))
    return y


def rope_round_rows(bits, positions, theta: float, dtype: int) -> np.ndarray:
    """Stored rows bits[n][D] rotated at positions[n], rounded once."""
    bits = _c(bits, np.uint16)
    n, D = bits.shape
    pos = _c(positions, np.int32)
    out = np.empty_like(bits)
    _load().orc_rope_round_rows(_p(bits), n, D, _p(pos), float(theta), dtype, _p(out))
    return out


# ---- sizes ----------------------------------------------------------------
def kv_bytes(layers, heads, head_dim, tokens, bytes_per_elem) -> int:
    return int(_load().orc_kv_bytes(layers, heads, head_dim, tokens, bytes_per_elem))


# ---- paging ---------------------------------------------------------------
def slot_mapping(block_tables, seq_ids, positions, block_size: int, num_blocks: int):
    bt = _c(block_tables, np.int32)
    sid = _c(seq_ids, np.int32)
    pos = _c(positions, np.int32)
    out = np.empty(pos.shape, np.int64)
    st = _load().orc_slot_mapping(_p(bt), bt.shape[1], bt.shape[0], num_blocks, _p(sid),
                                  _p(pos), pos.size, block_size, _p(out))
    return out, int(st)


def inject(pool_bits, chunk_ids, start_pos, slot_map, theta, dtype, k_cache, v_cache,
           layer_begin=0, layer_end=None, n_threads=1) -> int:
    """pool_bits[n_chunks][L][2][c][Hkv][D]; k/v_cache[L][NB][Hkv][B][D] (uint16, in place)."""
    pool = _c(pool_bits, np.uint16)
    n_chunks, L, two, c, Hkv, D = pool.shape
    assert two == 2
    NB, B = k_cache.shape[1], k_cache.shape[3]
    ids = _c(chunk_ids, np.int32)
    sp = _c(start_pos, np.int32)
    sm = _c(slot_map, np.int64)
    le = L if layer_end is None else layer_end
    return int(_load().orc_inject(_p(pool), L, Hkv, D, c, n_chunks, dtype, _p(ids), _p(sp),
                                  _p(sm), ids.size, layer_begin, le, float(theta),
                                  _p(k_cache), _p(v_cache), NB, B, n_threads))


def append(k_cache, v_cache, layer, k_new, v_new, positions, slot_map, theta, dtype,
           rotate=True) -> int:
    L, NB, Hkv, B, D = k_cache.shape
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    pos = _c(positions, np.int32)
    sm = _c(slot_map, np.int64)
    return int(_load().orc_append(_p(k_cache), _p(v_cache), Hkv, D, NB, B, dtype, layer,
                                  _p(kn), _p(vn), _p(pos), _p(sm), pos.size, int(rotate),
                                  float(theta)))


def copy_blocks(k_cache, v_cache, src, dst, layer_begin=0, layer_end=None) -> int:
    """In place: block src[i] -> dst[i] in layers [layer_begin, layer_end), K and V."""
    L, NB, Hkv, B, D = k_cache.shape
    s = _c(src, np.int32)
    d = _c(dst, np.int32)
    le = L if layer_end is None else layer_end
    return int(_load().orc_copy_blocks(_p(k_cache), _p(v_cache), Hkv, D, NB, B, _p(s), _p(d),
                                       s.size, layer_begin, le))


# ---- attention ------------------------------------------------------------
def attention(q, K, V, scale: float):
    """Textbook softmax(q K^T * scale) V for one query; returns (out, sum of weights)."""
    q, K, V = _c(q, np.float64), _c(K, np.float64), _c(V, np.float64)
    n, D = K.shape
    out = np.empty(D, np.float64)
    w = _load().orc_attention(_p(q), _p(K), _p(V), n, D, float(scale), _p(out))
    return out, float(w)


def attention_bits(q_bits, q_pos, theta, K_bits, V_bits, dtype, scale=0.0, rotate_q=True):
    """Attention of one stored query row over stored key/value rows [n][D]."""
    qb = _c(q_bits, np.uint16)
    Kb, Vb = _c(K_bits, np.uint16), _c(V_bits, np.uint16)
    n, D = Kb.shape
    if scale <= 0:
        scale = 1.0 / np.sqrt(D)
    out = np.empty(D, np.float64)
    _load().orc_attention_bits(_p(qb), int(rotate_q), float(q_pos), float(theta), _p(Kb),
                               _p(Vb), n, D, dtype, float(scale), _p(out))
    return out


def quantize_rows_i8(bits, dtype: int):
    """int8 codes and fp32 scales of 16-bit rows [..., D]: one scale per row."""
    b = _c(bits, np.uint16)
    D = b.shape[-1]
    q = np.empty(b.shape, np.int8)
    s = np.empty(b.shape[:-1], np.float32)
    _load().orc_quantize_rows_i8(_p(b), b.size // D, D, dtype, _p(q), _p(s))
    return q, s


def paged_decode_i8(kq, ks, vq, vs, layer, q_bits, q_pos, block_tables, context_lens, theta,
                    q_dtype, scale=0.0, rotate_q=True):
    """paged_decode over an int8 cache (codes [L][NB][Hkv][B][D], scales [L][NB][Hkv][B])."""
    L, NB, Hkv, B, D = kq.shape
    kq, vq = _c(kq, np.int8), _c(vq, np.int8)
    ks, vs = _c(ks, np.float32), _c(vs, np.float32)
    q = _c(q_bits, np.uint16)
    batch, Hq, _ = q.shape
    qp = _c(q_pos, np.int32)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.empty((batch, Hq, D), np.float64)
    st = _load().orc_paged_decode_i8(_p(kq), _p(ks), _p(vq), _p(vs), Hkv, D, NB, B, layer, Hq,
                                     _p(q), q_dtype, _p(qp), int(rotate_q), float(theta), _p(bt),
                                     bt.shape[1], _p(cl), batch, float(scale), _p(out))
    return out, int(st)


def paged_prefill(k_cache, v_cache, layer, q_bits, seq_ids, positions, block_tables, theta,
                  dtype, scale=0.0, n_threads=1):
    """Query tokens q_bits[n][Hq][D] of requests seq_ids[n] at positions[n], each attending
    causally to its request's tokens 0..position (already in the cache); returns (out fp64
    [n][Hq][D], status)."""
    L, NB, Hkv, B, D = k_cache.shape
    q = _c(q_bits, np.uint16)
    n, Hq, _ = q.shape
    sq = _c(seq_ids, np.int32)
    ps = _c(positions, np.int32)
    bt = _c(block_tables, np.int32)
    out = np.empty((n, Hq, D), np.float64)
    st = _load().orc_paged_prefill(_p(k_cache), _p(v_cache), Hkv, D, NB, B, dtype, layer, Hq,
                                   _p(q), _p(sq), _p(ps), n, float(theta), _p(bt), bt.shape[1],
                                   bt.shape[0], float(scale), _p(out), n_threads)
    return out, int(st)


def paged_decode(k_cache, v_cache, layer, q_bits, q_pos, block_tables, context_lens, theta,
                 dtype, scale=0.0, rotate_q=True, n_threads=1, window=0):
    """q_bits[batch][Hq][D]; returns (out fp64 [batch][Hq][D], status). window > 0: each
    query attends to the last `window` tokens of its context only."""
    L, NB, Hkv, B, D = k_cache.shape
    q = _c(q_bits, np.uint16)
    batch, Hq, _ = q.shape
    qp = _c(q_pos, np.int32)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    out = np.empty((batch, Hq, D), np.float64)
    st = _load().orc_paged_decode(_p(k_cache), _p(v_cache), Hkv, D, NB, B, dtype, layer, Hq,
                                  _p(q), _p(qp), int(rotate_q), float(theta), _p(bt),
                                  bt.shape[1], _p(cl), batch, float(scale), _p(out), n_threads,
                                  int(window))
    return out, int(st)
