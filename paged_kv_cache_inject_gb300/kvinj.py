"""Python binding of the C ABI in include/kvinj.h (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors that already live on the GPU, passes their device pointers and sizes
through ctypes, and raises KvinjError on a non-zero return code. All
computation happens in the CUDA kernels of libkvinj.so; there is no other
implementation behind these names, and loading fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvinj.so")

KVINJ_BF16, KVINJ_FP16 = 0, 1
KVINJ_OK, KVINJ_EINVAL, KVINJ_EUNSUPPORTED, KVINJ_EWORKSPACE, KVINJ_ECUDA = 0, 1, 2, 3, 4
ST_BAD_CHUNK, ST_BAD_SLOT, ST_BAD_BLOCK, ST_BAD_POS = 0x01, 0x02, 0x04, 0x08
ST_BAD_CTX, ST_BAD_SEQ, ST_TIMEOUT, ST_INTERNAL = 0x10, 0x20, 0x40, 0x80
KVINJ_STATIC_SCRATCH_BYTES = 24 << 20  # size of the fixed scratch of kvinj_paged_decode_static
KVINJ_DECODE_KV_READY = 1  # decode flag: pages/tables/lengths final before the previous decode call

EXPORTS = [
    "kvinj_rope_table_bytes", "kvinj_rope_table_host", "kvinj_slot_mapping", "kvinj_inject",
    "kvinj_append", "kvinj_decode_workspace_size", "kvinj_decode_workspace_init",
    "kvinj_paged_decode", "kvinj_paged_decode_ex", "kvinj_append_paged_decode",
    "kvinj_append_paged_decode_ex", "kvinj_paged_decode_static", "kvinj_kv_bytes",
    "kvinj_strerror", "kvinj_copy_blocks", "kvinj_paged_decode_window",
    "kvinj_prefill_workspace_size", "kvinj_paged_prefill", "kvinj_rope_table64_bytes",
    "kvinj_rope_table64_host", "kvinj_inject_i8", "kvinj_append_i8", "kvinj_paged_decode_i8",
]


class KvinjError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({kvinj_strerror(code)})")


class _Cache(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p)]


class _Pool(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("chunk_len", ctypes.c_int32),
                ("num_chunks", ctypes.c_int64), ("dtype", ctypes.c_int32),
                ("data", ctypes.c_void_p)]


class _Rope(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("max_pos", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("table64", ctypes.c_void_p)]


class _CacheI8(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int64), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libkvinj.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} not found: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "kvinj_rope_table_bytes": (sz, [i32, i32]),
            "kvinj_rope_table_host": (ctypes.c_int, [ctypes.c_double, i32, i32, P]),
            "kvinj_slot_mapping": (ctypes.c_int, [P, i32, i32, i64, i32, P, P, i64, P, P, P]),
            "kvinj_inject": (ctypes.c_int, [P, P, P, P, P, P, i32, i32, i32, P, P]),
            "kvinj_append": (ctypes.c_int, [P, P, i32, P, P, P, P, i64, P, P]),
            "kvinj_copy_blocks": (ctypes.c_int, [P, P, P, i64, i32, i32, P, P]),
            "kvinj_prefill_workspace_size": (sz, [i32, i32, i32, i32, i32]),
            "kvinj_paged_prefill": (ctypes.c_int, [P, P, i32, i32, P, P, P, i32, P, i32, i32,
                                                   ctypes.c_float, P, P, sz, P, P]),
            "kvinj_paged_decode_window": (ctypes.c_int, [P, P, i32, i32, P, P, P, P, P, i32, P,
                                                         i32, i32, ctypes.c_float, P, P, sz, P,
                                                         P, i32]),
            "kvinj_decode_workspace_size": (sz, [i32, i32, i32, i32]),
            "kvinj_decode_workspace_init": (ctypes.c_int, [P, sz, P]),
            "kvinj_paged_decode": (ctypes.c_int, [P, P, i32, i32, P, P, P, i32, P, i32,
                                                  ctypes.c_float, P, P, sz, P, P]),
            "kvinj_paged_decode_ex": (ctypes.c_int, [P, P, i32, i32, P, P, P, i32, P, i32,
                                                     ctypes.c_float, P, P, sz, P, P, i32, i32,
                                                     i32]),
            "kvinj_append_paged_decode": (ctypes.c_int, [P, P, i32, i32, P, P, P, P, P, i32, P,
                                                         i32, ctypes.c_float, P, P, sz, P, P]),
            "kvinj_append_paged_decode_ex": (ctypes.c_int, [P, P, i32, i32, P, P, P, P, P, i32,
                                                            P, i32, ctypes.c_float, P, P, sz, P,
                                                            P, i32, i32, i32]),
            "kvinj_paged_decode_static": (ctypes.c_int, [P, P, i32, i32, P, P, P, i32, P, i32,
                                                         ctypes.c_float, P, P, P]),
            "kvinj_kv_bytes": (i64, [i32, i32, i32, i64, i32]),
            "kvinj_rope_table64_bytes": (sz, [i32, i32]),
            "kvinj_rope_table64_host": (ctypes.c_int, [ctypes.c_double, i32, i32, P]),
            "kvinj_inject_i8": (ctypes.c_int, [P, P, P, P, P, P, i32, i32, i32, P, P]),
            "kvinj_append_i8": (ctypes.c_int, [P, P, i32, i32, P, P, P, P, i64, P, P]),
            "kvinj_paged_decode_i8": (ctypes.c_int, [P, P, i32, i32, i32, P, P, P, P, P, i32, P,
                                                     i32, ctypes.c_float, P, P, sz, P, P, i32]),
            "kvinj_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# descriptors
# ---------------------------------------------------------------------------
def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return KVINJ_BF16
    if t == torch.float16:
        return KVINJ_FP16
    raise TypeError(f"unsupported element type {t}")


class Cache:
    """Paged KV cache: k, v tensors [L][num_blocks][Hkv][block_size][D] on the GPU."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor):
        assert k.shape == v.shape and k.dim() == 5 and k.dtype == v.dtype
        assert k.is_cuda and v.is_cuda and k.is_contiguous() and v.is_contiguous()
        self.k, self.v = k, v
        L, NB, Hkv, B, D = k.shape
        self.num_layers, self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = \
            L, NB, Hkv, B, D
        self._s = _Cache(L, Hkv, D, B, NB, _dtype_code(k.dtype), k.data_ptr(), v.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self._s)


class CacheI8:
    """int8 paged cache: codes k, v int8 [L][num_blocks][Hkv][16][D], scales k_scale,
    v_scale float32 [L][num_blocks][Hkv][16], on the GPU."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor, k_scale: torch.Tensor,
                 v_scale: torch.Tensor):
        assert k.shape == v.shape and k.dim() == 5 and k.dtype == v.dtype == torch.int8
        assert k_scale.shape == v_scale.shape == k.shape[:4]
        assert k_scale.dtype == v_scale.dtype == torch.float32
        for t in (k, v, k_scale, v_scale):
            assert t.is_cuda and t.is_contiguous()
        self.k, self.v, self.k_scale, self.v_scale = k, v, k_scale, v_scale
        L, NB, Hkv, B, D = k.shape
        self.num_layers, self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = \
            L, NB, Hkv, B, D
        self._s = _CacheI8(L, Hkv, D, B, NB, k.data_ptr(), v.data_ptr(), k_scale.data_ptr(),
                           v_scale.data_ptr())

    @classmethod
    def empty(cls, layers, num_blocks, kv_heads, head_dim, block_size=16, device="cuda"):
        shape = (layers, num_blocks, kv_heads, block_size, head_dim)
        return cls(torch.empty(shape, dtype=torch.int8, device=device),
                   torch.empty(shape, dtype=torch.int8, device=device),
                   torch.empty(shape[:4], dtype=torch.float32, device=device),
                   torch.empty(shape[:4], dtype=torch.float32, device=device))

    @property
    def ref(self):
        return ctypes.byref(self._s)


class Pool:
    """Pre-RoPE chunk pool: data [num_chunks][L][2][chunk_len][Hkv][D] on the GPU, or in
    page-locked host memory (a pinned CPU tensor), which inject reads in place."""

    def __init__(self, data: torch.Tensor):
        assert data.dim() == 6 and data.shape[2] == 2 and data.is_contiguous()
        assert data.is_cuda or data.is_pinned(), "the pool is device or pinned host memory"
        n, L, _, c, Hkv, D = data.shape
        self.data = data
        self._s = _Pool(L, Hkv, D, c, n, _dtype_code(data.dtype), data.data_ptr())

    @property
    def ref(self):
        return ctypes.byref(self._s)


class Rope:
    """RoPE table (float4 [max_pos][D/2]) on the GPU, with the fp64 table (double2
    [max_pos][D/2] {cos, sin}) the int8 calls that rotate keys also need."""

    def __init__(self, table: torch.Tensor, head_dim: int, table64: torch.Tensor | None = None):
        assert table.is_cuda and table.dtype == torch.float32 and table.is_contiguous()
        self.table = table
        self.table64 = table64
        self.max_pos = table.shape[0]
        self.head_dim = head_dim
        if table64 is not None:
            assert table64.is_cuda and table64.dtype == torch.float64 and table64.is_contiguous()
            assert table64.shape[0] == self.max_pos
        self._s = _Rope(table.data_ptr(), self.max_pos, head_dim,
                        table64.data_ptr() if table64 is not None else None)

    @property
    def ref(self):
        return ctypes.byref(self._s)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, rc: int):
    if rc != KVINJ_OK:
        raise KvinjError(fn, rc)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def kvinj_strerror(code: int) -> str:
    return load().kvinj_strerror(code).decode()


def kvinj_kv_bytes(layers: int, heads: int, head_dim: int, tokens: int, bytes_per_elem: int) -> int:
    return int(load().kvinj_kv_bytes(layers, heads, head_dim, tokens, bytes_per_elem))


def kvinj_rope_table_bytes(head_dim: int, max_pos: int) -> int:
    return int(load().kvinj_rope_table_bytes(head_dim, max_pos))


def kvinj_rope_table_host(theta: float, head_dim: int, max_pos: int) -> np.ndarray:
    """Host table float32 [max_pos][head_dim/2][4] = {cos_hi, sin_hi, cos_lo, sin_lo}."""
    out = np.empty((max_pos, head_dim // 2, 4), np.float32)
    _check("kvinj_rope_table_host",
           load().kvinj_rope_table_host(float(theta), head_dim, max_pos,
                                        out.ctypes.data_as(ctypes.c_void_p)))
    return out


def kvinj_rope_table64_host(theta: float, head_dim: int, max_pos: int) -> np.ndarray:
    """Host table float64 [max_pos][head_dim/2][2] = {cos, sin}."""
    out = np.empty((max_pos, head_dim // 2, 2), np.float64)
    _check("kvinj_rope_table64_host",
           load().kvinj_rope_table64_host(float(theta), head_dim, max_pos,
                                          out.ctypes.data_as(ctypes.c_void_p)))
    return out


def make_rope(theta: float, head_dim: int, max_pos: int, device="cuda") -> Rope:
    """Build the tables on the host (fp64) and copy them to the device: the float hi/lo
    table every rotation uses and the fp64 one the int8 calls also need."""
    host = kvinj_rope_table_host(theta, head_dim, max_pos)
    host64 = kvinj_rope_table64_host(theta, head_dim, max_pos)
    return Rope(torch.from_numpy(host).to(device).contiguous(), head_dim,
                torch.from_numpy(host64).to(device).contiguous())


def kvinj_slot_mapping(block_tables, seq_ids, positions, num_blocks: int, block_size: int,
                       slot_out, status=None, stream=None):
    assert block_tables.dtype == torch.int32 and block_tables.dim() == 2
    n = positions.numel()
    _check("kvinj_slot_mapping",
           load().kvinj_slot_mapping(_ptr(block_tables), block_tables.shape[1],
                                     block_tables.shape[0], num_blocks, block_size,
                                     _ptr(seq_ids), _ptr(positions), n, _ptr(slot_out),
                                     _ptr(status), _stream(stream)))
    return slot_out


def kvinj_inject(pool: Pool, cache: Cache, rope: Rope, chunk_ids, start_pos, slot_mapping,
                 layer_begin: int = 0, layer_end: int | None = None, status=None, stream=None):
    le = cache.num_layers if layer_end is None else layer_end
    _check("kvinj_inject",
           load().kvinj_inject(pool.ref, cache.ref, rope.ref, _ptr(chunk_ids), _ptr(start_pos),
                               _ptr(slot_mapping), chunk_ids.numel(), layer_begin, le,
                               _ptr(status), _stream(stream)))


def kvinj_copy_blocks(cache: Cache, src, dst, layer_begin: int = 0, layer_end: int | None = None,
                      status=None, stream=None):
    """Copy physical block src[i] to dst[i] in every layer of [layer_begin, layer_end), K and
    V (int32 device tensors of equal length): the copy-on-write of a shared block."""
    assert src.dtype == torch.int32 and dst.dtype == torch.int32 and src.numel() == dst.numel()
    le = cache.num_layers if layer_end is None else layer_end
    _check("kvinj_copy_blocks",
           load().kvinj_copy_blocks(cache.ref, _ptr(src), _ptr(dst), src.numel(), layer_begin, le,
                                    _ptr(status), _stream(stream)))


def kvinj_paged_decode_window(cache: Cache, rope: Rope | None, layer: int, q, q_pos,
                              block_tables, context_lens, window: int, out, workspace,
                              k_new=None, v_new=None, scale: float = 0.0, status=None,
                              stream=None, flags: int = 0):
    """Paged decode over the last `window` tokens of each context (0: all of them), with
    the new token's append fused when k_new and v_new are given; flags: KVINJ_DECODE_*."""
    batch, Hq, _ = q.shape
    _check("kvinj_paged_decode_window",
           load().kvinj_paged_decode_window(
               cache.ref, rope.ref if rope is not None else None, layer, Hq, _ptr(q),
               _ptr(k_new) if k_new is not None else None,
               _ptr(v_new) if v_new is not None else None, _ptr(q_pos), _ptr(block_tables),
               block_tables.shape[1], _ptr(context_lens), batch, window, float(scale), _ptr(out),
               _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
               _stream(stream), int(flags)))


def kvinj_prefill_workspace_size(n: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                 max_blocks: int) -> int:
    return int(load().kvinj_prefill_workspace_size(n, num_q_heads, num_kv_heads, head_dim,
                                                   max_blocks))


def make_prefill_workspace(n, num_q_heads, num_kv_heads, head_dim, max_blocks, device="cuda"):
    nbytes = kvinj_prefill_workspace_size(n, num_q_heads, num_kv_heads, head_dim, max_blocks)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def kvinj_paged_prefill(cache: Cache, rope: Rope | None, layer: int, q, seq_ids, positions,
                        block_tables, out, workspace, scale: float = 0.0, status=None,
                        stream=None):
    """Query tokens q[n][Hq][D] of requests seq_ids[n] at positions[n] (their K/V already in
    the cache), each attending causally to its request's tokens 0..position."""
    n, Hq, _ = q.shape
    _check("kvinj_paged_prefill",
           load().kvinj_paged_prefill(cache.ref, rope.ref if rope is not None else None, layer,
                                      Hq, _ptr(q), _ptr(seq_ids), _ptr(positions), n,
                                      _ptr(block_tables), block_tables.shape[1],
                                      block_tables.shape[0], float(scale), _ptr(out),
                                      _ptr(workspace),
                                      workspace.numel() * workspace.element_size(),
                                      _ptr(status), _stream(stream)))


def kvinj_append(cache: Cache, rope: Rope | None, layer: int, k_new, v_new, positions,
                 slot_mapping, status=None, stream=None):
    _check("kvinj_append",
           load().kvinj_append(cache.ref, rope.ref if rope is not None else None, layer,
                               _ptr(k_new), _ptr(v_new), _ptr(positions), _ptr(slot_mapping),
                               positions.numel(), _ptr(status), _stream(stream)))


def kvinj_decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int,
                                head_dim: int) -> int:
    return int(load().kvinj_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim))


def kvinj_decode_workspace_init(workspace, stream=None):
    _check("kvinj_decode_workspace_init",
           load().kvinj_decode_workspace_init(_ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _stream(stream)))


def make_decode_workspace(batch, num_q_heads, num_kv_heads, head_dim, device="cuda", stream=None):
    n = kvinj_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    kvinj_decode_workspace_init(ws, stream)
    return ws


def kvinj_paged_decode(cache: Cache, rope: Rope | None, layer: int, q, q_pos, block_tables,
                       context_lens, out, workspace, scale: float = 0.0, status=None,
                       stream=None):
    batch, Hq, _ = q.shape
    _check("kvinj_paged_decode",
           load().kvinj_paged_decode(cache.ref, rope.ref if rope is not None else None, layer,
                                     Hq, _ptr(q), _ptr(q_pos), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(context_lens), batch,
                                     float(scale), _ptr(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(status), _stream(stream)))
    return out


def kvinj_paged_decode_static(cache: Cache, rope: Rope | None, layer: int, q, q_pos,
                              block_tables, context_lens, out, scale: float = 0.0, status=None,
                              stream=None):
    """kvinj_paged_decode with the library's fixed device scratch (no workspace)."""
    batch, Hq, _ = q.shape
    _check("kvinj_paged_decode_static",
           load().kvinj_paged_decode_static(cache.ref, rope.ref if rope is not None else None,
                                            layer, Hq, _ptr(q), _ptr(q_pos), _ptr(block_tables),
                                            block_tables.shape[1], _ptr(context_lens), batch,
                                            float(scale), _ptr(out), _ptr(status),
                                            _stream(stream)))
    return out


def kvinj_paged_decode_ex(cache: Cache, rope: Rope | None, layer: int, q, q_pos, block_tables,
                          context_lens, out, workspace, scale: float = 0.0, status=None,
                          stream=None, variant: int = 0, ctas: int = 0, flags: int = 0):
    batch, Hq, _ = q.shape
    _check("kvinj_paged_decode_ex",
           load().kvinj_paged_decode_ex(cache.ref, rope.ref if rope is not None else None,
                                        layer, Hq, _ptr(q), _ptr(q_pos), _ptr(block_tables),
                                        block_tables.shape[1], _ptr(context_lens), batch,
                                        float(scale), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _ptr(status), _stream(stream), variant, ctas,
                                        int(flags)))
    return out


def kvinj_append_paged_decode(cache: Cache, rope: Rope | None, layer: int, q, k_new, v_new,
                              q_pos, block_tables, context_lens, out, workspace,
                              scale: float = 0.0, status=None, stream=None, variant: int = 0,
                              ctas: int = 0, flags: int = 0):
    """Append the token at q_pos of every request (k_new, v_new [batch][Hkv][D]), then
    decode; variant/ctas/flags as in kvinj_paged_decode_ex (0: automatic, none)."""
    batch, Hq, _ = q.shape
    _check("kvinj_append_paged_decode_ex",
           load().kvinj_append_paged_decode_ex(
               cache.ref, rope.ref if rope is not None else None, layer, Hq, _ptr(q),
               _ptr(k_new), _ptr(v_new), _ptr(q_pos), _ptr(block_tables), block_tables.shape[1],
               _ptr(context_lens), batch, float(scale), _ptr(out), _ptr(workspace),
               workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream),
               variant, ctas, int(flags)))
    return out


# ---------------------------------------------------------------------------
# int8 cache
# ---------------------------------------------------------------------------
def kvinj_inject_i8(pool: Pool, cache: CacheI8, rope: Rope, chunk_ids, start_pos, slot_mapping,
                    layer_begin: int = 0, layer_end: int | None = None, status=None,
                    stream=None):
    """Inject into an int8 cache: each rotated K row and each V row quantized."""
    le = cache.num_layers if layer_end is None else layer_end
    _check("kvinj_inject_i8",
           load().kvinj_inject_i8(pool.ref, cache.ref, rope.ref, _ptr(chunk_ids),
                                  _ptr(start_pos), _ptr(slot_mapping), chunk_ids.numel(),
                                  layer_begin, le, _ptr(status), _stream(stream)))


def kvinj_append_i8(cache: CacheI8, rope: Rope | None, layer: int, k_new, v_new, positions,
                    slot_mapping, status=None, stream=None):
    """Append k_new, v_new [n][Hkv][D] (16-bit) at their slots, quantized."""
    _check("kvinj_append_i8",
           load().kvinj_append_i8(cache.ref, rope.ref if rope is not None else None,
                                  _dtype_code(k_new.dtype), layer, _ptr(k_new), _ptr(v_new),
                                  _ptr(positions), _ptr(slot_mapping), positions.numel(),
                                  _ptr(status), _stream(stream)))


def kvinj_paged_decode_i8(cache: CacheI8, rope: Rope | None, layer: int, q, q_pos,
                          block_tables, context_lens, out, workspace, k_new=None, v_new=None,
                          scale: float = 0.0, status=None, stream=None, ctas: int = 0):
    """Paged decode over an int8 cache (q, out [batch][Hq][D] 16-bit), with the new token's
    append fused when k_new and v_new are given."""
    batch, Hq, _ = q.shape
    _check("kvinj_paged_decode_i8",
           load().kvinj_paged_decode_i8(
               cache.ref, rope.ref if rope is not None else None, _dtype_code(q.dtype), layer,
               Hq, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(q_pos), _ptr(block_tables),
               block_tables.shape[1], _ptr(context_lens), batch, float(scale), _ptr(out),
               _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status),
               _stream(stream), ctas))
    return out
