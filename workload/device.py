"""Device side of the workload generator: fills GPU buffers with the same bits
as the host generator in ``workload`` (see ``workload/csrc/kvgen.cu``)."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np
import torch

from . import NORMAL_SCALE, Workload

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "kvgen.cu")
LIB = os.path.join(_HERE, "libkvgen.so")
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(_SRC):
        return LIB
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", _SRC, "-o", tmp], check=True)
    os.replace(tmp, LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} not built")
        lib = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        lib.kvgen_fill_linear.argtypes = [P, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_float, ctypes.c_int, P]
        lib.kvgen_fill_linear.restype = ctypes.c_int
        lib.kvgen_fill_rows.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_uint64,
                                        ctypes.c_float, ctypes.c_int, P]
        lib.kvgen_fill_rows.restype = ctypes.c_int
        _lib = lib
    return _lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def torch_dtype(code: int):
    return torch.float16 if code == 1 else torch.bfloat16


def fill_linear(dst: torch.Tensor, key: int, start: int, dtype: int):
    rc = _load().kvgen_fill_linear(ctypes.c_void_p(dst.data_ptr()), dst.numel(), key, start,
                                   float(NORMAL_SCALE), dtype, _stream())
    if rc:
        raise RuntimeError(f"kvgen_fill_linear: cuda error {rc}")


def fill_rows(dst: torch.Tensor, row_base: np.ndarray, key: int, dtype: int):
    n = row_base.size
    base = torch.from_numpy(np.ascontiguousarray(row_base, np.int64)).to(dst.device)
    row_len = dst.numel() // max(n, 1)
    rc = _load().kvgen_fill_rows(ctypes.c_void_p(dst.data_ptr()), n, row_len,
                                 ctypes.c_void_p(base.data_ptr()), key, float(NORMAL_SCALE),
                                 dtype, _stream())
    if rc:
        raise RuntimeError(f"kvgen_fill_rows: cuda error {rc}")
    return base  # keep alive until the stream has used it


def pool_tensor(wl: Workload, device="cuda", n_chunks: int | None = None) -> torch.Tensor:
    cfg = wl.cfg
    n = cfg.pool_chunks if n_chunks is None else n_chunks
    t = torch.empty((n, cfg.layers, 2, cfg.chunk_len, cfg.kv_heads, cfg.head_dim),
                    dtype=torch_dtype(cfg.dtype), device=device)
    fill_linear(t, wl.keys["pool"], 0, cfg.dtype)
    return t


def ctx_rows(wl: Workload, layer: int, kv: int, seq, pos, device="cuda") -> torch.Tensor:
    cfg = wl.cfg
    n = len(seq)
    t = torch.empty((n, cfg.kv_heads, cfg.head_dim), dtype=torch_dtype(cfg.dtype), device=device)
    keep = fill_rows(t, wl.ctx_row_base(layer, kv, seq, pos), wl.keys["ctx"], cfg.dtype)
    return t, keep


def q_rows(wl: Workload, step: int, layer: int, device="cuda") -> torch.Tensor:
    cfg = wl.cfg
    t = torch.empty((cfg.batch, cfg.q_heads, cfg.head_dim), dtype=torch_dtype(cfg.dtype),
                    device=device)
    fill_linear(t, wl.keys["q"], wl.q_base(step, layer), cfg.dtype)
    return t
