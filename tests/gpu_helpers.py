"""Helpers of the GPU parity tests: bit views, ulp distance, tolerances, and
the oracle's expectation for a workload (assembled from the shared input
generator and computed by oracle/ only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workload as W

# decode tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL, RTOL = 2e-3, 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(b: np.ndarray, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(dtype).to(device)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between 16-bit floats (sign-magnitude)."""
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    oa = np.where(a & 0x8000, -(a & 0x7FFF), a)
    ob = np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(oa - ob)


def assert_decode_close(got: np.ndarray, want: np.ndarray, what=""):
    err = np.abs(got - want) - (ATOL + RTOL * np.abs(want))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    worst = float(err.max()) if err.size else 0.0
    assert worst <= 0, f"{what}: beyond atol {ATOL} + rtol {RTOL}: excess {worst:.3e}"


def torch_dtype(code: int):
    return torch.float16 if code == W.FP16 else torch.bfloat16


# ---- expectations of a workload -------------------------------------------
def raw_rows(wl: W.Workload, layer: int, kv: int, r: int, positions: np.ndarray, h: int):
    """Stored (pre-RoPE) K or V rows [n][D] of request r at the given positions:
    pool rows for injected tokens, generator rows for appended / step tokens."""
    cfg = wl.cfg
    D = cfg.head_dim
    C = int(wl.context_lens[r])
    j_of, t_of = wl.source_of(r)
    positions = np.asarray(positions, np.int64)
    out = np.empty((positions.size, D), np.uint16)
    inside = positions < C
    inj = np.zeros(positions.size, bool)
    inj[inside] = j_of[positions[inside]] >= 0
    if inj.any():
        j = j_of[positions[inj]]
        t = t_of[positions[inj]]
        out[inj] = wl.pool_rows(wl.chunk_ids[j], np.full(j.size, layer), np.full(j.size, kv), t,
                                np.full(j.size, h))
    oth = ~inj
    if oth.any():
        base = wl.ctx_row_base(layer, kv, np.full(oth.sum(), r), positions[oth]) + h * D
        idx = base[:, None] + np.arange(D, dtype=np.int64)[None, :]
        out[oth] = W.normal_bits(wl.keys["ctx"], idx, cfg.dtype)
    return out


def expected_cache_rows(wl: W.Workload, layer: int, r: int, positions, h: int):
    """(K bits, V bits) the cache must hold for request r at these positions."""
    cfg = wl.cfg
    positions = np.asarray(positions, np.int64)
    k_raw = raw_rows(wl, layer, 0, r, positions, h)
    v_raw = raw_rows(wl, layer, 1, r, positions, h)
    k = oracle.rope_round_rows(k_raw, positions.astype(np.int32), cfg.theta, cfg.dtype)
    return k, v_raw


def expected_decode(wl: W.Workload, step: int, layer: int, r: int, qh: int):
    """fp64 oracle output of query head qh of request r at decode step `step`."""
    cfg = wl.cfg
    h = qh // cfg.group
    n = int(wl.context_lens[r]) + step + 1
    K, V = expected_cache_rows(wl, layer, r, np.arange(n), h)
    q = wl.q_rows(step, layer)[r, qh]
    return oracle.attention_bits(q, n - 1, cfg.theta, K, V, cfg.dtype)


def expected_request_rows(wl: W.Workload, layer: int, r: int, n: int):
    """(K bits, V bits) [Hkv][n][D] the cache must hold for request r's first n positions."""
    ks, vs = [], []
    for h in range(wl.cfg.kv_heads):
        k, v = expected_cache_rows(wl, layer, r, np.arange(n), h)
        ks.append(k)
        vs.append(v)
    return np.stack(ks), np.stack(vs)


def request_cache(k_rows: np.ndarray, v_rows: np.ndarray):
    """A one-request paged cache [1][NB][Hkv][16][D] (and its table) holding rows
    [Hkv][n][D] contiguously, for the oracle's paged decode."""
    Hkv, n, D = k_rows.shape
    NB = -(-n // 16)
    kc = np.zeros((1, NB * 16, Hkv, D), k_rows.dtype)
    vc = np.zeros_like(kc)
    kc[0, :n] = k_rows.transpose(1, 0, 2)
    vc[0, :n] = v_rows.transpose(1, 0, 2)
    kc = kc.reshape(1, NB, 16, Hkv, D).transpose(0, 1, 3, 2, 4).copy()
    vc = vc.reshape(1, NB, 16, Hkv, D).transpose(0, 1, 3, 2, 4).copy()
    return kc, vc, np.arange(NB, dtype=np.int32)[None]


def gpu_request_rows(cache_k: np.ndarray, cache_v: np.ndarray, layer: int, bt_row: np.ndarray,
                     n: int):
    """Rows [Hkv][n][...] of a request's first n positions gathered from host copies of the
    GPU cache ([L][NB][Hkv][16][...]) through its block table (values: plain indexing)."""
    p = np.arange(n)
    blk = bt_row[p // 16]
    return cache_k[layer, blk, :, p % 16].transpose(1, 0, 2), \
        cache_v[layer, blk, :, p % 16].transpose(1, 0, 2)
