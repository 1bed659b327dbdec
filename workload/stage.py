"""Put a seeded workload on the GPU: the chunk pool, the engine, the context
tokens that precede the measured step, and the inputs of one step.

Harness code for the tests, the smoke check and the benchmark. Values come
from ``workload.device`` (bit-identical to the host generator); every
computation is a call into the CUDA library through the engine.
"""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_inject_gb300.engine import Engine, StepInputs

from . import Workload
from . import device as gen


def make_engine(wl: Workload, device="cuda", pool: torch.Tensor | None = None,
                kv: str = "16") -> Engine:
    cfg = wl.cfg
    if pool is None:
        pool = gen.pool_tensor(wl, device)
    return Engine(layers=cfg.layers, q_heads=cfg.q_heads, kv_heads=cfg.kv_heads,
                  head_dim=cfg.head_dim, block_size=cfg.block_size,
                  dtype=gen.torch_dtype(cfg.dtype), num_blocks=wl.num_blocks,
                  max_pos=wl.max_pos, theta=cfg.theta, batch=cfg.batch, pool=pool, device=device,
                  kv=kv)


def compact_pool(wl: Workload, device="cuda"):
    """Only the chunks this batch draws, with their values (same bits as the
    full pool): returns (pool tensor, remapped chunk ids int32). The kernels
    and the bytes they move are those of the full pool; only capacity differs."""
    cfg = wl.cfg
    ids = np.unique(wl.chunk_ids)
    t = torch.empty((ids.size, cfg.layers, 2, cfg.chunk_len, cfg.kv_heads, cfg.head_dim),
                    dtype=gen.torch_dtype(cfg.dtype), device=device)
    keep = gen.fill_rows(t, ids.astype(np.int64) * cfg.chunk_elems, wl.keys["pool"], cfg.dtype)
    torch.cuda.synchronize()
    del keep
    return t, np.searchsorted(ids, wl.chunk_ids).astype(np.int32)


def _i32(a, device):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)


def fill_context(eng: Engine, wl: Workload, device="cuda", max_tokens: int = 1 << 16):
    """Append the context tokens that are not injected (all layers), as the
    tokens before the step would have been written."""
    seq, pos = wl.appended_tokens()
    bt = _i32(wl.block_tables, device)
    for o in range(0, seq.size, max_tokens):
        s, p = seq[o:o + max_tokens], pos[o:o + max_tokens]
        seq_d, pos_d = _i32(s, device), _i32(p, device)
        slots = eng.slot_mapping(bt, seq_d, pos_d)
        for layer in range(wl.cfg.layers):
            kn, keep_k = gen.ctx_rows(wl, layer, 0, s, p, device)
            vn, keep_v = gen.ctx_rows(wl, layer, 1, s, p, device)
            eng.append(layer, kn, vn, pos_d, slots)
            del keep_k, keep_v
    torch.cuda.synchronize()


def step_inputs(wl: Workload, device="cuda") -> StepInputs:
    cfg = wl.cfg
    S, L, Bt = cfg.steps, cfg.layers, cfg.batch
    inj_seq, inj_pos = wl.injected_tokens()
    step_seq = np.tile(np.arange(Bt, dtype=np.int32), S)
    step_pos = (wl.context_lens[None, :] + np.arange(S, dtype=np.int32)[:, None]).astype(np.int32)
    dt = gen.torch_dtype(cfg.dtype)
    q = torch.empty((S, L, Bt, cfg.q_heads, cfg.head_dim), dtype=dt, device=device)
    gen.fill_linear(q, wl.keys["q"], 0, cfg.dtype)  # q_base(s, l) is contiguous in (s, l)
    kv = []
    for kvi in (0, 1):
        t = torch.empty((S, L, Bt, cfg.kv_heads, cfg.head_dim), dtype=dt, device=device)
        base = np.stack([np.stack([wl.ctx_row_base(layer, kvi, np.arange(Bt), step_pos[s])
                                   for layer in range(L)]) for s in range(S)])
        keep = gen.fill_rows(t, base.reshape(-1), wl.keys["ctx"], cfg.dtype)
        kv.append((t, keep))
    inp = StepInputs(
        chunk_ids=_i32(wl.chunk_ids, device),
        start_pos=_i32(wl.start_pos, device),
        map_seq=_i32(np.concatenate([inj_seq, step_seq]), device),
        map_pos=_i32(np.concatenate([inj_pos, step_pos.reshape(-1)]), device),
        block_tables=_i32(wl.block_tables, device),
        ctx_lens=_i32(step_pos + 1, device),
        q_pos=_i32(step_pos, device),
        q=q, k_new=kv[0][0], v_new=kv[1][0],
    )
    torch.cuda.synchronize()
    return inp


def pinned_copy(inp: StepInputs) -> StepInputs:
    """Pinned host copies of a step's inputs (for the end-to-end measurement)."""
    return StepInputs(*[t.cpu().pin_memory() for t in inp.tensors()])


def algorithmic_bytes(wl: Workload, window: int = 0, kv: str = "16") -> dict:
    """Bytes one step must move at minimum, per part (the roofline numerator).

    inject: read the injected chunks' K/V rows and write them to the cache,
            2 * (2 * L * Hkv * D * b) per injected token;
    append: the same per new token and layer, read + write;
    decode: read every context token's K and V once per layer and step (under a sliding
            window of `window` tokens only the last `window`), plus q, out and the
            block-table entries of the pages read.
    With the int8 cache (kv = "int8") a cached row is D code bytes and a 4-byte scale
    instead of D 16-bit values: reads of the 16-bit pool and new tokens stay 16-bit."""
    cfg = wl.cfg
    b = cfg.elem_bytes
    row16 = cfg.kv_heads * cfg.head_dim * b
    row = cfg.kv_heads * (cfg.head_dim + 4) if kv == "int8" else row16
    n_inj_tok = wl.n_inj * cfg.chunk_len
    inject = 2 * cfg.layers * (row16 + row) * n_inj_tok
    append = 2 * (row16 + row) * cfg.batch * cfg.layers * cfg.steps
    decode = 0
    for s in range(cfg.steps):
        ctx = wl.context_lens.astype(np.int64) + s + 1
        lo = np.maximum(ctx - window, 0) if window > 0 else np.zeros_like(ctx)
        pages = -(-ctx // cfg.block_size) - lo // cfg.block_size
        kv_bytes = int((ctx - lo).sum()) * 2 * row
        small = cfg.batch * cfg.q_heads * cfg.head_dim * b * 2 + int(pages.sum()) * 4
        decode += cfg.layers * (kv_bytes + small)
    return {"inject": inject, "append": append, "decode": decode,
            "total": inject + append + decode}
