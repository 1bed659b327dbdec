"""A GPU-resident paged KV-injection engine built on the C ABI.

Holds what lives in HBM across requests -- the pre-RoPE chunk pool (the
store InferScale keeps resident, its §3.1 and §6.7), the paged KV cache of
all layers, the RoPE table and the decode workspace -- and runs one step of
the hot path through the library's kernels:

    slot mapping -> inject (all layers) -> per decode step, per layer:
    append the new token's K/V, paged decode attention (one fused call:
    kvinj_append_paged_decode)

Every operation here is a call into libkvinj.so; this module only sequences
the calls and owns the buffers. ``step_from_host`` is the end-to-end form a
caller with host-side request data uses: it copies the step's inputs from
pinned host memory, runs the step and copies the outputs back.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import kvinj as K


@dataclass
class StepInputs:
    """Device tensors of one step (one batch of requests)."""
    chunk_ids: torch.Tensor     # int32 [n_inj]
    start_pos: torch.Tensor     # int32 [n_inj]
    map_seq: torch.Tensor       # int32 [n_inj*c + steps*batch]: injected tokens, then step tokens
    map_pos: torch.Tensor       # int32 [same]
    block_tables: torch.Tensor  # int32 [batch][max_blocks]
    ctx_lens: torch.Tensor      # int32 [steps][batch]: context length seen by each decode step
    q_pos: torch.Tensor         # int32 [steps][batch]: position of each step's new token
    q: torch.Tensor             # [steps][L][batch][Hq][D]   pre-RoPE queries
    k_new: torch.Tensor         # [steps][L][batch][Hkv][D]  pre-RoPE keys of the new tokens
    v_new: torch.Tensor         # [steps][L][batch][Hkv][D]

    def tensors(self):
        return [self.chunk_ids, self.start_pos, self.map_seq, self.map_pos, self.block_tables,
                self.ctx_lens, self.q_pos, self.q, self.k_new, self.v_new]

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.tensors())


class Engine:
    """kv: "16" keeps the cache in the pool's 16-bit type; "int8" keeps it as int8 codes with
    one fp32 scale per row ("Latency Optimization > KV Cache Management", KV cache
    quantization), written by kvinj_inject_i8 / kvinj_append_i8 and read by
    kvinj_paged_decode_i8 (D = 128; block copies, prefill and the sliding window are
    16-bit calls)."""

    def __init__(self, *, layers: int, q_heads: int, kv_heads: int, head_dim: int,
                 block_size: int, dtype: torch.dtype, num_blocks: int, max_pos: int,
                 theta: float, batch: int, pool: torch.Tensor, device="cuda", kv: str = "16"):
        self.L, self.Hq, self.Hkv, self.D, self.B = layers, q_heads, kv_heads, head_dim, block_size
        self.dtype, self.batch, self.device = dtype, batch, device
        assert kv in ("16", "int8")
        self.kv = kv
        shape = (layers, num_blocks, kv_heads, block_size, head_dim)
        if kv == "int8":
            self.k_cache = self.v_cache = None
            self.cache = K.CacheI8.empty(layers, num_blocks, kv_heads, head_dim, block_size,
                                         device)
        else:
            self.k_cache = torch.empty(shape, dtype=dtype, device=device)
            self.v_cache = torch.empty(shape, dtype=dtype, device=device)
            self.cache = K.Cache(self.k_cache, self.v_cache)
        self.pool = K.Pool(pool)
        self.chunk_len = pool.shape[3]
        self.rope = K.make_rope(theta, head_dim, max_pos, device)
        self.workspace = K.make_decode_workspace(batch, q_heads, kv_heads, head_dim, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.decode_variant = 0
        self.decode_ctas = 0
        self.fused_append = True  # append + decode in one call
        self.overlap_inject = False  # inject on a low-priority stream beside the decode
        self.window = 0  # sliding window of the decode in tokens (0: whole context)
        # let decode calls after the first of a step stream their first pages before the
        # kernel ahead of them ends (KVINJ_DECODE_KV_READY). Off by default: on one GB300 it
        # took the multi-head fp16 70B-shaped layer from 88.2 to 85.3 us but added 0.6-1.0 us
        # to the GQA-shaped ones, whose stage ring, not the launch gap, sets the pace
        self.early_kv = False
        self._prefill_ws = None
        self._hi = self._lo = None

    # -- single operations ---------------------------------------------------
    def slot_mapping(self, block_tables, seq, pos, out=None):
        if out is None:
            out = torch.empty(pos.numel(), dtype=torch.int64, device=self.device)
        return K.kvinj_slot_mapping(block_tables, seq, pos, self.cache.num_blocks, self.B, out,
                                    self.status)

    def inject(self, chunk_ids, start_pos, slots, layer_begin=0, layer_end=None):
        if self.kv == "int8":
            K.kvinj_inject_i8(self.pool, self.cache, self.rope, chunk_ids, start_pos, slots,
                              layer_begin, layer_end, self.status)
            return
        K.kvinj_inject(self.pool, self.cache, self.rope, chunk_ids, start_pos, slots,
                       layer_begin, layer_end, self.status)

    def append(self, layer, k_new, v_new, positions, slots, rotate=True):
        if self.kv == "int8":
            K.kvinj_append_i8(self.cache, self.rope if rotate else None, layer, k_new, v_new,
                              positions, slots, self.status)
            return
        K.kvinj_append(self.cache, self.rope if rotate else None, layer, k_new, v_new,
                       positions, slots, self.status)

    def decode(self, layer, q, q_pos, block_tables, ctx_lens, out, rotate=True, kv_ready=False):
        """kv_ready: the pages of `layer`, the tables, lengths and q positions were written
        before the previous decode call on the stream, which was on another layer
        (KVINJ_DECODE_KV_READY: the call may stream pages before the kernel ahead ends)."""
        flags = K.KVINJ_DECODE_KV_READY if kv_ready and self.early_kv else 0
        if self.kv == "int8":
            K.kvinj_paged_decode_i8(self.cache, self.rope if rotate else None, layer, q, q_pos,
                                    block_tables, ctx_lens, out, self.workspace,
                                    status=self.status, ctas=self.decode_ctas)
            return
        if self.window:
            K.kvinj_paged_decode_window(self.cache, self.rope if rotate else None, layer, q, q_pos,
                                        block_tables, ctx_lens, self.window, out, self.workspace,
                                        status=self.status, flags=flags)
            return
        K.kvinj_paged_decode_ex(self.cache, self.rope if rotate else None, layer, q, q_pos,
                                block_tables, ctx_lens, out, self.workspace, 0.0, self.status,
                                None, self.decode_variant, self.decode_ctas, flags)

    def append_decode(self, layer, q, k_new, v_new, q_pos, block_tables, ctx_lens, out,
                      rotate=True, kv_ready=False):
        """Append + decode in one call; kv_ready as in decode()."""
        flags = K.KVINJ_DECODE_KV_READY if kv_ready and self.early_kv else 0
        if self.kv == "int8":
            K.kvinj_paged_decode_i8(self.cache, self.rope if rotate else None, layer, q, q_pos,
                                    block_tables, ctx_lens, out, self.workspace, k_new=k_new,
                                    v_new=v_new, status=self.status, ctas=self.decode_ctas)
            return
        if self.window:
            K.kvinj_paged_decode_window(self.cache, self.rope if rotate else None, layer, q, q_pos,
                                        block_tables, ctx_lens, self.window, out, self.workspace,
                                        k_new=k_new, v_new=v_new, status=self.status, flags=flags)
            return
        K.kvinj_append_paged_decode(self.cache, self.rope if rotate else None, layer, q, k_new,
                                    v_new, q_pos, block_tables, ctx_lens, out, self.workspace,
                                    0.0, self.status, None, self.decode_variant,
                                    self.decode_ctas, flags)

    def prefill(self, layer, q, seq_ids, positions, block_tables, out, rotate=True):
        """Query tokens q[n] of requests seq_ids[n] at positions[n] (K/V already appended),
        each attending causally to its request's tokens 0..position."""
        need = K.kvinj_prefill_workspace_size(q.shape[0], self.Hq, self.Hkv, self.D,
                                              block_tables.shape[1])
        if self._prefill_ws is None or self._prefill_ws.numel() < need:
            self._prefill_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        K.kvinj_paged_prefill(self.cache, self.rope if rotate else None, layer, q, seq_ids,
                              positions, block_tables, out, self._prefill_ws, status=self.status)

    def copy_blocks(self, src: torch.Tensor, dst: torch.Tensor, layer_begin: int = 0,
                    layer_end: int | None = None):
        """Copy-on-write: physical block src[i] -> dst[i] in every layer (K and V)."""
        K.kvinj_copy_blocks(self.cache, src, dst, layer_begin, layer_end, self.status)

    def uses_tcgen05(self) -> bool:
        """Whether decode runs a tcgen05 kernel (one launch per layer)."""
        if self.kv == "int8":
            return True
        G = self.Hq // self.Hkv
        ok = self.D == 128 and self.Hkv % 8 == 0 and G in (1, 2, 4, 8)  # the automatic choice
        return self.decode_variant == 3 or (self.decode_variant == 0 and ok)

    def launches_per_layer(self) -> int:
        """Kernel launches of one layer's append + decode."""
        if self.uses_tcgen05() and self.fused_append:
            return 2  # split-K pass with the append, combine pass
        return 3  # append, split-K pass, combine pass

    # -- one step of the hot path --------------------------------------------
    def alloc_outputs(self, steps: int) -> torch.Tensor:
        return torch.empty((steps, self.L, self.batch, self.Hq, self.D), dtype=self.dtype,
                           device=self.device)

    def _layer(self, s, layer, inp: StepInputs, out, step_slots, timer=None):
        """Append + decode of one layer of decode step s. Every call but the first of the
        step follows a decode call on another layer (or, with one layer, on the same one),
        after the inject: such a call may read its pages before the kernel ahead ends."""
        ready = (s > 0 or layer > 0) and self.L > 1 and timer is None
        if self.fused_append:
            # the step token's slot is the one its block table gives
            if timer:
                timer("decode", 0)
            self.append_decode(layer, inp.q[s, layer], inp.k_new[s, layer], inp.v_new[s, layer],
                               inp.q_pos[s], inp.block_tables, inp.ctx_lens[s], out[s, layer],
                               kv_ready=ready)
            if timer:
                timer("decode", 1)
            return
        self.append(layer, inp.k_new[s, layer], inp.v_new[s, layer], inp.q_pos[s], step_slots[s])
        if timer:
            timer("decode", 0)
        # the append kernel just before writes this layer's pages: no early reads
        self.decode(layer, inp.q[s, layer], inp.q_pos[s], inp.block_tables, inp.ctx_lens[s],
                    out[s, layer])
        if timer:
            timer("decode", 1)

    def _streams(self):
        if self._hi is None:
            # out-of-range priorities map to the device's highest / lowest
            self._hi = torch.cuda.Stream(device=self.device, priority=-100)
            self._lo = torch.cuda.Stream(device=self.device, priority=100)
        return self._hi, self._lo

    def step(self, inp: StepInputs, out: torch.Tensor, timer=None):
        """slot mapping + inject + (append, decode) per step and layer.

        With `overlap_inject` (and no timer), the inject runs layer by layer on a
        low-priority stream while the decode layers run on a high-priority one;
        decode of layer l waits for the inject of layer l only. The two are
        independent HBM traffic: the inject fills the DRAM time the decode
        launches leave idle (their start, tail and combine pass). The result is
        the same as the serial order.

        `timer`, when given, is called as timer(kind, stream_event_pair_index)
        around the inject and decode launches (used for per-kernel timing)."""
        n_tok = inp.map_pos.numel()
        slots = self.slot_mapping(inp.block_tables, inp.map_seq, inp.map_pos)
        n_inj_tok = inp.chunk_ids.numel() * self.chunk_len
        steps = inp.q.shape[0]
        step_slots = slots[n_inj_tok:n_tok].view(steps, self.batch)
        if self.overlap_inject and timer is None:
            cur = torch.cuda.current_stream(self.device)
            hi, lo = self._streams()
            lo.wait_stream(cur)
            hi.wait_stream(cur)
            ready = [torch.cuda.Event() for _ in range(self.L)]
            with torch.cuda.stream(lo):
                for layer in range(self.L):
                    self.inject(inp.chunk_ids, inp.start_pos, slots[:n_inj_tok], layer, layer + 1)
                    ready[layer].record(lo)
            with torch.cuda.stream(hi):
                for s in range(steps):
                    for layer in range(self.L):
                        if s == 0:
                            hi.wait_event(ready[layer])
                        self._layer(s, layer, inp, out, step_slots)
            cur.wait_stream(hi)
            cur.wait_stream(lo)
            return out
        if timer:
            timer("inject", 0)
        self.inject(inp.chunk_ids, inp.start_pos, slots[:n_inj_tok])
        if timer:
            timer("inject", 1)
        for s in range(steps):
            for layer in range(self.L):
                self._layer(s, layer, inp, out, step_slots, timer)
        return out

    def capture(self, inp: StepInputs, out: torch.Tensor, timer=None) -> torch.cuda.CUDAGraph:
        """Capture one step (all its launches) into a CUDA graph. The graph reads
        the tensors of `inp` and writes `out` in place: refill them, replay."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(inp, out, timer=timer)
        return g

    def step_from_host(self, host: StepInputs, dev: StepInputs, out: torch.Tensor,
                       host_out: torch.Tensor, graph: torch.cuda.CUDAGraph | None = None):
        """End to end: pinned host inputs -> device, step (or its captured graph),
        outputs -> pinned host."""
        for h, d in zip(host.tensors(), dev.tensors()):
            d.copy_(h, non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            self.step(dev, out)
        host_out.copy_(out, non_blocking=True)
        return host_out
