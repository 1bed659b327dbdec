"""Seeded synthetic workloads for paged KV injection + paged GQA decode.

This module holds no arithmetic of the method itself. It only produces inputs:
the shapes of the five workloads (Llama-3-8B/70B-shaped GQA, a multi-head
70B shape, a mixed-length load, and a tiny case), the integer structure of a
batch (context lengths, which chunks each request injects and where, block
tables drawn from a shuffled physical-block pool), and the bulk values
(pre-RoPE chunk K/V, the K/V of the tokens that are appended, the queries).

Bulk values are a pure function of (stream key, element index): a SplitMix64
hash (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) of the index, whose four 16-bit fields are summed
(an Irwin-Hall sum of four uniforms), centred, scaled to unit variance in one
fp32 multiply and rounded to the 16-bit cache type (nearest-even). The host
implementation here and the CUDA fill kernels in ``workload/csrc/kvgen.cu``
compute the same bits; the tests check that. Both the CUDA path and the
oracle read their inputs from these generators and from nothing else.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import numpy as np

BF16, FP16 = 0, 1
DTYPE_NAMES = {BF16: "bf16", FP16: "fp16"}

# ---------------------------------------------------------------------------
# counter-based generator (host side)
# ---------------------------------------------------------------------------
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# the Irwin-Hall sum of four uniform 16-bit integers has variance
# 4 * (65536^2 - 1) / 12; this fp32 factor scales it to unit variance
NORMAL_SCALE = np.float32(1.0 / math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0))
NORMAL_CENTRE = 2 * 65535  # mean of the four-field sum

STREAM_POOL, STREAM_CTX, STREAM_Q = 1, 2, 3


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def hash64(key: int, idx) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + (idx + np.uint64(1)) * _GAMMA)


def stream_key(seed: int, stream: int) -> int:
    with np.errstate(over="ignore"):
        v = _mix64(np.array([(seed << 8) | stream], dtype=np.uint64))
    return int(v[0])


def normal_f32(key: int, idx) -> np.ndarray:
    """Approximately N(0,1) fp32 values for the given element indices."""
    h = hash64(key, idx)
    m = np.uint64(0xFFFF)
    s = (h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m) + (h >> np.uint64(48))
    return (s.astype(np.int64) - NORMAL_CENTRE).astype(np.float32) * NORMAL_SCALE


def f32_to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round fp32 to bf16/fp16 (nearest-even) and return the bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == FP16:
        return x.astype(np.float16).view(np.uint16)
    b = x.view(np.uint32).astype(np.uint64)
    return ((b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)


def normal_bits(key: int, idx, dtype: int) -> np.ndarray:
    return f32_to_bits(normal_f32(key, idx), dtype)


# ---------------------------------------------------------------------------
# workload shapes
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Config:
    name: str
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    block_size: int
    dtype: int
    batch: int
    ctx: tuple                 # ("fixed", C) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    chunks_per_req: int
    chunk_len: int
    pool_chunks: int
    steps: int
    theta: float
    occupancy: float = 1.0     # fraction of the physical-block pool in use
    fixed_starts: tuple = ()   # chunk start positions, when the workload fixes them
    fixed_num_blocks: int = 0  # physical pool size, when the workload fixes it
    draw_once: bool = False    # every pool chunk drawn exactly once across the batch
    seed: int = 0

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def elem_bytes(self) -> int:
        return 2

    @property
    def chunk_elems(self) -> int:
        return 2 * self.layers * self.chunk_len * self.kv_heads * self.head_dim

    @property
    def pool_bytes(self) -> int:
        return self.pool_chunks * self.chunk_elems * self.elem_bytes

    def scaled(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    # 1 layer, 2 q / 1 kv heads, d 64, 8 physical blocks, one request of 64
    # tokens with chunks at 16 and 40, theta 1e4
    "tiny_1layer": Config("tiny_1layer", 1, 2, 1, 64, 16, BF16, 1, ("fixed", 64), 2, 16, 4, 1,
                          1e4, fixed_starts=(16, 40), fixed_num_blocks=8, seed=1001),
    # Llama-3-8B-shaped: 32 layers, 32/8 heads, d 128, batch 32, ctx U[512, 2048],
    # 8 chunks of 64 tokens per request from 4096, theta 5e5
    "llama3_8b_b32": Config("llama3_8b_b32", 32, 32, 8, 128, 16, BF16, 32, ("uniform", 512, 2048),
                            8, 64, 4096, 1, 5e5, seed=1002),
    # Llama-3-70B-shaped: 80 layers, 64/8 heads, batch 8, ctx 8192, 64 chunks of 32
    # tokens from 16384, 16 decode steps
    "llama3_70b_b8_8k": Config("llama3_70b_b8_8k", 80, 64, 8, 128, 16, BF16, 8, ("fixed", 8192),
                               64, 32, 16384, 16, 5e5, seed=1003),
    # multi-head 70B shape, fp16: 80 layers, 64/64 heads, batch 4, ctx 4096, 1024
    # injected tokens as 16-token chunks, theta 1e4
    "mha70b_b4_4k_fp16": Config("mha70b_b4_4k_fp16", 80, 64, 64, 128, 16, FP16, 4, ("fixed", 4096),
                                64, 16, 256, 1, 1e4, draw_once=True, seed=1004),
    # mixed lengths: 32 layers, 32/8 heads, batch 64, ctx log-uniform [16, 32768],
    # 32 chunks of 16 tokens from 100000, block pool at 90 % occupancy
    "mixed_b64_loguniform": Config("mixed_b64_loguniform", 32, 32, 8, 128, 16, BF16, 64,
                                   ("loguniform", 16, 32768), 32, 16, 100000, 1, 5e5,
                                   occupancy=0.9, seed=1005),
}
CONFIG_ORDER = ["tiny_1layer", "llama3_8b_b32", "llama3_70b_b8_8k", "mha70b_b4_4k_fp16",
                "mixed_b64_loguniform"]


# ---------------------------------------------------------------------------
# one batch of the workload: integer structure + value streams
# ---------------------------------------------------------------------------
@dataclass
class Workload:
    cfg: Config
    context_lens: np.ndarray      # int32 [batch]   tokens before the decode steps
    chunk_ids: np.ndarray         # int32 [n_inj]   pool chunk of each injected chunk
    chunk_req: np.ndarray         # int32 [n_inj]   request of each injected chunk
    start_pos: np.ndarray         # int32 [n_inj]   absolute position of its first token
    block_tables: np.ndarray      # int32 [batch][max_blocks], -1 past the end
    num_blocks: int
    keys: dict = field(default_factory=dict)

    # ---- derived structure -------------------------------------------------
    @property
    def batch(self) -> int:
        return self.cfg.batch

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    @property
    def n_inj(self) -> int:
        return int(self.chunk_ids.size)

    @property
    def max_pos(self) -> int:
        """Positions 0 .. max_pos-1 occur (context plus the decode steps)."""
        return int(self.context_lens.max()) + self.cfg.steps

    def injected_tokens(self):
        """(seq_ids, positions) of every injected token, chunk-major."""
        c = self.cfg.chunk_len
        seq = np.repeat(self.chunk_req, c).astype(np.int32)
        pos = (self.start_pos[:, None] + np.arange(c, dtype=np.int32)[None, :]).reshape(-1)
        return seq, pos.astype(np.int32)

    def injected_mask(self, r: int) -> np.ndarray:
        m = np.zeros(int(self.context_lens[r]), bool)
        c = self.cfg.chunk_len
        for s in self.start_pos[self.chunk_req == r]:
            m[s:s + c] = True
        return m

    def appended_tokens(self):
        """(seq_ids, positions) of the context tokens that are not injected."""
        seqs, poss = [], []
        for r in range(self.batch):
            p = np.nonzero(~self.injected_mask(r))[0].astype(np.int32)
            seqs.append(np.full(p.size, r, np.int32))
            poss.append(p)
        return np.concatenate(seqs), np.concatenate(poss)

    def step_tokens(self, step: int):
        """(seq_ids, positions) of the tokens appended by decode step `step`."""
        r = np.arange(self.batch, dtype=np.int32)
        return r, (self.context_lens + step).astype(np.int32)

    def source_of(self, r: int):
        """Per position of request r's context: (chunk index j, offset t) of the
        injected chunk covering it, or (-1, -1) for appended tokens."""
        C = int(self.context_lens[r])
        j_of = np.full(C, -1, np.int64)
        t_of = np.full(C, -1, np.int64)
        c = self.cfg.chunk_len
        for j in np.nonzero(self.chunk_req == r)[0]:
            s = int(self.start_pos[j])
            j_of[s:s + c] = j
            t_of[s:s + c] = np.arange(c)
        return j_of, t_of

    # ---- value streams (host) ----------------------------------------------
    def pool_index(self, chunk, layer, kv, t, h):
        """Flat element index of pool[chunk][layer][kv][t][h][0]."""
        cfg = self.cfg
        chunk, layer, kv, t, h = (np.asarray(a, np.int64) for a in (chunk, layer, kv, t, h))
        return ((((chunk * cfg.layers + layer) * 2 + kv) * cfg.chunk_len + t) * cfg.kv_heads + h) * cfg.head_dim

    def pool_rows(self, chunk, layer, kv, t, h) -> np.ndarray:
        """Stored pre-RoPE rows [n][D] (bits) of the chunk pool."""
        base = np.atleast_1d(self.pool_index(chunk, layer, kv, t, h))
        idx = base[:, None] + np.arange(self.cfg.head_dim, dtype=np.int64)[None, :]
        return normal_bits(self.keys["pool"], idx, self.cfg.dtype)

    def ctx_row_base(self, layer: int, kv: int, seq, pos) -> np.ndarray:
        """Flat index of element [h=0][d=0] of an appended token's K (kv=0) or V
        (kv=1) in the virtual array [L][2][batch][max_pos][Hkv][D]."""
        cfg = self.cfg
        seq = np.asarray(seq, np.int64)
        pos = np.asarray(pos, np.int64)
        return (((layer * 2 + kv) * cfg.batch + seq) * self.max_pos + pos) * cfg.kv_heads * cfg.head_dim

    def ctx_rows(self, layer: int, kv: int, seq, pos) -> np.ndarray:
        """Appended tokens' pre-RoPE K or V, bits [n][Hkv][D]."""
        cfg = self.cfg
        base = np.atleast_1d(self.ctx_row_base(layer, kv, seq, pos))
        idx = base[:, None] + np.arange(cfg.kv_heads * cfg.head_dim, dtype=np.int64)[None, :]
        return normal_bits(self.keys["ctx"], idx, cfg.dtype).reshape(-1, cfg.kv_heads, cfg.head_dim)

    def q_base(self, step: int, layer: int) -> int:
        cfg = self.cfg
        return (step * cfg.layers + layer) * cfg.batch * cfg.q_heads * cfg.head_dim

    def q_rows(self, step: int, layer: int) -> np.ndarray:
        """Pre-RoPE queries, bits [batch][Hq][D]."""
        cfg = self.cfg
        n = cfg.batch * cfg.q_heads * cfg.head_dim
        idx = self.q_base(step, layer) + np.arange(n, dtype=np.int64)
        return normal_bits(self.keys["q"], idx, cfg.dtype).reshape(cfg.batch, cfg.q_heads, cfg.head_dim)

    # ---- sizes -------------------------------------------------------------
    def cache_shape(self):
        cfg = self.cfg
        return (cfg.layers, self.num_blocks, cfg.kv_heads, cfg.block_size, cfg.head_dim)

    @property
    def cache_bytes(self) -> int:
        return 2 * int(np.prod(self.cache_shape())) * self.cfg.elem_bytes


def _context_lengths(cfg: Config, rng) -> np.ndarray:
    kind = cfg.ctx[0]
    if kind == "fixed":
        return np.full(cfg.batch, cfg.ctx[1], np.int32)
    lo, hi = cfg.ctx[1], cfg.ctx[2]
    if kind == "uniform":
        return rng.integers(lo, hi + 1, cfg.batch).astype(np.int32)
    if kind == "loguniform":
        v = np.exp(rng.uniform(math.log(lo), math.log(hi), cfg.batch))
        return np.clip(np.rint(v), lo, hi).astype(np.int32)
    raise ValueError(kind)


def make_workload(cfg: Config, seed: int | None = None) -> Workload:
    """Draw one batch of `cfg` from a seeded generator (exactly reproducible)."""
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    C = _context_lengths(cfg, rng)
    c = cfg.chunk_len
    # chunks per request: as many as the configuration asks, never more than fit
    k = np.minimum(cfg.chunks_per_req, C // c).astype(np.int64)
    # which pool chunks: distinct within a request (repeats across requests are
    # the point of a reusable store), or every chunk once when the workload says so
    if cfg.draw_once:
        assert k.sum() <= cfg.pool_chunks
        perm = rng.permutation(cfg.pool_chunks)
        ids = [perm[int(k[:r].sum()):int(k[:r + 1].sum())] for r in range(cfg.batch)]
    else:
        ids = [rng.choice(cfg.pool_chunks, size=int(k[r]), replace=False) for r in range(cfg.batch)]
    # where: non-overlapping offsets inside [0, C_r) -- sorted gaps (stars and bars)
    starts = []
    for r in range(cfg.batch):
        if cfg.fixed_starts:
            starts.append(np.array(cfg.fixed_starts[:k[r]], np.int64))
            continue
        free = int(C[r]) - int(k[r]) * c
        u = np.sort(rng.integers(0, free + 1, int(k[r])))
        starts.append(u + np.arange(int(k[r])) * c)
    # block tables from a shuffled physical pool
    blocks = -(-(C.astype(np.int64) + cfg.steps) // cfg.block_size)
    total = int(blocks.sum())
    if cfg.fixed_num_blocks:
        num_blocks = cfg.fixed_num_blocks
        assert total <= num_blocks
    else:
        num_blocks = int(math.ceil(total / cfg.occupancy))
    perm = rng.permutation(num_blocks).astype(np.int32)
    if cfg.fixed_num_blocks and cfg.batch == 1:
        max_blocks = num_blocks  # the whole permutation is the table
        bt = perm.reshape(1, -1)
    else:
        max_blocks = int(blocks.max())
        bt = np.full((cfg.batch, max_blocks), -1, np.int32)
        o = 0
        for r in range(cfg.batch):
            bt[r, :blocks[r]] = perm[o:o + blocks[r]]
            o += int(blocks[r])
    wl = Workload(
        cfg=cfg,
        context_lens=C,
        chunk_ids=np.concatenate(ids).astype(np.int32),
        chunk_req=np.repeat(np.arange(cfg.batch), k).astype(np.int32),
        start_pos=np.concatenate(starts).astype(np.int32),
        block_tables=bt,
        num_blocks=num_blocks,
    )
    wl.keys = {"pool": stream_key(seed, STREAM_POOL), "ctx": stream_key(seed, STREAM_CTX),
               "q": stream_key(seed, STREAM_Q)}
    return wl
