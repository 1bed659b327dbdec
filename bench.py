"""Benchmark of the paged KV-injection hot path on GB300.

One step = one pass of the whole hot path over one batch of requests. The
default workload is the largest one that fits one GPU, Llama-3-70B-shaped
(80 layers, 64 q / 8 kv heads, d 128, bf16, block 16, batch 8, contexts of
8192 tokens, 64 injected chunks of 32 tokens per request from a resident
pool of 16384 pre-RoPE chunks, 16 decode steps with per-step append):

    slot mapping -> inject (gather, RoPE, scatter; all layers) ->
    per decode step and layer: append the new token's K/V, paged GQA decode

The headline `value` is the step's algorithmic HBM traffic (bytes the step
must move at minimum: injected chunk rows read and written, appended rows,
every context K/V row read once per layer, plus q/out/block tables) divided
by the step time, in GB/s; the injection rate (injected tokens/s) and the
decode bandwidth are reported beside it. Inputs are resident in HBM when the
timed region starts and larger than L2 (no flush needed); `e2e` repeats the
measurement through the engine's host-buffer entry point with the per-step
inputs copied from pinned host memory and the outputs copied back. The other
target workloads (Llama-3-8B-shaped, multi-head 70B fp16, mixed lengths) are
measured in the same run, each step timed the same way, under
parts.other_workloads.

--impl reference times the fp64 CPU oracle on a bounded sample (layer 0 of
the same workload) on this machine's host cores. For N > 1 (torchrun) every
rank runs an independent replica on its own GPU (the path has no exchange
step); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode HBM GB/s (% of ~8 TB/s); KV-injection tokens/s"
NOMINAL_HBM_GBS = 8000.0
DEFAULT_CONFIG = "llama3_70b_b8_8k"
# the other workloads whose steps the same run measures (reported under parts.other_workloads)
OTHER_WORKLOADS = ["llama3_8b_b32", "mha70b_b4_4k_fp16", "mixed_b64_loguniform"]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# replicas: nothing on the path exchanges data between GPUs; each rank runs
# its own batch and only the timing is reduced
# ---------------------------------------------------------------------------
def workload_config(cfg, window: int = 0) -> dict:
    """The workload's identity in the JSON line (shared by both arms)."""
    c = {"workload": cfg.name, "layers": cfg.layers, "q_heads": cfg.q_heads,
         "kv_heads": cfg.kv_heads, "head_dim": cfg.head_dim, "block_size": cfg.block_size,
         "batch": cfg.batch, "context": list(cfg.ctx),
         "injected_chunks_per_request": cfg.chunks_per_req, "chunk_len": cfg.chunk_len,
         "pool_chunks": cfg.pool_chunks, "decode_steps": cfg.steps}
    if window:
        c["decode_window"] = window  # sliding window: the last `window` tokens of each context
    return c


def replica_seed(cfg_seed: int, rank: int) -> int:
    """Seed of rank `rank`'s batch: an independent replica per rank."""
    return cfg_seed + 1000 * rank


def max_over_ranks(x: float, device) -> float:
    """The maximum of a per-rank scalar over all ranks (the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank: int, ms: float) -> float:
    """Bytes of all ranks (equal per-rank work) over the slowest rank's time."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# the sources each profiled kernel's counters depend on: its own files, plus the shared
# device headers and the launch path
_KERNEL_SOURCES = {
    "decode_i8": ["kvinj_decode_i8.cu", "kvinj_decode_common.cuh"],
    "decode": ["kvinj_decode_umma.cuh", "kvinj_decode_umma.cu", "kvinj_decode_umma_early.cu",
               "kvinj_decode_common.cuh"],
    "inject_i8": ["kvinj_inject_i8.cu"],
    "inject": ["kvinj_inject.cu"],
    "copy_blocks": ["kvinj_inject.cu"],
    "prefill": ["kvinj_prefill.cu"],
}
_COMMON_SOURCES = ["kvinj_device.cuh", "kvinj_umma.cuh", "kvinj_internal.h", "kvinj_api.cu"]


def _kernel_kind(tag: str) -> str:
    # the longest kind the tag starts with ("decode_i8_..." before "decode_...")
    kinds = [k for k in _KERNEL_SOURCES if tag.startswith(k + "_")]
    return max(kinds, key=len) if kinds else ""


def _traffic_from_profile(kernel_tag: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current source of that kernel (the summary records the hash)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.txt")
    if not os.path.exists(path):
        return None
    src = _source_hash(_kernel_kind(kernel_tag))
    want_hash, value = None, None
    for ln in open(path):
        if ln.startswith("source_sha256:"):
            want_hash = ln.split(":", 1)[1].strip()
        if ln.startswith("dram_bytes_per_launch:"):
            try:
                value = float(ln.split(":", 1)[1].strip())
            except ValueError:
                value = None
    return value if want_hash == src else None


def _code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to one space:
    what the compiler sees, so that editing a comment or the layout keeps a summary valid.
    String and character literals are kept as written (a "//" inside one is not a comment)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif c == "/" and text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def _source_hash(kind: str = "") -> str:
    """sha256 (16 hex digits) of the code of one kernel kind's sources, comments and
    layout aside (every file under csrc/ for an unknown kind)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_inject_gb300", "csrc")
    if kind in _KERNEL_SOURCES:
        names = sorted(set(_KERNEL_SOURCES[kind] + _COMMON_SOURCES))
    else:
        names = sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    h = hashlib.sha256()
    for name in names:
        h.update(name.encode() + b"\0")
        h.update(_code_only(open(os.path.join(csrc, name), encoding="utf-8").read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
class OracleSample:
    """Layer 0 of the workload on the host: the oracle's slot mapping, inject,
    append of the context and step tokens, and paged decode of every query
    head, for the first `requests` requests of the batch (all of them by
    default). Inputs are generated once (not timed)."""

    def __init__(self, wl, threads: int, window: int = 0, requests: int | None = None):
        import numpy as np

        import oracle
        self.np, self.oracle, self.wl, self.threads, self.window = np, oracle, wl, threads, window
        cfg = wl.cfg
        n_req = cfg.batch if requests is None else max(1, min(int(requests), cfg.batch))
        self.n_req = n_req
        L0 = 0
        Hkv, D, c = cfg.kv_heads, cfg.head_dim, cfg.chunk_len
        keep = wl.chunk_req < n_req
        ids = np.unique(wl.chunk_ids[keep])
        # pool rows of the drawn chunks for layer 0, as [n][1][2][c][Hkv][D]
        pool = np.zeros((ids.size, 1, 2, c, Hkv, D), np.uint16)
        t = np.tile(np.repeat(np.arange(c), Hkv), ids.size)
        h = np.tile(np.arange(Hkv), c * ids.size)
        cid = np.repeat(ids, c * Hkv)
        for kv in (0, 1):
            pool[:, 0, kv] = wl.pool_rows(cid, np.zeros(cid.size, int), np.full(cid.size, kv), t,
                                          h).reshape(ids.size, c, Hkv, D)
        self.pool = pool
        self.ids = np.searchsorted(ids, wl.chunk_ids[keep]).astype(np.int32)
        self.start_pos = wl.start_pos[keep]
        inj_seq, inj_pos = wl.injected_tokens()
        tok_keep = np.repeat(keep, c)
        self.inj_seq, self.inj_pos = inj_seq[tok_keep], inj_pos[tok_keep]
        a_seq, a_pos = wl.appended_tokens()
        a_keep = a_seq < n_req
        a_seq, a_pos = a_seq[a_keep], a_pos[a_keep]
        s_seq, s_pos = wl.step_tokens(0)
        s_seq, s_pos = s_seq[:n_req], s_pos[:n_req]
        self.app = [(a_seq, a_pos, wl.ctx_rows(L0, 0, a_seq, a_pos), wl.ctx_rows(L0, 1, a_seq, a_pos)),
                    (s_seq, s_pos, wl.ctx_rows(L0, 0, s_seq, s_pos), wl.ctx_rows(L0, 1, s_seq, s_pos))]
        self.q = wl.q_rows(0, L0)[:n_req]
        self.q_pos = s_pos
        self.ctx = s_pos + 1
        self.block_tables = wl.block_tables[:n_req]
        row = Hkv * D * cfg.elem_bytes
        n_inj_tok = self.inj_pos.size
        n_app = sum(x[0].size for x in self.app)
        ctx = self.ctx.astype(np.int64)
        lo = np.maximum(ctx - window, 0) if window > 0 else np.zeros_like(ctx)
        pages = -(-ctx // cfg.block_size) - lo // cfg.block_size
        self.bytes = (2 * 2 * row * n_inj_tok + 2 * 2 * row * n_app + int((ctx - lo).sum()) * 2 * row
                      + n_req * cfg.q_heads * D * 2 * 2 + int(pages.sum()) * 4)
        self.inj_tokens = n_inj_tok

    def run(self):
        np, orc, wl, cfg = self.np, self.oracle, self.wl, self.wl.cfg
        shape = (1, wl.num_blocks, cfg.kv_heads, cfg.block_size, cfg.head_dim)
        kc = np.zeros(shape, np.uint16)
        vc = np.zeros(shape, np.uint16)
        slots, _ = orc.slot_mapping(self.block_tables, self.inj_seq, self.inj_pos, cfg.block_size,
                                    wl.num_blocks)
        orc.inject(self.pool, self.ids, self.start_pos, slots, cfg.theta, cfg.dtype, kc, vc,
                   n_threads=self.threads)
        for seq, pos, kn, vn in self.app:
            sl, _ = orc.slot_mapping(self.block_tables, seq, pos, cfg.block_size, wl.num_blocks)
            orc.append(kc, vc, 0, kn, vn, pos, sl, cfg.theta, cfg.dtype)
        out, _ = orc.paged_decode(kc, vc, 0, self.q, self.q_pos, self.block_tables, self.ctx,
                                  cfg.theta, cfg.dtype, n_threads=self.threads,
                                  window=self.window)
        return out

    @property
    def description(self):
        cfg = self.wl.cfg
        who = (f"{cfg.batch}" if self.n_req == cfg.batch else
               f"the first {self.n_req} of {cfg.batch}")
        return (f"layer 0 of 1/{cfg.layers} layers of {cfg.name}, {who} requests: slot mapping, "
                f"inject of {self.inj_tokens} tokens, append of the context and step tokens, "
                f"paged decode of {self.n_req}x{cfg.q_heads} query heads")

    def time(self, min_seconds: float):
        """Repeat run() for at least min_seconds; (bytes per second, runs, seconds)."""
        runs, t0 = 0, time.perf_counter()
        while True:
            self.run()
            runs += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                return self.bytes * runs / dt, runs, dt


def oracle_threads() -> int:
    import oracle
    return (os.cpu_count() or 1) if oracle.has_openmp() else 1


def single_thread_requests(cfg) -> int:
    """Requests of the single-threaded oracle sample: about a quarter of the
    batch's context tokens (at least one request), so that one run stays near
    ten seconds on one host core."""
    import numpy as np

    import workload as W
    wl = W.make_workload(cfg)
    ctx = np.cumsum(wl.context_lens.astype(np.int64))
    return int(max(1, np.searchsorted(ctx, ctx[-1] // 4) + 1))


def cpu_baseline(wl, window: int, min_seconds: float = 10.0) -> dict:
    """The oracle on the host cores (all of them, repeated for about ten seconds)
    and on one core (a bounded sub-sample, run once)."""
    threads = oracle_threads()
    sample = OracleSample(wl, threads, window)
    gbs, runs, dt = sample.time(min_seconds)
    one = OracleSample(wl, 1, window, requests=single_thread_requests(wl.cfg))
    g1, r1, d1 = one.time(0.0)
    return {"value": gbs / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{sample.description}; {runs} runs in {dt:.1f} s",
            "seconds": dt,
            "single_thread": {"value": g1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{one.description}; {r1} run in {d1:.1f} s",
                              "seconds": d1}}


def run_reference(args):
    """--impl reference: the fp64 CPU oracle, as it stands, on a bounded sample."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import workload as W
    wl = W.make_workload(W.CONFIGS[args.config])
    threads = oracle_threads()
    sample = OracleSample(wl, threads, args.window)
    for _ in range(args.warmup):
        sample.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.run()
    dt = (time.perf_counter() - t0) / args.steps
    gbs = sample.bytes / dt / 1e9
    cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": sample.description}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {**workload_config(wl.cfg, args.window), "sample": "layer 0 per step (oracle on host cores)"},
        "cpu_baseline": cpu,
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "inject_tokens_per_s": sample.inj_tokens / dt,
    }))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
POOL_MARGIN = 8 << 30  # device bytes kept free beside the pool, cache and step inputs


class Setup:
    """One workload on the GPU: chunk pool, engine (cache, RoPE table, workspace),
    the context before the step, the step's inputs and its outputs."""

    def __init__(self, cfg, args, dev, rank):
        import torch

        import workload as W
        from workload import stage
        self.cfg = cfg
        self.wl = wl = W.make_workload(cfg, seed=replica_seed(cfg.seed, rank))
        torch.cuda.empty_cache()
        free, _ = torch.cuda.mem_get_info()
        compact = args.compact_pool or cfg.pool_bytes + wl.cache_bytes + POOL_MARGIN > free
        remap = None
        if compact:
            pool, remap = stage.compact_pool(wl, dev)
            self.pool_note = ("drawn chunks only" + ("" if args.compact_pool else
                              f" (the full {cfg.pool_bytes / 1e9:.1f} GB pool does not fit beside "
                              f"the cache in {free / 1e9:.1f} GB free)"))
        else:
            from workload import device as wgen
            pool = wgen.pool_tensor(wl, dev)
            self.pool_note = f"full, {cfg.pool_bytes / 1e9:.1f} GB resident"
        if args.pool_host:
            # the chunk pool in page-locked host memory: inject reads it over the host link
            host = torch.empty(pool.shape, dtype=pool.dtype, pin_memory=True)
            host.copy_(pool)
            del pool
            torch.cuda.synchronize()
            pool = host
            self.pool_note = "pinned host memory, read in place over the host link; " + self.pool_note
        self.pool = pool
        self.eng = eng = stage.make_engine(wl, dev, pool=pool)
        eng.decode_variant = args.variant
        eng.overlap_inject = args.overlap_inject
        eng.window = args.window
        stage.fill_context(eng, wl, dev)
        self.inp = stage.step_inputs(wl, dev)
        if remap is not None:
            self.inp.chunk_ids.copy_(torch.from_numpy(remap).to(dev))
        self.out = eng.alloc_outputs(cfg.steps)
        self.nbytes = stage.algorithmic_bytes(wl, args.window)
        self.slots = eng.slot_mapping(self.inp.block_tables, self.inp.map_seq, self.inp.map_pos)
        self.n_inj_tok = self.inp.chunk_ids.numel() * eng.chunk_len

    def inject_only(self):
        self.eng.inject(self.inp.chunk_ids, self.inp.start_pos, self.slots[:self.n_inj_tok])

    def decode_only(self):
        """The layer calls as the step makes them (append fused into decode by default;
        re-appending the same token writes the same bits)."""
        eng, inp, out, cfg = self.eng, self.inp, self.out, self.cfg
        for s in range(cfg.steps):
            for layer in range(cfg.layers):
                # as in the step: every call after the first follows one on another layer
                ready = (s > 0 or layer > 0) and cfg.layers > 1
                if eng.fused_append:
                    eng.append_decode(layer, inp.q[s, layer], inp.k_new[s, layer],
                                      inp.v_new[s, layer], inp.q_pos[s], inp.block_tables,
                                      inp.ctx_lens[s], out[s, layer], kv_ready=ready)
                else:
                    eng.decode(layer, inp.q[s, layer], inp.q_pos[s], inp.block_tables,
                               inp.ctx_lens[s], out[s, layer])

    def release(self):
        import torch
        for name in ("eng", "inp", "out", "pool", "slots"):
            setattr(self, name, None)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def graph_ms(fn, reps, use_graph=True):
    """Average ms of fn (captured in a CUDA graph) over `reps` replays, CUDA events on
    the launching stream, after two untimed replays."""
    import torch
    stream = torch.cuda.current_stream()
    g = None
    if use_graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
    run = g.replay if g is not None else fn
    for _ in range(2):
        run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def decode_inject_parts(st: Setup, reps: int, use_graph: bool, peak: float) -> dict:
    """Per-kernel times of one setup: inject (all layers, one launch) and decode (one
    call -- split-K pass + combine, with the fused append -- per layer and step)."""
    cfg, nbytes, eng = st.cfg, st.nbytes, st.eng
    inj_ms = graph_ms(st.inject_only, reps, use_graph)
    dec_ms = graph_ms(st.decode_only, reps, use_graph) / (cfg.layers * cfg.steps)
    dec_bytes = nbytes["decode"] + (nbytes["append"] if eng.fused_append else 0)
    per_launch = dec_bytes / (cfg.layers * cfg.steps)
    dec_gbs = per_launch / (dec_ms * 1e-3) / 1e9
    inj_gbs = nbytes["inject"] / (inj_ms * 1e-3) / 1e9
    return {
        "inject": {"tokens_per_s": st.wl.n_inj * cfg.chunk_len / (inj_ms * 1e-3), "gbs": inj_gbs,
                   "ms": inj_ms, "pct_of_8tbs": 100 * inj_gbs / NOMINAL_HBM_GBS,
                   "frac_of_measured": inj_gbs / peak, "bytes": nbytes["inject"]},
        "decode": {"gbs": dec_gbs, "ms_per_layer": dec_ms,
                   "pct_of_8tbs": 100 * dec_gbs / NOMINAL_HBM_GBS,
                   "frac_of_measured": dec_gbs / peak, "bytes_per_launch": per_launch},
    }


def time_steps(st: Setup, args, ws, dev, clocks=None):
    """Time exactly args.steps replays of the captured step (a barrier and a synchronize on
    both sides); the maximum over ranks. Returns (ms per step, the graph)."""
    import torch

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    eng, inp, out = st.eng, st.inp, st.out
    # warm-up (also checks the device status word)
    for _ in range(args.warmup):
        eng.step(inp, out)
    torch.cuda.synchronize()
    if eng.status.item() != 0:
        raise RuntimeError(f"device status {eng.status.item():#x} after warm-up")
    # The timed region replays one CUDA graph of the whole step (the decode loop is
    # launch-bound from Python otherwise); nothing but the step's own kernels is inside it.
    g = None if args.no_graph else eng.capture(inp, out)
    run = g.replay if g is not None else (lambda: eng.step(inp, out))
    for _ in range(args.warmup):
        run()
    barrier()
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.__enter__()
    t0.record(stream)
    for _ in range(args.steps):
        run()
    t1.record(stream)
    barrier()
    if clocks is not None:
        clocks.__exit__(None, None, None)
    return max_over_ranks(t0.elapsed_time(t1), dev) / args.steps, g


def measure_int8(st: Setup, args, ws, dev, reps, use_graph, peak, ms16) -> dict:
    """The same step and per-kernel timings with the KV cache stored as int8 codes and row
    scales ("Latency Optimization > KV Cache Management", KV cache quantization): an
    engine with the int8 cache over the same resident pool, the same step inputs; bytes
    are the int8 cache's (a row: D code bytes + a 4-byte scale)."""
    import copy

    import torch

    from workload import stage
    eng = stage.make_engine(st.wl, dev, pool=st.pool, kv="int8")
    eng.decode_variant = args.variant
    stage.fill_context(eng, st.wl, dev)
    s8 = copy.copy(st)
    s8.eng = eng
    s8.out = eng.alloc_outputs(st.cfg.steps)
    s8.nbytes = stage.algorithmic_bytes(st.wl, 0, kv="int8")
    ms8, g8 = time_steps(s8, args, ws, dev)
    parts = decode_inject_parts(s8, reps, use_graph, peak)
    if eng.status.item() != 0:
        raise RuntimeError(f"int8 cache: device status {eng.status.item():#x}")
    value = whole_job_gbs(ws, s8.nbytes["total"], ms8)
    out = {"value": value, "unit": "GB/s", "ms_per_step": ms8,
           "step_time_vs_16bit": ms8 / ms16, "pct_of_8tbs": 100 * value / NOMINAL_HBM_GBS,
           "step_bytes": s8.nbytes, **parts,
           "note": "the step's algorithmic bytes with the cache as int8 codes + one fp32 scale "
                   "per row; decode turns codes into fp16 tensor-core operands on the chip"}
    g8 = s8 = eng = None
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def host_link_copy_gbs(st: Setup, max_bytes: int = 2 << 30) -> dict:
    """Copy rate of the host link for the pool records the inject reads: one copy per
    drawn chunk record from the page-locked pool into device memory (a ring of device
    buffers), CUDA events around the copies, at most max_bytes."""
    import numpy as np
    import torch
    pool = st.pool
    ids = np.unique(st.inp.chunk_ids.cpu().numpy())
    rec = pool[0].numel() * pool.element_size()
    n = int(max(1, min(ids.size, max_bytes // rec)))
    ring = [torch.empty_like(pool[0], device="cuda") for _ in range(min(8, n))]
    for i in range(min(4, n)):  # warm
        ring[i % len(ring)].copy_(pool[int(ids[i])], non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n):
        ring[i % len(ring)].copy_(pool[int(ids[i])], non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return {"gbs": n * rec / (ms * 1e-3) / 1e9, "records": n, "record_bytes": rec,
            "method": "one cudaMemcpyAsync (torch copy_) per drawn chunk record, page-locked "
                      "host -> device, CUDA events around the copies"}


def run_gpu(args):
    import numpy as np
    import torch

    import workload as W

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    import __graft_entry__
    __graft_entry__.build()

    cfg = W.CONFIGS[args.config]
    if args.layers:
        cfg = cfg.scaled(layers=args.layers)  # batch structure does not depend on L
    peak, peak_kind = _peaks()
    use_graph = not args.no_graph
    reps = max(3, args.steps)
    st = Setup(cfg, args, dev, rank)
    wl, eng, inp, out, nbytes = st.wl, st.eng, st.inp, st.out, st.nbytes
    stream = torch.cuda.current_stream()

    clk = ClockSampler(local)
    ms_step, g_step = time_steps(st, args, ws, dev, clocks=clk)
    value = whole_job_gbs(ws, nbytes["total"], ms_step)
    parts = decode_inject_parts(st, reps, use_graph, peak)
    parts["decode"]["tokens_per_s"] = ws * cfg.batch * cfg.steps / (ms_step * 1e-3)

    # copy-on-write block copies: one call over distinct blocks in use, each copied onto
    # itself (the cache keeps its contents; every record is read and written in full)
    n_copy = min(1024, cfg.batch * max(1, int(wl.context_lens.min()) // cfg.block_size))
    copy_ids = inp.block_tables[:, : max(1, n_copy // cfg.batch)].reshape(-1)[:n_copy].contiguous()
    n_copy = copy_ids.numel()
    rec_bytes = cfg.kv_heads * cfg.block_size * cfg.head_dim * 2
    copy_bytes = 2 * 2 * n_copy * cfg.layers * rec_bytes  # K and V, read and write
    copy_avg = graph_ms(lambda: eng.copy_blocks(copy_ids, copy_ids), reps, use_graph)
    copy_gbs = copy_bytes / (copy_avg * 1e-3) / 1e9
    # paged prefill: the last nq tokens of every context taken as layer 0's query tokens (their
    # K/V are in the cache); each token is a decode row over its own causal context
    ctx_h = wl.context_lens.astype(np.int64) + 1
    nq = int(min(16, ctx_h.min()))
    pos_h = (ctx_h[:, None] - nq + np.arange(nq)[None, :]).reshape(-1)
    pf_seq = torch.from_numpy(np.repeat(np.arange(cfg.batch), nq).astype(np.int32)).to(dev)
    pf_pos = torch.from_numpy(pos_h.astype(np.int32)).to(dev)
    pf_q = inp.q[0, 0].repeat_interleave(nq, dim=0).contiguous()
    pf_out = torch.empty_like(pf_q)
    eng.prefill(0, pf_q, pf_seq, pf_pos, inp.block_tables, pf_out)  # workspace allocated here
    pf_avg = graph_ms(lambda: eng.prefill(0, pf_q, pf_seq, pf_pos, inp.block_tables, pf_out),
                      reps, use_graph)
    kv_row = cfg.kv_heads * cfg.head_dim * cfg.elem_bytes
    # the tensor-core prefill reads, per tile of up to 128 / G consecutive tokens of one
    # request, K and V of the request's tokens 0 .. the tile's last position once
    T = 128 // (cfg.q_heads // cfg.kv_heads)
    tile_last = [int(p[min(t + T, nq) - 1]) for p in pos_h.reshape(cfg.batch, nq)
                 for t in range(0, nq, T)]
    pf_read = sum(m + 1 for m in tile_last) * 2 * kv_row
    pf_qo = 2 * pos_h.size * cfg.q_heads * cfg.head_dim * cfg.elem_bytes  # q in, out
    pf_unique = int(ctx_h.sum()) * 2 * kv_row
    # slot mapping, inject (one launch, or one per layer when overlapped), then per step and
    # layer the append + decode launches
    inject_launches = cfg.layers if eng.overlap_inject else 1
    launches_per_step = 1 + inject_launches + eng.launches_per_layer() * cfg.layers * cfg.steps
    link = host_link_copy_gbs(st) if args.pool_host else None
    int8 = None
    if not args.no_int8 and cfg.head_dim == 128 and cfg.kv_heads % 8 == 0 and not args.window:
        int8 = measure_int8(st, args, ws, dev, reps, use_graph, peak, ms_step)

    # end to end through host buffers (pinned), same metric
    e2e = None
    if not args.no_e2e:
        from workload import stage
        host = stage.pinned_copy(inp)
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        for _ in range(max(1, args.warmup)):
            eng.step_from_host(host, inp, out, host_out, g_step)
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            eng.step_from_host(host, inp, out, host_out, g_step)
        e1.record(stream)
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
        e2e = {"value": whole_job_gbs(ws, nbytes["total"], e_ms), "unit": "GB/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": host.nbytes,
               "d2h_bytes_per_step": host_out.numel() * host_out.element_size()}
        del host, host_out
    if eng.status.item() != 0:
        raise RuntimeError(f"device status {eng.status.item():#x}")
    pool_note = st.pool_note
    # drop every reference to this setup's buffers (the pool alone can be 170+ GB) before
    # the next workload allocates its own
    g_step = eng = inp = out = copy_ids = pf_q = pf_out = pf_seq = pf_pos = None
    st.release()

    # the other workloads the target names, measured in the same run (each step timed the
    # same way; their per-kernel parts as above)
    others = {}
    if not args.no_others and not args.layers:
        for name in OTHER_WORKLOADS:
            if name == cfg.name:
                continue
            o = Setup(W.CONFIGS[name], args, dev, rank)
            o_ms, _ = time_steps(o, args, ws, dev)
            o_val = whole_job_gbs(ws, o.nbytes["total"], o_ms)
            p = decode_inject_parts(o, reps, use_graph, peak)
            if o.eng.status.item() != 0:
                raise RuntimeError(f"{name}: device status {o.eng.status.item():#x}")
            others[name] = {"value": o_val, "unit": "GB/s", "ms_per_step": o_ms,
                            "pct_of_8tbs": 100 * o_val / NOMINAL_HBM_GBS,
                            "frac_of_measured": o_val / peak, "steps": args.steps,
                            "pool": o.pool_note, "step_bytes": o.nbytes, **p}
            o.release()
            del o, p

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.window)

    if rank != 0:
        return
    parts.update({
        "prefill": {"query_tokens": int(pos_h.size), "per_request": nq, "layers": 1,
                    "ms": pf_avg, "tokens_per_s": pos_h.size / (pf_avg * 1e-3),
                    "kv_bytes_read": pf_read, "q_out_bytes": pf_qo,
                    "gbs": (pf_read + pf_qo) / (pf_avg * 1e-3) / 1e9,
                    "frac_of_measured": (pf_read + pf_qo) / (pf_avg * 1e-3) / 1e9 / peak,
                    "unique_kv_bytes": pf_unique,
                    "traffic": _traffic_from_profile(f"prefill_{cfg.name}"),
                    "note": "tensor-core tiles of up to 128/G query tokens of one request: "
                            "K/V of the request's tokens up to the tile's last position read "
                            "once per tile and kv head; unique bytes = each context once"},
        "copy_blocks": {"blocks": n_copy, "layers": cfg.layers, "bytes": copy_bytes,
                        "ms": copy_avg, "gbs": copy_gbs,
                        "note": "each block copied onto itself: full reads and writes, "
                                "cache unchanged"},
        "step_bytes": nbytes,
        "step_pct_of_8tbs": 100 * value / NOMINAL_HBM_GBS,
        "other_workloads": others,
        "int8_cache": int8,
    })
    inj = parts["inject"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": W.DTYPE_NAMES[cfg.dtype],
        "data": "synthetic",
        "config": {**workload_config(cfg, args.window), "parallelism": f"replicas x{ws}",
                   "l2": (f"inputs larger than L2: {nbytes['total'] / 1e9:.2f} GB touched per "
                          f"step; no flush"),
                   "decode_variant": args.variant,
                   "inject_schedule": ("per layer, low-priority stream beside the decode"
                                       if args.overlap_inject else "all layers, then decode"),
                   "launch": "cuda graph per step" if use_graph else "eager",
                   "pool": pool_note},
        "parts": parts,
        "roofline": {"kernel": "decode", "bound": "hbm", "achieved": parts["decode"]["gbs"],
                     "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                     "frac": parts["decode"]["gbs"] / peak,
                     "traffic": _traffic_from_profile(f"decode_{cfg.name}")},
        "roofline_inject": ({"kernel": "inject", "bound": "host link (pool reads)",
                             "achieved": inj["gbs"] / 2, "peak": link["gbs"],
                             "peak_source": "measured in this run: " + link["method"],
                             "unit": "GB/s", "frac": inj["gbs"] / 2 / link["gbs"],
                             "traffic": None,
                             "note": "achieved = pool bytes read from host memory per second"}
                            if args.pool_host else
                            {"kernel": "inject", "bound": "hbm", "achieved": inj["gbs"],
                             "peak": peak, "unit": "GB/s", "frac": inj["gbs"] / peak,
                             "traffic": _traffic_from_profile(f"inject_{cfg.name}")}),
        "roofline_decode_int8": ({"kernel": "decode_i8", "bound": "hbm",
                                  "achieved": int8["decode"]["gbs"], "peak": peak, "unit": "GB/s",
                                  "frac": int8["decode"]["gbs"] / peak,
                                  "traffic": _traffic_from_profile(f"decode_i8_{cfg.name}")}
                                 if int8 else None),
        "roofline_copy_blocks": {"kernel": "copy_blocks", "bound": "hbm", "achieved": copy_gbs,
                                 "peak": peak, "unit": "GB/s", "frac": copy_gbs / peak,
                                 "traffic": _traffic_from_profile(f"copy_blocks_{cfg.name}")},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--variant", type=int, default=0, help="decode kernel: 0 auto, 1 FMA, 2 mma.sync, 3 tcgen05")
    ap.add_argument("--overlap-inject", dest="overlap_inject", action="store_true",
                    help="inject layer by layer on a low-priority stream beside the decode")
    ap.add_argument("--serial", dest="overlap_inject", action="store_false",
                    help="inject all layers, then decode (one stream)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly from Python")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling cases only)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window decode over the last W tokens (0: whole context)")
    ap.add_argument("--pool-host", action="store_true",
                    help="keep the chunk pool in pinned host memory (inject reads it in place)")
    ap.add_argument("--compact-pool", action="store_true",
                    help="keep only the drawn chunks resident (small profiling cases only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-int8", action="store_true",
                    help="skip the int8-cache measurement of the chosen workload")
    ap.add_argument("--no-others", action="store_true",
                    help="measure the chosen workload only (not the other target workloads)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
