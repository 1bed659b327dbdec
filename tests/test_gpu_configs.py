"""The five workloads at full size, in the launch configuration the benchmark
times, checked against the oracle on sampled outputs.

For each workload: the chunk pool and the preceding context are put on the
GPU, one full step runs (slot mapping, inject over all layers, then per
decode step and layer: append + paged decode), and then
  - every slot the step mapped is compared bit for bit with the oracle's,
  - sampled cache rows (injected, appended and step tokens) match the
    oracle's rotated keys within one ulp and its values bit for bit,
  - sampled decode outputs match the oracle within atol 2e-3 + rtol 1e-2.
Also: the device generator reproduces the host generator's bits."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from tests.gpu_helpers import (assert_decode_close, bits, expected_cache_rows, expected_decode,
                               ulp_distance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()


def test_device_generator_matches_host():
    import workload.device as gen
    wl = W.make_workload(W.CONFIGS["llama3_8b_b32"])
    pool = gen.pool_tensor(wl, "cuda", n_chunks=3)
    flat = bits(pool).reshape(-1)
    idx = np.random.default_rng(0).integers(0, flat.size, 20000)
    idx = np.concatenate([idx, np.arange(17), [flat.size - 1]])
    assert np.array_equal(flat[idx], W.normal_bits(wl.keys["pool"], idx.astype(np.uint64), W.BF16))
    seq = np.array([0, 3, 31], np.int32)
    pos = np.array([5, 700, 12], np.int32)
    rows, keep = gen.ctx_rows(wl, 7, 1, seq, pos)
    assert np.array_equal(bits(rows), wl.ctx_rows(7, 1, seq, pos))
    q = gen.q_rows(wl, 0, 3)
    assert np.array_equal(bits(q), wl.q_rows(0, 3))
    wl16 = W.make_workload(W.CONFIGS["mha70b_b4_4k_fp16"])
    p16 = gen.pool_tensor(wl16, "cuda", n_chunks=1)
    f16 = bits(p16).reshape(-1)
    assert np.array_equal(f16[:5000], W.normal_bits(wl16.keys["pool"], np.arange(5000), W.FP16))


def _pool_for(wl, device="cuda"):
    """The full pool when it fits in free memory, else only the drawn chunks
    (same values, remapped ids): the kernels and the bytes they move are the same."""
    import workload.device as gen
    from workload import stage
    cfg = wl.cfg
    free, _ = torch.cuda.mem_get_info()
    need = cfg.pool_bytes + wl.cache_bytes + (8 << 30)
    if need < free:
        return gen.pool_tensor(wl, device), None
    return stage.compact_pool(wl, device)


@pytest.mark.parametrize("name", W.CONFIG_ORDER)
def test_config_full_size(name):
    from workload import stage
    cfg = W.CONFIGS[name]
    wl = W.make_workload(cfg)
    torch.cuda.empty_cache()
    pool, remap = _pool_for(wl)
    eng = stage.make_engine(wl, "cuda", pool=pool)
    stage.fill_context(eng, wl)
    inp = stage.step_inputs(wl)
    if remap is not None:
        inp.chunk_ids = torch.from_numpy(remap).cuda()
    out = eng.alloc_outputs(cfg.steps)
    eng.step(inp, out)
    torch.cuda.synchronize()
    assert eng.status.item() == 0
    rng = np.random.default_rng(42)

    # slot mapping of every token the step touched: bit-exact
    slots = eng.slot_mapping(inp.block_tables, inp.map_seq, inp.map_pos)
    want, st = oracle.slot_mapping(wl.block_tables, inp.map_seq.cpu().numpy(),
                                   inp.map_pos.cpu().numpy(), cfg.block_size, wl.num_blocks)
    assert st == 0
    assert np.array_equal(slots.cpu().numpy(), want)

    # sampled cache rows: injected, appended and step tokens of every kind
    B, D = cfg.block_size, cfg.head_dim
    n_rows = 256 if cfg.layers > 1 else 64
    worst = 0
    for _ in range(n_rows):
        r = int(rng.integers(cfg.batch))
        n = int(wl.context_lens[r]) + cfg.steps
        p = int(rng.integers(n))
        layer, h = int(rng.integers(cfg.layers)), int(rng.integers(cfg.kv_heads))
        k_want, v_want = expected_cache_rows(wl, layer, r, [p], h)
        blk = int(wl.block_tables[r, p // B])
        k_got = bits(eng.k_cache[layer, blk, h, p % B])
        v_got = bits(eng.v_cache[layer, blk, h, p % B])
        assert np.array_equal(v_got, v_want[0]), (r, p, layer, h)
        d = ulp_distance(k_got, k_want[0])
        worst = max(worst, int(d.max()))
    assert worst <= 1

    # sampled decode outputs: the longest request, the shortest, and random ones
    order = np.argsort(wl.context_lens)
    reqs = [int(order[-1]), int(order[0])] + [int(x) for x in rng.integers(cfg.batch, size=6)]
    for i, r in enumerate(reqs):
        s = cfg.steps - 1 if i % 2 == 0 else int(rng.integers(cfg.steps))
        layer = int(rng.integers(cfg.layers))
        qh = int(rng.integers(cfg.q_heads))
        want = expected_decode(wl, s, layer, r, qh)
        got = out[s, layer, r, qh].float().cpu().numpy().astype(np.float64)
        assert_decode_close(got, want, f"{name} step {s} layer {layer} req {r} head {qh}")
    del eng, pool, inp, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["llama3_8b_b32", "llama3_70b_b8_8k"])
def test_overlapped_inject_schedule_matches_serial_bitwise(name):
    # inject layer by layer on a low-priority stream beside the decode: the same cache and
    # outputs, bit for bit, as inject-then-decode on one stream (graph-captured, as timed)
    from workload import stage
    cfg = W.CONFIGS[name].scaled(layers=4, steps=min(W.CONFIGS[name].steps, 2))
    wl = W.make_workload(cfg)
    pool, remap = stage.compact_pool(wl)
    results = []
    for overlap in (False, True):
        eng = stage.make_engine(wl, pool=pool)
        eng.overlap_inject = overlap
        stage.fill_context(eng, wl)
        inp = stage.step_inputs(wl)
        inp.chunk_ids.copy_(torch.from_numpy(remap).cuda())
        out = eng.alloc_outputs(cfg.steps)
        g = eng.capture(inp, out)
        g.replay()
        torch.cuda.synchronize()
        assert eng.status.item() == 0
        results.append((bits(out), bits(eng.k_cache), bits(eng.v_cache)))
        del eng, g
    for a, b in zip(*results):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("name,ctas,window", [("llama3_8b_b32", 0, 0), ("llama3_8b_b32", 37, 0),
                                              ("llama3_70b_b8_8k", 0, 0),
                                              ("mixed_b64_loguniform", 0, 0),
                                              ("llama3_8b_b32", 0, 512)])
def test_early_page_reads_match_waiting_calls_bitwise(name, ctas, window):
    # decode calls that stream their first pages before the kernel ahead of them ends
    # (every call of a step after the first) give the same outputs and cache, bit for
    # bit, as calls that wait before every read; graph-captured, as timed
    from workload import stage
    base = W.CONFIGS[name]
    cfg = base.scaled(layers=4, steps=min(base.steps, 3))
    wl = W.make_workload(cfg)
    pool, remap = stage.compact_pool(wl)
    results = []
    for early in (False, True):
        eng = stage.make_engine(wl, pool=pool)
        eng.early_kv = early
        eng.decode_ctas = ctas
        eng.window = window
        stage.fill_context(eng, wl)
        inp = stage.step_inputs(wl)
        inp.chunk_ids.copy_(torch.from_numpy(remap).cuda())
        out = eng.alloc_outputs(cfg.steps)
        g = eng.capture(inp, out)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert eng.status.item() == 0
        results.append((bits(out), bits(eng.k_cache), bits(eng.v_cache)))
        del eng, g
    for a, b in zip(*results):
        assert np.array_equal(a, b)
