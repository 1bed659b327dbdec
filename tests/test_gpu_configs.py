"""The five workloads at full size, in the launch configuration the benchmark
times, checked against the oracle.

For each workload: the chunk pool and the preceding context are put on the
GPU, one full step runs (slot mapping, inject over all layers, then per
decode step and layer: append + paged decode), and then
  - every slot the step mapped is compared bit for bit with the oracle's,
  - every cache row of the last layer (injected, appended and step tokens)
    matches the oracle's rotated keys within one ulp and its values bit for
    bit,
  - every output of the first and the last layer at the first and the last
    decode step (every request, every query head) matches the oracle within
    atol 2e-3 + rtol 1e-2.
The int8 cache runs the same step on two workloads and is checked the same
way against the oracle's quantization and int8 decode. Also: the device
generator reproduces the host generator's bits."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from tests.gpu_helpers import (assert_decode_close, bits, expected_request_rows, gpu_request_rows,
                               request_cache, ulp_distance)

pytestmark = pytest.mark.gpu


def oracle_threads():
    import os
    return (os.cpu_count() or 1) if oracle.has_openmp() else 1


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

    # every cache row of the last layer (K within one ulp of the oracle's rotation, V bit
    # for bit), and every output of the first and last layer at the first and last decode
    # step, each against the oracle's attention over the request's rows
    L = cfg.layers
    layers = sorted({0, L - 1})
    steps = sorted({0, cfg.steps - 1})
    gk = bits(eng.k_cache[L - 1]).reshape((1,) + tuple(eng.k_cache.shape[1:]))
    gv = bits(eng.v_cache[L - 1]).reshape((1,) + tuple(eng.v_cache.shape[1:]))
    got_all = {(s, l): out[s, l].float().cpu().numpy().astype(np.float64)
               for s in steps for l in layers}
    worst = 0
    for layer in layers:
        for r in range(cfg.batch):
            n_max = int(wl.context_lens[r]) + cfg.steps
            k_want, v_want = expected_request_rows(wl, layer, r, n_max)
            if layer == L - 1:
                k_got, v_got = gpu_request_rows(gk, gv, 0, wl.block_tables[r], n_max)
                assert np.array_equal(v_got, v_want), (name, r)
                worst = max(worst, int(ulp_distance(k_got, k_want).max()))
            for s in steps:
                n = int(wl.context_lens[r]) + s + 1
                kc, vc, bt1 = request_cache(k_want[:, :n], v_want[:, :n])
                q = wl.q_rows(s, layer)[r:r + 1]
                want, st = oracle.paged_decode(kc, vc, 0, q, np.array([n - 1], np.int32), bt1,
                                               np.array([n], np.int32), cfg.theta, cfg.dtype,
                                               n_threads=oracle_threads())
                assert st == 0
                assert_decode_close(got_all[(s, layer)][r], want[0],
                                    f"{name} step {s} layer {layer} req {r}")
    assert worst <= 1
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


@pytest.mark.parametrize("name,layers,steps", [("llama3_8b_b32", 4, 1), ("llama3_70b_b8_8k", 2, 3)])
def test_int8_cache_step_matches_oracle(name, layers, steps):
    # the whole step with the int8 cache (inject, then per step and layer the fused append +
    # decode), graph-captured as timed: every cache row of the last layer holds the oracle's
    # codes and scales, and every output of the first and last layer at the first and last
    # step matches the oracle's int8 decode over those codes
    from workload import stage
    cfg = W.CONFIGS[name].scaled(layers=layers, steps=steps)
    wl = W.make_workload(cfg)
    pool, remap = stage.compact_pool(wl)
    eng = stage.make_engine(wl, pool=pool, kv="int8")
    stage.fill_context(eng, wl)
    inp = stage.step_inputs(wl)
    inp.chunk_ids.copy_(torch.from_numpy(remap).cuda())
    out = eng.alloc_outputs(cfg.steps)
    g = eng.capture(inp, out)
    g.replay()
    torch.cuda.synchronize()
    assert eng.status.item() == 0
    L = cfg.layers
    c = eng.cache
    gkq = c.k[L - 1:].cpu().numpy()
    gvq = c.v[L - 1:].cpu().numpy()
    gks = c.k_scale[L - 1:].cpu().numpy()[..., None]
    gvs = c.v_scale[L - 1:].cpu().numpy()[..., None]
    for layer in sorted({0, L - 1}):
        for r in range(cfg.batch):
            n_max = int(wl.context_lens[r]) + cfg.steps
            k16, v16 = expected_request_rows(wl, layer, r, n_max)
            kq, ks = oracle.quantize_rows_i8(k16, cfg.dtype)
            vq, vs = oracle.quantize_rows_i8(v16, cfg.dtype)
            if layer == L - 1:
                a, b = gpu_request_rows(gkq, gvq, 0, wl.block_tables[r], n_max)
                assert np.array_equal(a, kq) and np.array_equal(b, vq), (name, r)
                a, b = gpu_request_rows(gks, gvs, 0, wl.block_tables[r], n_max)
                assert np.array_equal(a[..., 0], ks) and np.array_equal(b[..., 0], vs), (name, r)
            for s in sorted({0, cfg.steps - 1}):
                n = int(wl.context_lens[r]) + s + 1
                kc, vc, bt1 = request_cache(kq[:, :n], vq[:, :n])
                ksc, vsc, _ = request_cache(ks[:, :n, None], vs[:, :n, None])
                want, st = oracle.paged_decode_i8(kc, ksc[..., 0], vc, vsc[..., 0], 0,
                                                  wl.q_rows(s, layer)[r:r + 1],
                                                  np.array([n - 1], np.int32), bt1,
                                                  np.array([n], np.int32), cfg.theta, cfg.dtype)
                assert st == 0
                got = out[s, layer, r].float().cpu().numpy().astype(np.float64)
                assert_decode_close(got, want[0], f"int8 {name} step {s} layer {layer} req {r}")
