"""The seeded workload generator (host side): known answers of the hash, the
value distribution, and the integer structure of every workload."""
import numpy as np
import pytest

import workload as W


def test_splitmix64_known_answers():
    # SplitMix64 from state 0: the first outputs of the published generator
    got = W.hash64(0, np.arange(3, dtype=np.uint64))
    assert int(got[0]) == 0xE220A8397B1DCDAF
    assert int(got[1]) == 0x6E789E6AA1B965F4


def test_normal_values_moments_and_determinism():
    key = W.stream_key(7, W.STREAM_POOL)
    x = W.normal_f32(key, np.arange(2_000_000, dtype=np.uint64)).astype(np.float64)
    assert abs(x.mean()) < 3e-3
    assert abs(x.var() - 1.0) < 5e-3
    assert np.max(np.abs(x)) <= 131070 * float(W.NORMAL_SCALE) + 1e-6
    y = W.normal_f32(key, np.arange(1000, 2000, dtype=np.uint64))
    assert np.array_equal(y, x[1000:2000].astype(np.float32))
    assert W.stream_key(7, W.STREAM_POOL) != W.stream_key(7, W.STREAM_CTX)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -1.00390625, 3.0e-39], np.float32)
    bits = W.f32_to_bits(x, W.BF16)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: goes to the even (1.0)
    assert list(bits[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xBF80]


@pytest.mark.parametrize("name", W.CONFIG_ORDER)
def test_workload_structure(name):
    cfg = W.CONFIGS[name]
    wl = W.make_workload(cfg)
    c = cfg.chunk_len
    assert wl.block_tables.shape[0] == cfg.batch
    used = []
    for r in range(cfg.batch):
        C = int(wl.context_lens[r])
        js = np.nonzero(wl.chunk_req == r)[0]
        assert js.size == min(cfg.chunks_per_req, C // c)
        s = np.sort(wl.start_pos[js])
        assert np.all(s >= 0) and np.all(s + c <= C)
        assert np.all(np.diff(s) >= c), "chunks overlap"
        ids = wl.chunk_ids[js]
        assert len(set(ids.tolist())) == ids.size
        assert np.all((ids >= 0) & (ids < cfg.pool_chunks))
        nb = -(-(C + cfg.steps) // cfg.block_size)
        row = wl.block_tables[r, :nb]
        assert np.all((row >= 0) & (row < wl.num_blocks))
        used.extend(row.tolist())
    assert len(set(used)) == len(used), "physical blocks shared between requests"
    if cfg.draw_once:
        assert len(set(wl.chunk_ids.tolist())) == wl.chunk_ids.size
    if cfg.occupancy < 1.0:
        assert abs(len(used) / wl.num_blocks - cfg.occupancy) < 0.01
    # the appended and injected tokens partition each context
    a_seq, a_pos = wl.appended_tokens()
    i_seq, i_pos = wl.injected_tokens()
    for r in range(cfg.batch):
        allp = np.sort(np.concatenate([a_pos[a_seq == r], i_pos[i_seq == r]]))
        assert np.array_equal(allp, np.arange(wl.context_lens[r]))


def test_tiny_workload_fixed_shape():
    wl = W.make_workload(W.CONFIGS["tiny_1layer"])
    assert list(wl.start_pos) == [16, 40]
    assert sorted(wl.block_tables[0].tolist()) == list(range(8))
    assert int(wl.context_lens[0]) == 64 and wl.n_inj == 2


def test_workload_sizes_match_the_shapes():
    # pool record = 2 L c Hkv D b (InferScale section 3.4)
    cfg = W.CONFIGS["llama3_8b_b32"]
    assert cfg.chunk_elems * 2 == 2 * 32 * 64 * 8 * 128 * 2
    assert abs(cfg.pool_bytes / 1e9 - 34.36) < 0.01
    assert abs(W.CONFIGS["llama3_70b_b8_8k"].pool_bytes / 1e9 - 171.80) < 0.01
    assert abs(W.CONFIGS["mixed_b64_loguniform"].pool_bytes / 1e9 - 209.72) < 0.01


def test_algorithmic_bytes_under_a_window():
    # under a sliding window of W tokens a decode call reads the K and V of the last
    # min(ctx, W) tokens of each context and the table entries of the pages holding them;
    # a window longer than every context counts the same bytes as none
    from workload import stage
    wl = W.make_workload(W.CONFIGS["llama3_70b_b8_8k"])
    cfg = wl.cfg
    full = stage.algorithmic_bytes(wl)
    assert stage.algorithmic_bytes(wl, 10 ** 6) == full
    win = stage.algorithmic_bytes(wl, 4096)
    row = cfg.kv_heads * cfg.head_dim * 2
    small = cfg.batch * cfg.q_heads * cfg.head_dim * 2 * 2
    want = 0
    for s in range(cfg.steps):
        c = 8192 + s + 1  # fixed contexts, plus the tokens appended by steps 0..s
        pages = -(-c // 16) - (c - 4096) // 16
        want += cfg.layers * (cfg.batch * (4096 * 2 * row + pages * 4) + small)
    assert win["decode"] == want
    assert win["inject"] == full["inject"] and win["append"] == full["append"]
    assert win["total"] == win["inject"] + win["append"] + win["decode"]
