"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: printed
worked examples (tests/golden), closed forms, invariants the pages state, or a
library routine a special case reduces to. Runs on CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

BF16, FP16 = oracle.BF16, oracle.FP16


# ---------------------------------------------------------------------------
# 16-bit formats
# ---------------------------------------------------------------------------
def _special_doubles(rng, n):
    x = rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, n))
    return x


def test_fp16_encode_matches_numpy_rne():
    # numpy's float64 -> float16 conversion rounds once, ties to even
    rng = np.random.default_rng(1)
    x = np.concatenate([
        _special_doubles(rng, 200000),
        rng.standard_normal(100000),
        # exact ties between neighbouring fp16 values, normal and subnormal
        (np.arange(-3000, 3000) + 0.5) * 2.0 ** -10,
        (np.arange(-3000, 3000) + 0.5) * 2.0 ** -24,
        np.array([65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0, 2.0 ** -25, 2.0 ** -26]),
    ])
    ours = oracle.encode(x, FP16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_encode_matches_torch_on_float32_inputs():
    # for fp32-representable inputs torch's fp32 -> bf16 is a single RNE rounding
    rng = np.random.default_rng(2)
    x32 = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(50000) * 1e-38).astype(np.float32),  # subnormal range
        np.array([3.3895314e38, 3.4e38, -3.4e38, 1e-45, 0.0], np.float32),
    ])
    # exact ties: low 16 bits = 0x8000
    ties = (rng.integers(0, 2 ** 31, 20000, dtype=np.uint32) & 0xFFFF0000) | 0x8000
    x32 = np.concatenate([x32, ties.view(np.float32)])
    x32 = x32[np.isfinite(x32)]
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = oracle.encode(x32.astype(np.float64), BF16)
    assert np.array_equal(ours, ref)


def test_bf16_encode_is_nearest_even_on_doubles():
    # definition: the result is the nearer of the two bf16 neighbours of x,
    # the even one on a tie
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000), _special_doubles(rng, 100000)])
    b = oracle.encode(x, BF16)
    r = oracle.decode(b, BF16)
    mag = b & 0x7FFF
    other = np.where(np.abs(r) <= np.abs(x), mag + 1, mag - 1).astype(np.uint16) | (b & 0x8000)
    ro = oracle.decode(other, BF16)
    lo, hi = np.minimum(r, ro), np.maximum(r, ro)
    assert np.all((lo <= x) & (x <= hi)), "result does not bracket x with its neighbour"
    d_r, d_o = np.abs(x - r), np.abs(x - ro)
    assert np.all(d_r <= d_o)
    tie = d_r == d_o
    assert np.all((b[tie] & 1) == 0)


def test_decode_matches_library_views():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin16 = np.isfinite(bits.view(np.float16))
    assert np.array_equal(oracle.decode(bits, FP16)[fin16],
                          bits.view(np.float16)[fin16].astype(np.float64))
    as32 = (bits.astype(np.uint32) << 16).view(np.float32)
    fin = np.isfinite(as32)
    assert np.array_equal(oracle.decode(bits, BF16)[fin], as32[fin].astype(np.float64))


# ---------------------------------------------------------------------------
# RoPE: InferScale page, section 2.3 (R_p block-diagonal rotation,
# R_a^T R_b = R_{b-a}); pairing rotate-half is the reading of apply_rotary_pos_emb
# ---------------------------------------------------------------------------
def test_rope_small_closed_form():
    # D = 4, theta = 1e4: inverse frequencies 1 and 1e4^(-1/2) = 0.01; the pairs
    # are (0, 2) and (1, 3), each a plane rotation by position * frequency
    th = 1e4
    y = oracle.rope([1.0, 0.0, 0.0, 0.0], 1.0, th)
    np.testing.assert_allclose(y, [math.cos(1.0), 0.0, math.sin(1.0), 0.0], rtol=0, atol=1e-15)
    y = oracle.rope([0.0, 1.0, 0.0, 0.0], 1.0, th)
    np.testing.assert_allclose(y, [0.0, math.cos(0.01), 0.0, math.sin(0.01)], rtol=0, atol=1e-15)
    y = oracle.rope([0.0, 0.0, 1.0, 0.0], 2.0, th)
    np.testing.assert_allclose(y, [-math.sin(2.0), 0.0, math.cos(2.0), 0.0], rtol=0, atol=1e-15)
    y = oracle.rope([0.0, 0.0, 0.0, 1.0], 300.0, th)
    np.testing.assert_allclose(y, [0.0, -math.sin(3.0), 0.0, math.cos(3.0)], rtol=0, atol=1e-14)
    # D = 2: a single pair rotated by position radians
    for p in (0.0, 1.0, 7.0, 32767.0):
        y = oracle.rope([0.3, -1.7], p, 5e5)
        c, s = math.cos(p), math.sin(p)
        np.testing.assert_allclose(y, [0.3 * c + 1.7 * s, -1.7 * c + 0.3 * s], rtol=0, atol=1e-13)


def test_rope_frequency_schedule():
    # the i-th pair turns at theta^(-2i/D): at position 1 a unit vector in pair i
    # comes out at angle theta^(-2i/D)
    D, th = 128, 5e5
    for i in (0, 1, 17, 63):
        x = np.zeros(D)
        x[i] = 1.0
        y = oracle.rope(x, 1.0, th)
        ang = math.atan2(y[i + D // 2], y[i])
        assert abs(ang - th ** (-2.0 * i / D)) < 1e-15


def test_rope_identity_relative_position():
    # <R_a q, R_b k> = <q, R_{b-a} k> for random vectors and positions <= 40000
    rng = np.random.default_rng(4)
    for D in (64, 128):
        for _ in range(200):
            q, k = rng.standard_normal(D), rng.standard_normal(D)
            a, b = rng.integers(0, 40000, 2)
            lhs = np.dot(oracle.rope(q, a, 5e5), oracle.rope(k, b, 5e5))
            rhs = np.dot(q, oracle.rope(k, b - a, 5e5))
            assert abs(lhs - rhs) <= 1e-12 * np.linalg.norm(q) * np.linalg.norm(k)


def test_rope_relocation_composes():
    # Theorem 1 (InferScale section 5.1): a chunk rotated at offset t and then moved
    # by P equals the chunk rotated directly at P + t (R_P R_t = R_{P+t}); R_0 = I;
    # rotations preserve the norm
    rng = np.random.default_rng(5)
    for _ in range(200):
        x = rng.standard_normal(128)
        P, t = int(rng.integers(0, 32768)), int(rng.integers(0, 64))
        two = oracle.rope(oracle.rope(x, t, 5e5), P, 5e5)
        one = oracle.rope(x, P + t, 5e5)
        assert np.max(np.abs(two - one)) <= 1e-11
        assert abs(np.linalg.norm(one) - np.linalg.norm(x)) <= 1e-12 * np.linalg.norm(x)
    x = rng.standard_normal(64)
    assert np.array_equal(oracle.rope(x, 0, 1e4), x)


def test_rope_round_rows_is_round_of_rope():
    rng = np.random.default_rng(6)
    n, D = 64, 128
    bits = oracle.encode(rng.standard_normal((n, D)), BF16)
    pos = rng.integers(0, 33000, n).astype(np.int32)
    out = oracle.rope_round_rows(bits, pos, 5e5, BF16)
    x = oracle.decode(bits, BF16)
    for i in range(n):
        y = oracle.rope(x[i], pos[i], 5e5)
        assert np.array_equal(out[i], oracle.encode(y, BF16))
    # position 0 is the identity: the row comes back bit for bit
    assert np.array_equal(oracle.rope_round_rows(bits, np.zeros(n, np.int32), 5e5, BF16), bits)


# ---------------------------------------------------------------------------
# sizes: pages' printed figures (tests/golden/kv_sizes.txt)
# ---------------------------------------------------------------------------
def _read_sizes(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "kv_sizes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, L, H, D, N, b, printed, unit, check = line.split()
            rows.append((name, int(L), int(H), int(D), int(N), int(b), float(printed),
                         int(unit), check))
    return rows


def test_kv_sizes_match_pages(golden_dir):
    rows = _read_sizes(golden_dir)
    assert len(rows) >= 10
    for name, L, H, D, N, b, printed, unit, check in rows:
        got = oracle.kv_bytes(L, H, D, N, b)
        if check == "exact":
            assert got == printed * unit, name
        elif check.startswith("round"):
            k = int(check[5:])
            assert round(got / unit, k) == printed, (name, got / unit)
        elif check == "gt":
            assert got / unit > printed, name
        else:
            raise AssertionError(check)


def test_kv_size_llama70b_exact_value():
    # 2 x 80 x 8 x 128 x 2 x 8192 = 2,684,354,560 bytes (the page's "~2.68 GB")
    assert oracle.kv_bytes(80, 8, 128, 8192, 2) == 2_684_354_560
    # and per fact (InferScale section 3.4) = 2 x L x c x h x d x b
    assert oracle.kv_bytes(32, 8, 128, 64, 2) == 2 * 32 * 64 * 8 * 128 * 2


# ---------------------------------------------------------------------------
# slot mapping: worked block tables (tests/golden/paging_examples.txt)
# ---------------------------------------------------------------------------
def _read_paging(golden_dir):
    tables, slots = {}, []
    with open(os.path.join(golden_dir, "paging_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "table":
                tables[parts[1]] = [int(v) for v in parts[2:]]
            else:
                slots.append((parts[1], int(parts[2]), int(parts[3])))
    return tables, slots


def test_slot_mapping_worked_examples(golden_dir):
    tables, slots = _read_paging(golden_dir)
    names = sorted(tables)
    max_blocks = max(len(t) for t in tables.values())
    bt = np.full((len(names), max_blocks), -1, np.int32)
    for i, nm in enumerate(names):
        bt[i, :len(tables[nm])] = tables[nm]
    seq = np.array([names.index(s[0]) for s in slots], np.int32)
    pos = np.array([s[1] for s in slots], np.int32)
    want = np.array([s[2] for s in slots], np.int64)
    got, st = oracle.slot_mapping(bt, seq, pos, 16, 100)
    assert np.array_equal(got, want)
    # position 48 of A lies past its 3-entry table; position 32 of B hits a -1 pad
    assert st == oracle.ST_BLOCK | oracle.ST_POS


def test_slot_mapping_invalid_inputs():
    bt = np.array([[3, 7, 1]], np.int32)
    got, st = oracle.slot_mapping(bt, np.array([0, 1, 0, 0], np.int32),
                                  np.array([5, 5, -1, 48], np.int32), 16, 8)
    assert list(got) == [53, -1, -1, -1]
    assert st == oracle.ST_SEQ | oracle.ST_POS
    got, st = oracle.slot_mapping(bt, np.zeros(1, np.int32), np.array([0], np.int32), 16, 3)
    assert list(got) == [-1] and st == oracle.ST_BLOCK


# ---------------------------------------------------------------------------
# attention: "LLM Inference: KV Caching", softmax(QK^T / sqrt(d)) V
# ---------------------------------------------------------------------------
def test_attention_weights_sum_to_one():
    rng = np.random.default_rng(7)
    for n in (1, 2, 17, 1000):
        q, K, V = rng.standard_normal(64) * 3, rng.standard_normal((n, 64)), rng.standard_normal((n, 64))
        _, w = oracle.attention(q, K, V, 1 / 8)
        assert abs(1 - w) <= 1e-12


def test_attention_special_cases():
    rng = np.random.default_rng(8)
    D = 64
    # one key: out = V
    V = rng.standard_normal((1, D))
    out, _ = oracle.attention(rng.standard_normal(D), rng.standard_normal((1, D)), V, 0.125)
    np.testing.assert_allclose(out, V[0], rtol=0, atol=1e-15)
    # identical keys: mean of V
    K = np.tile(rng.standard_normal(D), (9, 1))
    V = rng.standard_normal((9, D))
    out, _ = oracle.attention(rng.standard_normal(D), K, V, 0.125)
    np.testing.assert_allclose(out, V.mean(0), rtol=0, atol=1e-14)
    # q = 0: mean of V
    out, _ = oracle.attention(np.zeros(D), rng.standard_normal((9, D)), V, 0.125)
    np.testing.assert_allclose(out, V.mean(0), rtol=0, atol=1e-14)


def test_attention_two_keys_closed_form_and_scale():
    # keys 0 and a*e0, query b*e0: weight of key 1 is the logistic of a*b/sqrt(D)
    D = 128
    for a, b in ((1.0, 2.0), (3.0, -4.0), (10.0, 7.5)):
        q = np.zeros(D); q[0] = b
        K = np.zeros((2, D)); K[1, 0] = a
        V = np.zeros((2, D)); V[0, 5] = 1.0; V[1, 5] = 3.0
        out, _ = oracle.attention(q, K, V, 1 / math.sqrt(D))
        w1 = 1 / (1 + math.exp(-a * b / math.sqrt(D)))
        assert abs(out[5] - ((1 - w1) * 1.0 + w1 * 3.0)) <= 1e-14


def _scatter_to_paged(Kc, Vc, perm, B, NB, Hkv, D, dtype):
    """Place a contiguous per-request [ctx][Hkv][D] K/V into a paged cache,
    page i of the request going to physical block perm[i]."""
    kc = np.zeros((1, NB, Hkv, B, D), np.uint16)
    vc = np.zeros_like(kc)
    ctx = Kc.shape[0]
    for p in range(ctx):
        blk, off = perm[p // B], p % B
        kc[0, blk, :, off, :] = Kc[p]
        vc[0, blk, :, off, :] = Vc[p]
    return kc, vc


def test_paged_equals_contiguous_under_block_permutations():
    # paged attention reads the same keys as contiguous attention, whatever the
    # physical order of the blocks ("LLM Inference: KV Caching", "Paged attention")
    rng = np.random.default_rng(9)
    B, NB, Hkv, G, D = 16, 12, 2, 3, 64
    Hq = Hkv * G
    ctx = 150  # 10 pages, ragged last page
    Kc = oracle.encode(rng.standard_normal((ctx, Hkv, D)), BF16)
    Vc = oracle.encode(rng.standard_normal((ctx, Hkv, D)), BF16)
    q = oracle.encode(rng.standard_normal((1, Hq, D)), BF16)
    results = []
    for trial in range(4):
        perm = rng.permutation(NB)[:10].astype(np.int32)
        kc, vc = _scatter_to_paged(Kc, Vc, perm, B, NB, Hkv, D, BF16)
        bt = perm.reshape(1, -1)
        out, st = oracle.paged_decode(kc, vc, 0, q, np.array([ctx - 1], np.int32), bt,
                                      np.array([ctx], np.int32), 5e5, BF16)
        assert st == 0
        results.append(out)
    for out in results[1:]:
        assert np.array_equal(out, results[0])
    # against the textbook on the contiguous arrays (consecutive GQA groups)
    for qh in range(Hq):
        h = qh // G
        want = oracle.attention_bits(q[0, qh], ctx - 1, 5e5, Kc[:, h], Vc[:, h], BF16)
        assert np.array_equal(results[0][0, qh], want)


def test_copy_on_write_shared_prefix():
    # Two sequences point at the same physical blocks; one of them writes into the shared,
    # partly filled last block, which is therefore duplicated first and the writer's table
    # pointed at the copy ("LLM Inference: KV Caching", Paged attention; "Inside LLM
    # Inference Engines", PagedAttention, copy-on-write). Afterwards the reader's attention
    # is unchanged, and the writer's equals textbook attention over its own logical token
    # list (the shared prefix, then its new token), computed from contiguous arrays.
    rng = np.random.default_rng(21)
    L, B, NB, Hkv, G, D, theta = 2, 16, 8, 2, 2, 64, 5e5
    Hq = Hkv * G
    ctx = 37  # three pages, the last one holds 5 tokens
    Kc = oracle.encode(rng.standard_normal((ctx, Hkv, D)), BF16)
    Vc = oracle.encode(rng.standard_normal((ctx, Hkv, D)), BF16)
    shared = np.array([5, 2, 6], np.int32)
    kc = oracle.encode(rng.standard_normal((L, NB, Hkv, B, D)), BF16)  # anything elsewhere
    vc = oracle.encode(rng.standard_normal((L, NB, Hkv, B, D)), BF16)
    for p in range(ctx):
        kc[1, shared[p // B], :, p % B] = Kc[p]
        vc[1, shared[p // B], :, p % B] = Vc[p]
    qa = oracle.encode(rng.standard_normal((1, Hq, D)), BF16)
    qb = oracle.encode(rng.standard_normal((1, Hq, D)), BF16)
    bt_a = shared[None]
    out_a, st = oracle.paged_decode(kc, vc, 1, qa, [ctx - 1], bt_a, [ctx], theta, BF16)
    assert st == 0
    k0, v0 = kc.copy(), vc.copy()
    # the writer's copy of the last shared block, then its new token at position ctx
    free = 3
    assert oracle.copy_blocks(kc, vc, [shared[-1]], [free]) == 0
    bt_b = np.array([[shared[0], shared[1], free]], np.int32)
    kn = oracle.encode(rng.standard_normal((1, Hkv, D)), BF16)
    vn = oracle.encode(rng.standard_normal((1, Hkv, D)), BF16)
    assert oracle.append(kc, vc, 1, kn, vn, [ctx], [free * B + ctx % B], theta, BF16) == 0
    # the reader sees exactly what it saw before
    again, _ = oracle.paged_decode(kc, vc, 1, qa, [ctx - 1], bt_a, [ctx], theta, BF16)
    assert np.array_equal(again, out_a)
    # the writer sees the shared prefix and its own token
    out_b, st = oracle.paged_decode(kc, vc, 1, qb, [ctx], bt_b, [ctx + 1], theta, BF16)
    assert st == 0
    for qh in range(Hq):
        h = qh // G
        k_new = oracle.rope_round_rows(kn[0, h][None], [ctx], theta, BF16)
        K = np.concatenate([Kc[:, h], k_new])
        V = np.concatenate([Vc[:, h], vn[0, h][None]])
        want = oracle.attention_bits(qb[0, qh], ctx, theta, K, V, BF16)
        assert np.array_equal(out_b[0, qh], want)
    # every layer was copied; no block other than the copy changed
    for l in range(L):
        assert np.array_equal(kc[l, free, :, : ctx % B], k0[l, shared[-1], :, : ctx % B])
        assert np.array_equal(vc[0, free], v0[0, shared[-1]])
    others = [b for b in range(NB) if b != free]
    assert np.array_equal(kc[:, others], k0[:, others]) and np.array_equal(vc[:, others], v0[:, others])
    # ids outside the cache are flagged and skipped
    k1, v1 = kc.copy(), vc.copy()
    assert oracle.copy_blocks(kc, vc, [0, NB], [1, 2]) == 4
    assert np.array_equal(kc[:, 1], k1[:, 0]) and np.array_equal(kc[:, 2], k1[:, 2])


def test_sliding_window_decode():
    # under a sliding window a query attends only to the last W tokens ("LLM Inference: KV
    # Caching", sliding window attention): equal to textbook attention over the contiguous
    # last W tokens; W >= ctx is full attention; blocks wholly before the window are not read
    rng = np.random.default_rng(23)
    B, NB, Hkv, G, D, theta = 16, 12, 2, 2, 64, 5e5
    Hq = Hkv * G
    ctx = 150
    Kc = oracle.encode(rng.standard_normal((ctx, Hkv, D)), BF16)
    Vc = oracle.encode(rng.standard_normal((ctx, Hkv, D)), BF16)
    q = oracle.encode(rng.standard_normal((1, Hq, D)), BF16)
    perm = rng.permutation(NB)[:10].astype(np.int32)
    kc, vc = _scatter_to_paged(Kc, Vc, perm, B, NB, Hkv, D, BF16)
    bt = perm.reshape(1, -1)
    full, st = oracle.paged_decode(kc, vc, 0, q, [ctx - 1], bt, [ctx], theta, BF16)
    assert st == 0
    for W in (ctx, ctx + 7):
        out, st = oracle.paged_decode(kc, vc, 0, q, [ctx - 1], bt, [ctx], theta, BF16, window=W)
        assert st == 0 and np.array_equal(out, full)
    for W in (1, 16, 37, 149):
        out, st = oracle.paged_decode(kc, vc, 0, q, [ctx - 1], bt, [ctx], theta, BF16, window=W)
        assert st == 0
        for qh in range(Hq):
            h = qh // G
            want = oracle.attention_bits(q[0, qh], ctx - 1, theta, Kc[ctx - W:, h], Vc[ctx - W:, h],
                                         BF16)
            assert np.array_equal(out[0, qh], want)
    # table entries of pages wholly before the window may be anything
    bt2 = bt.copy()
    bt2[0, :5] = -1
    out, st = oracle.paged_decode(kc, vc, 0, q, [ctx - 1], bt2, [ctx], theta, BF16, window=60)
    want, _ = oracle.paged_decode(kc, vc, 0, q, [ctx - 1], bt, [ctx], theta, BF16, window=60)
    assert st == 0 and np.array_equal(out, want)


def test_paged_prefill_is_causal_attention_over_memory_and_query():
    # only the query tokens are prefilled, attending to the injected memory as if it had been
    # prefilled ("InferScale" §3.4 step 4): query token i at position p attends to tokens 0..p
    # of its request (memory, earlier query tokens, itself); checked against textbook
    # attention on contiguous arrays, two requests interleaved in the token list
    rng = np.random.default_rng(29)
    B, NB, Hkv, G, D, theta = 16, 20, 2, 2, 64, 5e5
    Hq = Hkv * G
    mem, nq = [40, 7], [5, 9]  # memory tokens and query tokens per request
    total = [m + n for m, n in zip(mem, nq)]
    Ks = [oracle.encode(rng.standard_normal((t, Hkv, D)), BF16) for t in total]
    Vs = [oracle.encode(rng.standard_normal((t, Hkv, D)), BF16) for t in total]
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((2, 5), -1, np.int32)
    kc = np.zeros((1, NB, Hkv, B, D), np.uint16)
    vc = np.zeros_like(kc)
    o = 0
    for r, t in enumerate(total):
        pages = -(-t // B)
        bt[r, :pages] = perm[o:o + pages]
        o += pages
        for p in range(t):
            kc[0, bt[r, p // B], :, p % B] = Ks[r][p]
            vc[0, bt[r, p // B], :, p % B] = Vs[r][p]
    toks = [(r, mem[r] + i) for i in range(max(nq)) for r in range(2) if i < nq[r]]
    seq = np.array([t[0] for t in toks], np.int32)
    pos = np.array([t[1] for t in toks], np.int32)
    q = oracle.encode(rng.standard_normal((len(toks), Hq, D)), BF16)
    out, st = oracle.paged_prefill(kc, vc, 0, q, seq, pos, bt, theta, BF16)
    assert st == 0
    for i, (r, p) in enumerate(toks):
        for qh in range(Hq):
            h = qh // G
            want = oracle.attention_bits(q[i, qh], p, theta, Ks[r][: p + 1, h], Vs[r][: p + 1, h],
                                         BF16)
            assert np.array_equal(out[i, qh], want)
    # causal: a later token's key changes later outputs only
    kc2 = kc.copy()
    r, p = 1, mem[1] + 4
    kc2[0, bt[r, p // B], :, p % B] ^= 0x0040
    out2, _ = oracle.paged_prefill(kc2, vc, 0, q, seq, pos, bt, theta, BF16)
    for i, (ri, pi) in enumerate(toks):
        same = np.array_equal(out2[i], out[i])
        assert same == (ri != r or pi < p), (ri, pi)
    # a position past the table or a request outside the batch is flagged
    _, st = oracle.paged_prefill(kc, vc, 0, q[:1], [0], [5 * B], bt, theta, BF16)
    assert st == 8
    _, st = oracle.paged_prefill(kc, vc, 0, q[:1], [2], [3], bt, theta, BF16)
    assert st == 32


def test_int8_rows_round_within_half_a_step():
    # int8 KV ("KV Cache Management", KV cache quantization): each row read back within half
    # a quantization step of its value, its largest magnitude on the extreme code, a zero row
    # all zeros; scaling a row by a power of two scales its step and keeps its codes
    rng = np.random.default_rng(37)
    x = rng.standard_normal((60, 64)) * np.exp2(rng.integers(-12, 12, (60, 1)))
    x[7] = 0.0
    bits = oracle.encode(x, BF16)
    xd = oracle.decode(bits, BF16)
    q, s = oracle.quantize_rows_i8(bits, BF16)
    back = q.astype(np.float64) * s[:, None].astype(np.float64)
    assert (np.abs(back - xd) <= s[:, None].astype(np.float64) * (0.5 + 1e-6)).all()
    nz = np.arange(60) != 7
    assert (np.abs(q[nz].astype(int)).max(axis=1) == 127).all()
    assert s[7] == 0 and not q[7].any()
    q2, s2 = oracle.quantize_rows_i8(oracle.encode(xd * 8.0, BF16), BF16)
    assert np.array_equal(q2, q) and np.array_equal(s2, s * np.float32(8.0))


def test_int8_decode_equals_16bit_decode_on_exact_codes():
    # rows whose values are codes times a power-of-two step (each row reaching +-127) are
    # exactly representable in bf16 and quantize back to the same codes: decoding the int8
    # cache must then give the 16-bit decode's outputs bit for bit
    rng = np.random.default_rng(41)
    L, NB, Hkv, B, D, G, theta = 1, 9, 2, 16, 64, 3, 5e5
    codes = rng.integers(-127, 128, (2, L, NB, Hkv, B, D))
    codes[..., 0] = np.where(rng.random(codes.shape[:-1]) < 0.5, 127, -127)
    step = np.exp2(rng.integers(-9, -3, (2, L, NB, Hkv, B, 1))).astype(np.float64)
    kc = oracle.encode(codes[0] * step[0], BF16)
    vc = oracle.encode(codes[1] * step[1], BF16)
    kq, ks = oracle.quantize_rows_i8(kc, BF16)
    vq, vs = oracle.quantize_rows_i8(vc, BF16)
    assert np.array_equal(kq, codes[0]) and np.array_equal(ks, step[0][..., 0].astype(np.float32))
    assert np.array_equal(vq, codes[1])
    ctx = np.array([60, 33], np.int32)  # 4 and 3 pages of 16
    bt = rng.permutation(NB)[:8].astype(np.int32).reshape(2, 4)
    bt[1, 3] = -1
    q = oracle.encode(rng.standard_normal((2, Hkv * G, D)), BF16)
    want, st = oracle.paged_decode(kc, vc, 0, q, ctx - 1, bt, ctx, theta, BF16)
    assert st == 0
    got, st = oracle.paged_decode_i8(kq, ks, vq, vs, 0, q, ctx - 1, bt, ctx, theta, BF16)
    assert st == 0 and np.array_equal(got, want)


def test_gqa_groups_are_consecutive_query_heads():
    # "groups of four share one key and value head" ("LLM Inference: KV Caching");
    # reading: query heads g*G .. g*G+G-1 use kv head g
    B, NB, Hkv, G, D = 16, 2, 2, 4, 64
    kc = np.zeros((1, NB, Hkv, B, D), np.uint16)
    vc = np.zeros_like(kc)
    vc[0, :, 0] = oracle.encode(np.full((NB, B, D), 1.0), BF16)
    vc[0, :, 1] = oracle.encode(np.full((NB, B, D), -1.0), BF16)
    q = oracle.encode(np.random.default_rng(10).standard_normal((1, Hkv * G, D)), BF16)
    out, st = oracle.paged_decode(kc, vc, 0, q, np.array([5], np.int32),
                                  np.array([[1, 0]], np.int32), np.array([20], np.int32),
                                  1e4, BF16)
    assert st == 0
    want = np.repeat([1.0, -1.0], G)
    np.testing.assert_allclose(out[0, :, 0], want, rtol=0, atol=1e-15)


def test_decode_relative_position_invariance_before_rounding():
    # the score of a key depends only on its position relative to the query
    # (InferScale section 2.3): rotate keys and query in fp64 at positions shifted
    # by any offset and the attention output does not change
    rng = np.random.default_rng(11)
    D, n = 128, 40
    q, K, V = rng.standard_normal(D), rng.standard_normal((n, D)), rng.standard_normal((n, D))
    pos = rng.permutation(1000)[:n]
    outs = []
    for shift in (0, 1, 777, 30000):
        qr = oracle.rope(q, 1000 + shift, 5e5)
        Kr = np.stack([oracle.rope(K[j], pos[j] + shift, 5e5) for j in range(n)])
        outs.append(oracle.attention(qr, Kr, V, 1 / math.sqrt(D))[0])
    for o in outs[1:]:
        np.testing.assert_allclose(o, outs[0], rtol=0, atol=1e-11)


def test_decode_invalid_context_is_flagged():
    kc = np.zeros((1, 2, 1, 16, 64), np.uint16)
    q = np.zeros((2, 1, 64), np.uint16)
    out, st = oracle.paged_decode(kc, kc, 0, q, np.array([0, 0], np.int32),
                                  np.array([[0, 1], [1, 0]], np.int32),
                                  np.array([0, 33], np.int32), 1e4, BF16)
    assert st == oracle.ST_CTX and not out.any()


# ---------------------------------------------------------------------------
# inject / append layout (InferScale section 3.4 scatter via the slot mapping)
# ---------------------------------------------------------------------------
def _tiny_pool(rng, n_chunks, L, c, Hkv, D):
    # distinct small integers: exact in bf16, every element traceable
    vals = rng.permutation(n_chunks * L * 2 * c * Hkv * D) % 251 - 125
    return oracle.encode(vals.reshape(n_chunks, L, 2, c, Hkv, D).astype(np.float64), BF16)


def test_inject_layout_and_relocation():
    rng = np.random.default_rng(12)
    n_chunks, L, c, Hkv, D, B, NB = 3, 2, 5, 2, 8, 4, 6
    pool = _tiny_pool(rng, n_chunks, L, c, Hkv, D)
    bt = np.array([[4, 1, 5, 0, 2, 3]], np.int32)
    ids = np.array([2, 0], np.int32)
    start = np.array([0, 9], np.int32)  # chunk 1 straddles a block boundary
    pos = np.concatenate([start[j] + np.arange(c) for j in range(2)]).astype(np.int32)
    slots, st = oracle.slot_mapping(bt, np.zeros(pos.size, np.int32), pos, B, NB)
    assert st == 0
    sentinel = np.uint16(0x7FC1)
    kc = np.full((L, NB, Hkv, B, D), sentinel, np.uint16)
    vc = kc.copy()
    st = oracle.inject(pool, ids, start, slots, 1e4, BF16, kc, vc)
    assert st == 0
    written = np.zeros(kc.shape[:4], bool)
    for j in range(2):
        for t in range(c):
            p = start[j] + t
            blk, off = bt[0, p // B], p % B
            for l in range(L):
                for h in range(Hkv):
                    # V: bit copy; K: the stored pre-RoPE row rotated directly at p
                    assert np.array_equal(vc[l, blk, h, off], pool[ids[j], l, 1, t, h])
                    want = oracle.rope_round_rows(pool[ids[j], l, 0, t, h][None], [p], 1e4, BF16)[0]
                    assert np.array_equal(kc[l, blk, h, off], want)
                    if p == 0:
                        assert np.array_equal(kc[l, blk, h, off], pool[ids[j], l, 0, t, h])
                    written[l, blk, h, off] = True
    assert np.all(kc[~written] == sentinel) and np.all(vc[~written] == sentinel)


def test_inject_layer_range_and_bad_ids():
    rng = np.random.default_rng(13)
    pool = _tiny_pool(rng, 2, 3, 2, 1, 4)
    kc = np.zeros((3, 4, 1, 2, 4), np.uint16)
    vc = kc.copy()
    st = oracle.inject(pool, [1], [2], [2, 3], 1e4, BF16, kc, vc, layer_begin=1, layer_end=2)
    assert st == 0
    assert not kc[0].any() and not kc[2].any() and kc[1].any()
    st = oracle.inject(pool, [5, 0], [0, 0], [0, 1, 99, 2], 1e4, BF16, kc, vc)
    assert st == oracle.ST_CHUNK | oracle.ST_SLOT


def test_append_writes_rotated_row():
    rng = np.random.default_rng(14)
    L, NB, Hkv, B, D = 2, 3, 2, 4, 8
    kc = np.zeros((L, NB, Hkv, B, D), np.uint16)
    vc = kc.copy()
    kn = oracle.encode(rng.standard_normal((2, Hkv, D)), BF16)
    vn = oracle.encode(rng.standard_normal((2, Hkv, D)), BF16)
    st = oracle.append(kc, vc, 1, kn, vn, [6, 0], [9, 4], 1e4, BF16)
    assert st == 0
    for i, (p, s) in enumerate(((6, 9), (0, 4))):
        for h in range(Hkv):
            assert np.array_equal(vc[1, s // B, h, s % B], vn[i, h])
            want = oracle.rope_round_rows(kn[i, h][None], [p], 1e4, BF16)[0]
            assert np.array_equal(kc[1, s // B, h, s % B], want)
    assert not kc[0].any()
    # already-rotated keys are copied as given
    kc2 = np.zeros_like(kc)
    oracle.append(kc2, vc, 0, kn, vn, [6, 0], [9, 4], 1e4, BF16, rotate=False)
    assert np.array_equal(kc2[0, 2, :, 1], kn[0])


def test_brute_force_tiny_decode_against_loop():
    # a second, naive statement of paged decode (Python loops, math.exp) on a
    # tiny case with a ragged last page
    rng = np.random.default_rng(15)
    B, NB, Hkv, G, D, ctx = 4, 5, 1, 2, 4, 11
    kc = oracle.encode(rng.standard_normal((1, NB, Hkv, B, D)), BF16)
    vc = oracle.encode(rng.standard_normal((1, NB, Hkv, B, D)), BF16)
    bt = np.array([[3, 0, 4]], np.int32)
    q = oracle.encode(rng.standard_normal((1, G, D)), BF16)
    out, st = oracle.paged_decode(kc, vc, 0, q, [10], bt, [ctx], 1e4, BF16)
    assert st == 0
    Kf, Vf = oracle.decode(kc, BF16), oracle.decode(vc, BF16)
    for qh in range(G):
        qv = oracle.decode(q[0, qh], BF16)
        qr = [0.0] * D
        for i in range(D // 2):
            ang = 10 * 1e4 ** (-2 * i / D)
            qr[i] = qv[i] * math.cos(ang) - qv[i + D // 2] * math.sin(ang)
            qr[i + D // 2] = qv[i + D // 2] * math.cos(ang) + qv[i] * math.sin(ang)
        s = []
        for j in range(ctx):
            k = Kf[0, bt[0, j // B], 0, j % B]
            s.append(sum(qr[d] * k[d] for d in range(D)) / math.sqrt(D))
        m = max(s)
        e = [math.exp(x - m) for x in s]
        want = [sum(e[j] * Vf[0, bt[0, j // B], 0, j % B][d] for j in range(ctx)) / sum(e)
                for d in range(D)]
        np.testing.assert_allclose(out[0, qh], want, rtol=0, atol=1e-13)
