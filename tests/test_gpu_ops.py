"""GPU parity of each entry point against the fp64 oracle, element by element,
on seeded inputs that span several pages, CTAs and a ragged tail; plus the
edge cases (empty, ragged, single token, invalid indices, workspace size).

Inputs come from the shared seeded generator (workload); expectations only
from oracle/. Calls go through the C ABI (ctypes binding)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workload as W
from paged_kv_cache_inject_gb300 import kvinj as K
from tests.gpu_helpers import assert_decode_close, bits, from_bits, torch_dtype, ulp_distance

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC1  # a NaN pattern no kernel writes


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()


def gen_bits(seed: int, shape, dt):
    key = W.stream_key(seed, W.STREAM_POOL)
    n = int(np.prod(shape))
    return W.normal_bits(key, np.arange(n, dtype=np.uint64), dt).reshape(shape)


def i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------------------
# slot mapping
# ---------------------------------------------------------------------------
def test_slot_mapping_bit_exact():
    rng = np.random.default_rng(1)
    batch, max_blocks, NB, B = 7, 40, 300, 16
    bt = rng.permutation(NB)[:batch * max_blocks].reshape(batch, max_blocks).astype(np.int32)
    n = 100_003
    seq = rng.integers(0, batch, n).astype(np.int32)
    pos = rng.integers(0, max_blocks * B, n).astype(np.int32)
    want, st = oracle.slot_mapping(bt, seq, pos, B, NB)
    assert st == 0
    out = torch.empty(n, dtype=torch.int64, device="cuda")
    status = status_tensor()
    K.kvinj_slot_mapping(i32(bt), i32(seq), i32(pos), NB, B, out, status)
    assert np.array_equal(out.cpu().numpy(), want)
    assert status.item() == 0


def test_slot_mapping_invalid_entries_flagged():
    bt = np.array([[3, 7, 1], [2, 9, -1]], np.int32)
    seq = np.array([0, 1, 5, 0, 1, -1, 0], np.int32)
    pos = np.array([20, 16, 0, 48, 40, 0, -3], np.int32)
    want, st = oracle.slot_mapping(bt, seq, pos, 16, 10)
    out = torch.empty(seq.size, dtype=torch.int64, device="cuda")
    status = status_tensor()
    K.kvinj_slot_mapping(i32(bt), i32(seq), i32(pos), 10, 16, out, status)
    assert np.array_equal(out.cpu().numpy(), want)
    assert list(want) == [116, 144, -1, -1, -1, -1, -1]
    assert status.item() == K.ST_BAD_SEQ | K.ST_BAD_POS | K.ST_BAD_BLOCK


# ---------------------------------------------------------------------------
# inject
# ---------------------------------------------------------------------------
def _inject_case(D, dt, seed=3):
    rng = np.random.default_rng(seed)
    L, Hkv, c, n_chunks, B, NB = 3, 4, 5, 7, 16, 24
    pool = gen_bits(seed, (n_chunks, L, 2, c, Hkv, D), dt)
    perm = rng.permutation(NB).astype(np.int32)
    bt = perm.reshape(2, 12)
    ids = np.array([3, 0, 6, 3], np.int32)
    req = np.array([0, 0, 1, 1], np.int32)
    start = np.array([0, 13, 100, 187], np.int32)  # one chunk straddles a block, one ends the table
    seq = np.repeat(req, c).astype(np.int32)
    pos = (start[:, None] + np.arange(c)).reshape(-1).astype(np.int32)
    slots, st = oracle.slot_mapping(bt, seq, pos, B, NB)
    assert st == 0
    return dict(L=L, Hkv=Hkv, c=c, B=B, NB=NB, pool=pool, bt=bt, ids=ids, start=start, seq=seq,
                pos=pos, slots=slots)


@pytest.mark.parametrize("D,dt", [(64, W.BF16), (128, W.BF16), (128, W.FP16), (256, W.BF16)])
def test_inject_matches_oracle(D, dt):
    cs = _inject_case(D, dt)
    L, Hkv, B, NB = cs["L"], cs["Hkv"], cs["B"], cs["NB"]
    tdt = torch_dtype(dt)
    theta = 5e5 if D == 128 else 1e4
    kc = np.full((L, NB, Hkv, B, D), SENTINEL, np.uint16)
    vc = kc.copy()
    assert oracle.inject(cs["pool"], cs["ids"], cs["start"], cs["slots"], theta, dt, kc, vc) == 0

    cache = K.Cache(from_bits(np.full_like(kc, SENTINEL), tdt), from_bits(np.full_like(kc, SENTINEL), tdt))
    pool = K.Pool(from_bits(cs["pool"], tdt))
    rope = K.make_rope(theta, D, 200)
    slots_d = torch.empty(cs["pos"].size, dtype=torch.int64, device="cuda")
    status = status_tensor()
    K.kvinj_slot_mapping(i32(cs["bt"]), i32(cs["seq"]), i32(cs["pos"]), NB, B, slots_d, status)
    assert np.array_equal(slots_d.cpu().numpy(), cs["slots"])
    K.kvinj_inject(pool, cache, rope, i32(cs["ids"]), i32(cs["start"]), slots_d, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    gk, gv = bits(cache.k), bits(cache.v)
    assert np.array_equal(gv, vc), "V must be a bit copy and nothing else may change"
    written = kc != SENTINEL
    assert np.array_equal(gk[~written], kc[~written])
    d = ulp_distance(gk[written], kc[written])
    assert d.max() <= 1, f"rotated K beyond one ulp: {d.max()}"
    assert (d == 0).mean() > 0.99


def test_inject_layer_range_and_bad_indices():
    D, dt = 128, W.BF16
    cs = _inject_case(D, dt, seed=4)
    L, Hkv, B, NB = cs["L"], cs["Hkv"], cs["B"], cs["NB"]
    tdt = torch_dtype(dt)
    kc = np.full((L, NB, Hkv, B, D), SENTINEL, np.uint16)
    vc = kc.copy()
    # layers [1, 2) only; chunk 1 has a bad id, chunk 2 a bad slot on token 0 and chunk 3 runs
    # past the rope table (max_pos 190: positions 187..191)
    ids = cs["ids"].copy()
    ids[1] = 99
    slots = cs["slots"].copy()
    slots[2 * cs["c"]] = -1
    ok_ids = ids.copy()
    orc_slots = slots.copy()
    st = oracle.inject(cs["pool"], ok_ids, cs["start"], orc_slots, 1e4, dt, kc, vc,
                       layer_begin=1, layer_end=2)
    assert st == oracle.ST_CHUNK | oracle.ST_SLOT
    # the oracle has no table limit: undo what it wrote past position 189
    for j in range(len(ids)):
        for t in range(cs["c"]):
            if cs["start"][j] + t >= 190 and ids[j] < 7 and slots[j * cs["c"] + t] >= 0:
                s = slots[j * cs["c"] + t]
                kc[1, s // B, :, s % B] = SENTINEL
                vc[1, s // B, :, s % B] = SENTINEL
    cache = K.Cache(from_bits(np.full_like(kc, SENTINEL), tdt), from_bits(np.full_like(kc, SENTINEL), tdt))
    pool = K.Pool(from_bits(cs["pool"], tdt))
    rope = K.make_rope(1e4, D, 190)
    status = status_tensor()
    K.kvinj_inject(pool, cache, rope, i32(ids), i32(cs["start"]),
                   torch.from_numpy(slots).cuda(), 1, 2, status)
    torch.cuda.synchronize()
    assert status.item() == K.ST_BAD_CHUNK | K.ST_BAD_SLOT | K.ST_BAD_POS
    gk, gv = bits(cache.k), bits(cache.v)
    assert np.array_equal(gv, vc)
    assert ulp_distance(gk, kc).max() <= 1
    assert np.all(gk[0] == SENTINEL) and np.all(gk[2] == SENTINEL)


@pytest.mark.parametrize("D,dt", [(128, W.BF16), (64, W.FP16)])
def test_inject_from_pinned_host_pool(D, dt):
    # the chunk pool kept in page-locked host memory ("InferScale" §6.7, Table 6) and read
    # in place: the same cache bits as with the pool in device memory, within one ulp of
    # the oracle for rotated K, V copied exactly
    cs = _inject_case(D, dt, seed=11)
    L, Hkv, B, NB = cs["L"], cs["Hkv"], cs["B"], cs["NB"]
    tdt = torch_dtype(dt)
    theta = 5e5
    kc = np.full((L, NB, Hkv, B, D), SENTINEL, np.uint16)
    vc = kc.copy()
    assert oracle.inject(cs["pool"], cs["ids"], cs["start"], cs["slots"], theta, dt, kc, vc) == 0
    rope = K.make_rope(theta, D, 200)
    slots_d = torch.from_numpy(cs["slots"]).cuda()
    got = {}
    for where in ("device", "host"):
        data = from_bits(cs["pool"], tdt)
        if where == "host":
            data = data.cpu().pin_memory()
            assert not data.is_cuda and data.is_pinned()
        cache = K.Cache(from_bits(np.full_like(kc, SENTINEL), tdt),
                        from_bits(np.full_like(kc, SENTINEL), tdt))
        status = status_tensor()
        K.kvinj_inject(K.Pool(data), cache, rope, i32(cs["ids"]), i32(cs["start"]), slots_d,
                       status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        got[where] = (bits(cache.k), bits(cache.v))
    (dk, dv), (hk, hv) = got["device"], got["host"]
    assert np.array_equal(hk, dk) and np.array_equal(hv, dv)
    assert np.array_equal(hv, vc)
    written = kc != SENTINEL
    assert np.array_equal(hk[~written], kc[~written])
    assert ulp_distance(hk[written], kc[written]).max() <= 1


def test_inject_refuses_pageable_host_pool():
    # host memory that is not page-locked has no device mapping: refused on the host,
    # nothing launched, the cache untouched
    D, dt = 128, W.BF16
    cs = _inject_case(D, dt, seed=12)
    L, Hkv, B, NB, c = cs["L"], cs["Hkv"], cs["B"], cs["NB"], cs["c"]
    host = np.ascontiguousarray(cs["pool"])
    assert host.ctypes.data % 16 == 0

    class PageablePool:  # the descriptor as a C caller would fill it
        def __init__(self):
            self._s = K._Pool(L, Hkv, D, c, host.shape[0], dt, host.ctypes.data)

        @property
        def ref(self):
            return ctypes.byref(self._s)

    cache = K.Cache(torch.zeros((L, NB, Hkv, B, D), dtype=torch.bfloat16, device="cuda"),
                    torch.zeros((L, NB, Hkv, B, D), dtype=torch.bfloat16, device="cuda"))
    rope = K.make_rope(1e4, D, 200)
    with pytest.raises(K.KvinjError) as e:
        K.kvinj_inject(PageablePool(), cache, rope, i32(cs["ids"]), i32(cs["start"]),
                       torch.from_numpy(cs["slots"]).cuda())
    assert e.value.code == K.KVINJ_EINVAL
    torch.cuda.synchronize()
    assert not cache.k.any() and not cache.v.any()


@pytest.mark.parametrize("D,dt", [(128, W.BF16), (64, W.FP16), (256, W.BF16)])
def test_copy_blocks_matches_oracle(D, dt):
    # copy-on-write block copies: bit-exact, only the listed layers, bad ids skipped
    rng = np.random.default_rng(31 + D)
    L, NB, Hkv, B = 3, 40, 4, 16
    tdt = torch_dtype(dt)
    kc = gen_bits(31, (L, NB, Hkv, B, D), dt)
    vc = gen_bits(32, (L, NB, Hkv, B, D), dt)
    perm = rng.permutation(NB).astype(np.int32)
    src, dst = perm[:13].copy(), perm[13:26].copy()
    src[4] = NB + 3  # an id outside the cache: skipped, flagged
    want_k, want_v = kc.copy(), vc.copy()
    assert oracle.copy_blocks(want_k, want_v, src, dst, 1, 3) == 4
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    status = status_tensor()
    K.kvinj_copy_blocks(cache, i32(src), i32(dst), 1, 3, status=status)
    torch.cuda.synchronize()
    assert status.item() == K.ST_BAD_BLOCK
    assert np.array_equal(bits(cache.k), want_k) and np.array_equal(bits(cache.v), want_v)
    # empty calls change nothing
    K.kvinj_copy_blocks(cache, i32(src[:0]), i32(dst[:0]))
    K.kvinj_copy_blocks(cache, i32(src), i32(dst), 2, 2)
    torch.cuda.synchronize()
    assert np.array_equal(bits(cache.k), want_k)


def test_copy_on_write_then_append_and_decode():
    # two requests share a prefix of blocks; the second writes into the shared, partly
    # filled last block: it gets a private copy first, then appends its token and both
    # decode (the reader's output bit for bit as before the write)
    D, G, dt, Hkv, theta = 128, 4, W.BF16, 8, 5e5
    tdt = torch_dtype(dt)
    ctx = 1000  # 63 pages, the last holding 8 tokens
    kc, vc, q, bt = _decode_case(D, G, dt, [ctx], Hkv=Hkv, L=2, seed=33, spare=4)
    NB = kc.shape[1]
    free = int(np.setdiff1d(np.arange(NB), bt[0][bt[0] >= 0])[0])
    pages = -(-ctx // 16)
    bt_a = bt.copy()
    bt_b = bt.copy()
    bt_b[0, pages - 1] = free
    qb = gen_bits(34, q.shape, dt)
    kn = gen_bits(35, (1, Hkv, D), dt)
    vn = gen_bits(36, (1, Hkv, D), dt)
    slot = np.array([free * 16 + ctx % 16], np.int64)
    # oracle
    ek, ev = kc.copy(), vc.copy()
    assert oracle.copy_blocks(ek, ev, [bt[0, pages - 1]], [free]) == 0
    assert oracle.append(ek, ev, 1, kn, vn, [ctx], slot, theta, dt) == 0
    want_a, _ = oracle.paged_decode(ek, ev, 1, q, [ctx - 1], bt_a, [ctx], theta, dt)
    want_b, _ = oracle.paged_decode(ek, ev, 1, qb, [ctx], bt_b, [ctx + 1], theta, dt)
    # library
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(theta, D, ctx + 8)
    ws = K.make_decode_workspace(1, Hkv * G, Hkv, D)
    status = status_tensor()

    def decode(qbits, pos, table, c):
        out = torch.empty((1, Hkv * G, D), dtype=tdt, device="cuda")
        K.kvinj_paged_decode(cache, rope, 1, from_bits(qbits, tdt), i32(np.array([pos])),
                             i32(table), i32(np.array([c])), out, ws, 0.0, status)
        torch.cuda.synchronize()
        return out.float().cpu().numpy().astype(np.float64)

    before_a = decode(q, ctx - 1, bt_a, ctx)
    K.kvinj_copy_blocks(cache, i32(np.array([bt[0, pages - 1]])), i32(np.array([free])),
                        status=status)
    K.kvinj_append(cache, rope, 1, from_bits(kn, tdt), from_bits(vn, tdt),
                   i32(np.array([ctx])), torch.from_numpy(slot).cuda(), status=status)
    got_a = decode(q, ctx - 1, bt_a, ctx)
    got_b = decode(qb, ctx, bt_b, ctx + 1)
    assert status.item() == 0
    assert np.array_equal(got_a, before_a)
    assert_decode_close(got_a, want_a, "reader after copy-on-write")
    assert_decode_close(got_b, want_b, "writer after copy-on-write")
    assert ulp_distance(bits(cache.k), ek).max() <= 1  # the appended K is rotated
    assert np.array_equal(bits(cache.v), ev)


def test_inject_empty_is_noop():
    D = 64
    cache = K.Cache(torch.zeros((1, 2, 1, 16, D), dtype=torch.bfloat16, device="cuda"),
                    torch.zeros((1, 2, 1, 16, D), dtype=torch.bfloat16, device="cuda"))
    pool = K.Pool(torch.ones((1, 1, 2, 4, 1, D), dtype=torch.bfloat16, device="cuda"))
    rope = K.make_rope(1e4, D, 16)
    e32 = torch.empty(0, dtype=torch.int32, device="cuda")
    K.kvinj_inject(pool, cache, rope, e32, e32, torch.empty(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert not cache.k.any() and not cache.v.any()


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D,dt,rotate", [(128, W.BF16, True), (64, W.FP16, True),
                                         (128, W.BF16, False), (256, W.FP16, True)])
def test_append_matches_oracle(D, dt, rotate):
    rng = np.random.default_rng(5)
    L, Hkv, B, NB, n = 2, 3, 16, 9, 37
    tdt = torch_dtype(dt)
    kn = gen_bits(10 + D, (n, Hkv, D), dt)
    vn = gen_bits(20 + D, (n, Hkv, D), dt)
    slots = rng.permutation(NB * B)[:n].astype(np.int64)
    pos = rng.integers(0, 4000, n).astype(np.int32)
    kc = np.full((L, NB, Hkv, B, D), SENTINEL, np.uint16)
    vc = kc.copy()
    assert oracle.append(kc, vc, 1, kn, vn, pos, slots, 5e5, dt, rotate=rotate) == 0
    cache = K.Cache(from_bits(np.full_like(kc, SENTINEL), tdt), from_bits(np.full_like(kc, SENTINEL), tdt))
    rope = K.make_rope(5e5, D, 4000) if rotate else None
    status = status_tensor()
    K.kvinj_append(cache, rope, 1, from_bits(kn, tdt), from_bits(vn, tdt), i32(pos),
                   torch.from_numpy(slots).cuda(), status)
    torch.cuda.synchronize()
    assert status.item() == 0
    gk, gv = bits(cache.k), bits(cache.v)
    assert np.array_equal(gv, vc)
    d = ulp_distance(gk, kc)
    assert d.max() <= (1 if rotate else 0)


# ---------------------------------------------------------------------------
# paged decode
# ---------------------------------------------------------------------------
def _decode_case(D, G, dt, ctx, Hkv=2, L=2, seed=7, spare=3):
    rng = np.random.default_rng(seed)
    B = 16
    ctx = np.asarray(ctx, np.int32)
    pages = -(-ctx // B)
    NB = int(pages.sum()) + spare
    max_blocks = int(pages.max()) + 2
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((ctx.size, max_blocks), -1, np.int32)
    o = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[o:o + p]
        o += p
    kc = gen_bits(seed, (L, NB, Hkv, B, D), dt)
    vc = gen_bits(seed + 1, (L, NB, Hkv, B, D), dt)
    q = gen_bits(seed + 2, (ctx.size, Hkv * G, D), dt)
    return kc, vc, q, bt


def _run_decode(kc, vc, q, bt, ctx, q_pos, dt, layer, theta, rope_max, variant=0, ctas=0,
                rotate=True, ws_bytes=None, status=None, scale=0.0):
    tdt = torch_dtype(dt)
    D = kc.shape[-1]
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(theta, D, rope_max) if rotate else None
    batch, Hq, _ = q.shape
    Hkv = kc.shape[2]
    n = K.kvinj_decode_workspace_size(batch, Hq, Hkv, D) if ws_bytes is None else ws_bytes
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.full((batch, Hq, D), float("nan"), dtype=tdt, device="cuda")
    K.kvinj_paged_decode_ex(cache, rope, layer, from_bits(q, tdt), i32(q_pos), i32(bt), i32(ctx),
                            out, ws, scale, status, None, variant, ctas)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), ws


DECODE_SHAPES = [(64, 1, W.BF16), (64, 2, W.BF16), (128, 4, W.BF16), (128, 8, W.BF16),
                 (128, 1, W.FP16), (128, 4, W.FP16), (64, 8, W.FP16), (128, 2, W.BF16),
                 (128, 16, W.BF16), (64, 16, W.FP16)]


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("D,G,dt", DECODE_SHAPES)
@pytest.mark.parametrize("ctas", [0, 1, 5, 37])
def test_decode_matches_oracle(D, G, dt, ctas, variant):
    if variant == 1 and G == 16:
        pytest.skip("the CUDA-core kernel covers G <= 8")
    ctx = [1, 16, 17, 250, 611]
    kc, vc, q, bt = _decode_case(D, G, dt, ctx)
    ctx = np.array(ctx, np.int32)
    q_pos = ctx - 1
    theta = 5e5
    status = status_tensor()
    got, _ = _run_decode(kc, vc, q, bt, ctx, q_pos, dt, 1, theta, 1000, ctas=ctas, status=status,
                         variant=variant)
    assert status.item() == 0
    want, st = oracle.paged_decode(kc, vc, 1, q, q_pos, bt, ctx, theta, dt)
    assert st == 0
    assert_decode_close(got, want, f"D{D} G{G} dt{dt} ctas{ctas} variant{variant}")


@pytest.mark.parametrize("variant", [1, 2])
def test_decode_long_context_and_unrotated_query(variant):
    D, G, dt = 128, 8, W.BF16
    ctx = np.array([9000, 3, 4097], np.int32)
    kc, vc, q, bt = _decode_case(D, G, dt, ctx, Hkv=1, L=1, seed=11)
    got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 0, 5e5, 9000, variant=variant)
    want, _ = oracle.paged_decode(kc, vc, 0, q, ctx - 1, bt, ctx, 5e5, dt)
    assert_decode_close(got, want, "long")
    got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 0, 5e5, 9000, rotate=False,
                         variant=variant)
    want, _ = oracle.paged_decode(kc, vc, 0, q, ctx - 1, bt, ctx, 5e5, dt, rotate_q=False)
    assert_decode_close(got, want, "unrotated")


def test_decode_deterministic_and_workspace_reusable():
    D, G, dt = 128, 4, W.BF16
    ctx = np.array([700, 33, 1500, 16], np.int32)
    kc, vc, q, bt = _decode_case(D, G, dt, ctx, seed=12)
    tdt = torch_dtype(dt)
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(5e5, D, 2000)
    ws = K.make_decode_workspace(4, 4 * 2, 2, D)
    outs = []
    for _ in range(3):
        out = torch.empty((4, 8, D), dtype=tdt, device="cuda")
        K.kvinj_paged_decode(cache, rope, 0, from_bits(q, tdt), i32(ctx - 1), i32(bt), i32(ctx),
                             out, ws)
        outs.append(bits(out))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    # a workspace needs no initialisation: garbage in it changes nothing
    ws.fill_(0xAB)
    out = torch.empty((4, 8, D), dtype=tdt, device="cuda")
    K.kvinj_paged_decode(cache, rope, 0, from_bits(q, tdt), i32(ctx - 1), i32(bt), i32(ctx), out, ws)
    assert np.array_equal(bits(out), outs[0])


@pytest.mark.parametrize("variant", [1, 2])
def test_decode_invalid_context_and_block(variant):
    D, G, dt = 64, 2, W.BF16
    ctx_ok = [40, 50, 60]
    kc, vc, q, bt = _decode_case(D, G, dt, ctx_ok, seed=13)
    ctx = np.array([0, 50, 10 ** 6], np.int32)
    status = status_tensor()
    got, _ = _run_decode(kc, vc, q, bt, ctx, np.array([0, 49, 0], np.int32), dt, 0, 1e4, 100,
                         status=status, variant=variant)
    assert status.item() == K.ST_BAD_CTX
    assert not got[0].any() and not got[2].any()
    want, _ = oracle.paged_decode(kc, vc, 0, q[1:2], [49], bt[1:2], [50], 1e4, dt)
    assert_decode_close(got[1:2], want, "valid request next to invalid ones")
    # a block-table entry outside the cache: flagged, other requests unaffected
    bt2 = bt.copy()
    bt2[0, 1] = kc.shape[1] + 5
    status = status_tensor()
    got, _ = _run_decode(kc, vc, q, bt2, np.array(ctx_ok, np.int32), np.array(ctx_ok) - 1, dt, 0,
                         1e4, 100, status=status, variant=variant)
    assert status.item() == K.ST_BAD_BLOCK
    want, _ = oracle.paged_decode(kc, vc, 0, q[1:], np.array(ctx_ok[1:]) - 1, bt[1:], ctx_ok[1:],
                                  1e4, dt)
    assert_decode_close(got[1:], want, "requests after a bad block")


def test_decode_workspace_too_small_is_refused():
    D, G, dt = 64, 1, W.BF16
    kc, vc, q, bt = _decode_case(D, G, dt, [20], seed=14)
    with pytest.raises(K.KvinjError) as e:
        _run_decode(kc, vc, q, bt, np.array([20], np.int32), np.array([19], np.int32), dt, 0, 1e4,
                    40, ws_bytes=64)
    assert e.value.code == K.KVINJ_EWORKSPACE


def _umma_covers(D, G, Hkv):
    return D == 128 and Hkv % 8 == 0 and G in (1, 2, 4, 8)


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("Hkv,G,D", [(4, 4, 128), (8, 4, 128), (12, 2, 64), (16, 1, 128),
                                     (8, 8, 128)])
def test_decode_head_groups(Hkv, G, D, variant):
    # units cover a block of up to 8 kv heads; several groups per block when Hkv > 8
    if variant == 3 and not _umma_covers(D, G, Hkv):
        pytest.skip("the tcgen05 kernel needs D = 128 and groups of 8 kv heads")
    dt = W.BF16
    ctx = [3, 100, 257, 48]
    kc, vc, q, bt = _decode_case(D, G, dt, ctx, Hkv=Hkv, L=2, seed=21 + Hkv)
    ctx = np.array(ctx, np.int32)
    for ctas in (0, 7):
        status = status_tensor()
        got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 1, 5e5, 400, ctas=ctas,
                             status=status, variant=variant)
        assert status.item() == 0
        want, _ = oracle.paged_decode(kc, vc, 1, q, ctx - 1, bt, ctx, 5e5, dt)
        assert_decode_close(got, want, f"Hkv{Hkv} G{G} D{D} ctas{ctas} variant{variant}")


# ---------------------------------------------------------------------------
# tcgen05 decode (variant 3): D = 128, head groups of 8 kv heads
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("dt", [W.BF16, W.FP16])
@pytest.mark.parametrize("Hkv", [8, 16])
@pytest.mark.parametrize("ctas", [0, 1, 5, 37])
def test_decode_umma_matches_oracle(G, dt, Hkv, ctas):
    ctx = [1, 16, 17, 250, 611]
    kc, vc, q, bt = _decode_case(128, G, dt, ctx, Hkv=Hkv, seed=40 + G + Hkv)
    ctx = np.array(ctx, np.int32)
    status = status_tensor()
    got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 1, 5e5, 1000, ctas=ctas, status=status,
                         variant=3)
    assert status.item() == 0
    want, st = oracle.paged_decode(kc, vc, 1, q, ctx - 1, bt, ctx, 5e5, dt)
    assert st == 0
    assert_decode_close(got, want, f"umma G{G} dt{dt} Hkv{Hkv} ctas{ctas}")


@pytest.mark.parametrize("scale", [0.0, 0.5, 3.0])
@pytest.mark.parametrize("G", [4, 8])
def test_decode_umma_large_logits_move_the_maximum(scale, G):
    # with large logit scales the per-head maximum jumps by far more than the
    # lazy-rescale threshold from unit to unit: exercises the O / l rescaling
    dt = W.BF16
    ctx = np.array([2000, 517, 64, 1300], np.int32)
    kc, vc, q, bt = _decode_case(128, G, dt, ctx, Hkv=8, L=1, seed=50 + G)
    for ctas in (0, 3):
        status = status_tensor()
        got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 0, 5e5, 2100, ctas=ctas,
                             status=status, variant=3, scale=scale)
        assert status.item() == 0
        want, _ = oracle.paged_decode(kc, vc, 0, q, ctx - 1, bt, ctx, 5e5, dt, scale=scale)
        assert_decode_close(got, want, f"umma scale{scale} G{G} ctas{ctas}")


@pytest.mark.parametrize("G", [4, 8])
def test_decode_umma_long_context_unrotated_and_bad_inputs(G):
    # at G = 8 a unit spans two blocks: a bad entry in either half is caught
    D, dt = 128, W.BF16
    ctx = np.array([9000, 3, 4097], np.int32)
    kc, vc, q, bt = _decode_case(D, G, dt, ctx, Hkv=8, L=1, seed=61)
    got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 0, 5e5, 9000, variant=3)
    want, _ = oracle.paged_decode(kc, vc, 0, q, ctx - 1, bt, ctx, 5e5, dt)
    assert_decode_close(got, want, "umma long")
    got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 0, 5e5, 9000, rotate=False, variant=3)
    want, _ = oracle.paged_decode(kc, vc, 0, q, ctx - 1, bt, ctx, 5e5, dt, rotate_q=False)
    assert_decode_close(got, want, "umma unrotated")
    # invalid context lengths: zero output and a status bit, neighbours intact
    bad = np.array([0, 3, 10 ** 6], np.int32)
    status = status_tensor()
    got, _ = _run_decode(kc, vc, q, bt, bad, np.array([0, 2, 0], np.int32), dt, 0, 5e5, 9000,
                         status=status, variant=3)
    assert status.item() == K.ST_BAD_CTX
    assert not got[0].any() and not got[2].any()
    want, _ = oracle.paged_decode(kc, vc, 0, q[1:2], [2], bt[1:2], [3], 5e5, dt)
    assert_decode_close(got[1:2], want, "umma valid request next to invalid ones")
    for idx in (4, 5):
        bt2 = bt.copy()
        bt2[0, idx] = kc.shape[1] + 7  # a block-table entry outside the cache
        status = status_tensor()
        got, _ = _run_decode(kc, vc, q, bt2, ctx, ctx - 1, dt, 0, 5e5, 9000, status=status,
                             variant=3)
        assert status.item() == K.ST_BAD_BLOCK
        want, _ = oracle.paged_decode(kc, vc, 0, q[1:], ctx[1:] - 1, bt[1:], ctx[1:], 5e5, dt)
        assert_decode_close(got[1:], want, f"umma requests after bad block {idx}")


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("G", [4, 8])
def test_decode_ignores_nan_rows_past_the_context(variant, G):
    # rows of a request's last block past its context may hold anything; NaN
    # bit patterns there must not reach the output (at G = 8 the tcgen05 kernel's
    # units span two blocks: also the second block's rows of a unit the context
    # ends before, e.g. 7 or 16 tokens)
    D, dt, Hkv = 128, W.BF16, 8
    ctx = np.array([33, 250, 7, 16], np.int32)
    kc, vc, q, bt = _decode_case(D, G, dt, ctx, Hkv=Hkv, L=2, seed=71)
    for r, c in enumerate(ctx):
        if c % 16:
            blk = bt[r, c // 16]
            kc[1, blk, :, c % 16:, :] = 0x7FC0
            vc[1, blk, :, c % 16:, :] = 0xFFC1
    got, _ = _run_decode(kc, vc, q, bt, ctx, ctx - 1, dt, 1, 5e5, 300, variant=variant)
    assert np.isfinite(got).all()
    want, _ = oracle.paged_decode(kc, vc, 1, q, ctx - 1, bt, ctx, 5e5, dt)
    assert_decode_close(got, want, f"nan tail variant{variant} G{G}")


def test_decode_umma_refuses_shapes_it_does_not_cover():
    dt = W.BF16
    for D, G, Hkv in [(64, 4, 8), (128, 4, 4), (128, 16, 8)]:
        kc, vc, q, bt = _decode_case(D, G, dt, [20], Hkv=Hkv, seed=81)
        with pytest.raises(K.KvinjError) as e:
            _run_decode(kc, vc, q, bt, np.array([20], np.int32), np.array([19], np.int32), dt, 0,
                        1e4, 40, variant=3)
        assert e.value.code == K.KVINJ_EUNSUPPORTED


# ---------------------------------------------------------------------------
# sliding-window decode (tcgen05 kernel)
# ---------------------------------------------------------------------------
def _run_window(kc, vc, q, bt, ctx, window, dt, theta, rope_max, kn=None, vn=None, status=None):
    tdt = torch_dtype(dt)
    D = kc.shape[-1]
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(theta, D, rope_max)
    batch, Hq, _ = q.shape
    ws = K.make_decode_workspace(batch, Hq, kc.shape[2], D)
    out = torch.full((batch, Hq, D), float("nan"), dtype=tdt, device="cuda")
    K.kvinj_paged_decode_window(cache, rope, 1, from_bits(q, tdt), i32(ctx - 1), i32(bt), i32(ctx),
                                window, out, ws,
                                k_new=None if kn is None else from_bits(kn, tdt),
                                v_new=None if vn is None else from_bits(vn, tdt), status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), cache


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("window", [1, 16, 37, 100, 1000])
def test_decode_window_matches_oracle(G, window):
    dt, theta = W.BF16, 5e5
    ctx = np.array([1, 16, 17, 250, 611, 33], np.int32)
    kc, vc, q, bt = _decode_case(128, G, dt, ctx, Hkv=8, L=2, seed=60 + G)
    status = status_tensor()
    got, _ = _run_window(kc, vc, q, bt, ctx, window, dt, theta, 700, status=status)
    assert status.item() == 0
    want, st = oracle.paged_decode(kc, vc, 1, q, ctx - 1, bt, ctx, theta, dt, window=window)
    assert st == 0
    assert_decode_close(got, want, f"window {window} G{G}")


@pytest.mark.parametrize("G", [4, 8])
def test_decode_window_ignores_pages_before_it(G):
    # table entries of pages wholly before the window are never read (here: -1), and a
    # two-block unit that starts one page before the window still sees the right tokens
    dt, theta = W.BF16, 5e5
    ctx = np.array([611, 250, 1000], np.int32)
    kc, vc, q, bt = _decode_case(128, G, dt, ctx, Hkv=8, L=2, seed=70 + G)
    window = 150  # first attended tokens 461, 100, 850: pages 28, 6, 53 (even and odd)
    bt2 = bt.copy()
    for r, c in enumerate(ctx):
        bt2[r, : (c - window) // 16] = -1
    status = status_tensor()
    got, _ = _run_window(kc, vc, q, bt2, ctx, window, dt, theta, 1100, status=status)
    assert status.item() == 0
    want, st = oracle.paged_decode(kc, vc, 1, q, ctx - 1, bt2, ctx, theta, dt, window=window)
    assert st == 0
    assert_decode_close(got, want, f"window before-pages G{G}")


def test_decode_window_fused_append_and_refusals():
    D, G, dt, Hkv, theta = 128, 4, W.BF16, 8, 5e5
    ctx = np.array([700, 33, 1500, 16], np.int32)
    kc, vc, q, bt, kn, vn, ctx, pos, slots, theta, ek, ev, _ = _fused_case(D, G, dt, list(ctx),
                                                                         Hkv, seed=77)
    want, st = oracle.paged_decode(ek, ev, 1, q, pos, bt, ctx, theta, dt, window=200)
    assert st == 0
    status = status_tensor()
    got, cache = _run_window(kc, vc, q, bt, ctx, 200, dt, theta, int(ctx.max()) + 4, kn=kn, vn=vn,
                             status=status)
    assert status.item() == 0
    assert np.array_equal(bits(cache.v), ev) and ulp_distance(bits(cache.k), ek).max() <= 1
    assert_decode_close(got, want, "window + fused append")
    # shapes the tcgen05 kernel does not take, and bad arguments
    for D2, G2, Hkv2 in [(64, 4, 8), (128, 16, 8), (128, 4, 4)]:
        k2, v2, q2, bt2 = _decode_case(D2, G2, dt, [40], Hkv=Hkv2, L=2, seed=78)
        with pytest.raises(K.KvinjError) as e:
            _run_window(k2, v2, q2, bt2, np.array([40], np.int32), 8, dt, theta, 64)
        assert e.value.code == K.KVINJ_EUNSUPPORTED
    with pytest.raises(K.KvinjError) as e:
        _run_window(kc, vc, q, bt, ctx, -1, dt, theta, int(ctx.max()) + 4)
    assert e.value.code == K.KVINJ_EINVAL


# ---------------------------------------------------------------------------
# paged prefill of query tokens
# ---------------------------------------------------------------------------
def _prefill_case(D, G, dt, mem, nq, Hkv, seed):
    # requests of mem[r] memory tokens then nq[r] query tokens, all already in the cache;
    # the query tokens of the requests interleaved in the token list
    ctx = [m + n for m, n in zip(mem, nq)]
    kc, vc, _, bt = _decode_case(D, G, dt, ctx, Hkv=Hkv, L=2, seed=seed)
    toks = [(r, mem[r] + i) for i in range(max(nq)) for r in range(len(mem)) if i < nq[r]]
    seq = np.array([t[0] for t in toks], np.int32)
    pos = np.array([t[1] for t in toks], np.int32)
    q = gen_bits(seed + 9, (len(toks), Hkv * G, D), dt)
    return kc, vc, bt, seq, pos, q


def _prefill_grouped(D, G, dt, mem, nq, Hkv, seed, runs=0):
    # as _prefill_case, with each request's query tokens consecutive in the token list, or
    # (runs > 0) cut into runs of `runs` tokens, the runs of the requests interleaved
    ctx = [m + n for m, n in zip(mem, nq)]
    kc, vc, _, bt = _decode_case(D, G, dt, ctx, Hkv=Hkv, L=2, seed=seed)
    per = [[(r, mem[r] + i) for i in range(nq[r])] for r in range(len(mem))]
    if runs:
        parts = [[p[i:i + runs] for i in range(0, len(p), runs)] for p in per]
        toks = [t for k in range(max(len(c) for c in parts)) for c in parts if k < len(c)
                for t in c[k]]
    else:
        toks = [t for p in per for t in p]
    seq = np.array([t[0] for t in toks], np.int32)
    pos = np.array([t[1] for t in toks], np.int32)
    q = gen_bits(seed + 9, (len(toks), Hkv * G, D), dt)
    return kc, vc, bt, seq, pos, q


def _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, rope_max, status=None, scale=0.0):
    tdt = torch_dtype(dt)
    D = kc.shape[-1]
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(theta, D, rope_max)
    n, Hq, _ = q.shape
    ws = K.make_prefill_workspace(n, Hq, kc.shape[2], D, bt.shape[1])
    out = torch.full((n, Hq, D), float("nan"), dtype=tdt, device="cuda")
    K.kvinj_paged_prefill(cache, rope, 1, from_bits(q, tdt), i32(seq), i32(pos), i32(bt), out, ws,
                          scale=scale, status=status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("D,G,Hkv", [(128, 4, 8), (128, 8, 8), (128, 1, 16), (64, 2, 4)])
def test_paged_prefill_matches_oracle(D, G, Hkv):
    dt, theta = W.BF16, 5e5
    mem, nq = [40, 300, 7], [5, 17, 9]
    kc, vc, bt, seq, pos, q = _prefill_case(D, G, dt, mem, nq, Hkv, seed=80 + G)
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 400, status=status)
    assert status.item() == 0
    want, st = oracle.paged_prefill(kc, vc, 1, q, seq, pos, bt, theta, dt)
    assert st == 0
    assert_decode_close(got, want, f"prefill D{D} G{G} Hkv{Hkv}")


def test_paged_prefill_more_tokens_than_a_launch_and_bad_tokens():
    # 1300 query tokens: two launches of rows; a token with a request id outside the batch
    # or a position past the table gives a zero row and a status bit, its neighbours are
    # unaffected
    D, G, dt, Hkv, theta = 128, 4, W.BF16, 8, 5e5
    mem, nq = [20, 3], [700, 600]
    kc, vc, bt, seq, pos, q = _prefill_case(D, G, dt, mem, nq, Hkv, seed=91)
    seq, pos = seq.copy(), pos.copy()
    seq[5] = 7
    pos[9] = 10 ** 6
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 1000, status=status)
    assert status.item() & K.ST_BAD_SEQ and status.item() & K.ST_BAD_POS
    assert not got[5].any() and not got[9].any()
    keep = np.setdiff1d(np.arange(seq.size), [5, 9])
    want, st = oracle.paged_prefill(kc, vc, 1, q[keep], seq[keep], pos[keep], bt, theta, dt,
                                    n_threads=16)
    assert st == 0
    assert_decode_close(got[keep], want, "prefill over two launches")


@pytest.mark.parametrize("dt", [W.BF16, W.FP16])
@pytest.mark.parametrize("G,Hkv", [(1, 8), (2, 8), (4, 8), (8, 8), (4, 16)])
def test_paged_prefill_tiles_match_oracle(G, Hkv, dt):
    # consecutive query tokens of a request share tiles of 128 / G tokens (70 tokens: several
    # tiles, the last one ragged); contexts up to 4070 tokens stream 32 chunks of 128 keys per
    # tile and kv head, split over the CTAs (cut segments are merged by the combine pass);
    # a 1-token request and a 3-token memory
    D, theta = 128, 5e5
    mem, nq = [2900, 640, 100, 4000, 3], [40, 17, 5, 70, 1]
    kc, vc, bt, seq, pos, q = _prefill_grouped(D, G, dt, mem, nq, Hkv, seed=300 + 7 * G + Hkv)
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 4200, status=status)
    assert status.item() == 0
    want, st = oracle.paged_prefill(kc, vc, 1, q, seq, pos, bt, theta, dt, n_threads=16)
    assert st == 0
    assert_decode_close(got, want, f"prefill tiles G{G} Hkv{Hkv} dt{dt}")


@pytest.mark.parametrize("scale", [0.5, 2.0])
def test_paged_prefill_large_logits(scale):
    # logits 5.7x and 23x the default scale: the running maximum moves within and across
    # chunks, and the hi + lo parts of q and P carry the precision
    D, G, Hkv, dt, theta = 128, 8, 8, W.BF16, 5e5
    mem, nq = [1500, 260], [16, 16]
    kc, vc, bt, seq, pos, q = _prefill_grouped(D, G, dt, mem, nq, Hkv, seed=330)
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 2000, status=status, scale=scale)
    assert status.item() == 0
    want, st = oracle.paged_prefill(kc, vc, 1, q, seq, pos, bt, theta, dt, scale=scale,
                                    n_threads=16)
    assert st == 0
    assert_decode_close(got, want, f"prefill scale {scale}")


def test_paged_prefill_runs_bad_block_and_determinism():
    # each request's tokens in runs of 5 interleaved with the others' (tiles never span two
    # runs); request 1's table points page 10 outside the cache: its rows are flagged, the
    # other requests' rows are unaffected; a second call gives the same bits
    D, G, Hkv, dt, theta = 128, 4, 8, W.BF16, 5e5
    mem, nq = [700, 1200, 300], [33, 21, 12]
    kc, vc, bt, seq, pos, q = _prefill_grouped(D, G, dt, mem, nq, Hkv, seed=340, runs=5)
    bt = bt.copy()
    bt[1, 10] = 10 ** 6
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 1600, status=status)
    assert status.item() == K.ST_BAD_BLOCK
    keep = seq != 1
    want, st = oracle.paged_prefill(kc, vc, 1, q[keep], seq[keep], pos[keep], bt, theta, dt,
                                    n_threads=16)
    assert st == 0
    assert_decode_close(got[keep], want, "prefill runs")
    again = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 1600)
    assert np.array_equal(got, again, equal_nan=True)


def test_paged_prefill_many_pieces_per_cta():
    # 1300 query tokens listed request by request: full tiles of 32 tokens (every row
    # live), several pieces per CTA, so every piece transition -- the last PV of one piece,
    # the next piece's query rows, the combine of cut segments -- runs many times
    D, G, Hkv, dt, theta = 128, 4, 8, W.BF16, 5e5
    kc, vc, bt, seq, pos, q = _prefill_grouped(D, G, dt, [20, 3], [700, 600], Hkv, seed=92)
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 1000, status=status)
    assert status.item() == 0
    want, st = oracle.paged_prefill(kc, vc, 1, q, seq, pos, bt, theta, dt, n_threads=16)
    assert st == 0
    assert_decode_close(got, want, "prefill, many pieces per CTA")


def test_paged_prefill_ignores_nan_rows_past_the_context():
    # every cache row that no query token may attend to -- slots past each request's last
    # token, blocks of no request -- holds NaN bit patterns; request 1's first page of its
    # second chunk points outside the cache (its copy then comes from block 0, NaN too)
    D, G, Hkv, dt, theta = 128, 4, 8, W.BF16, 5e5
    mem, nq = [300, 500, 37], [20, 9, 3]
    kc, vc, bt, seq, pos, q = _prefill_grouped(D, G, dt, mem, nq, Hkv, seed=360)
    ctx = np.array([m + n for m, n in zip(mem, nq)])
    used = np.zeros(kc.shape[1:3] + (16,), bool)[:, 0]  # [NB][16] slots holding a token
    for r, c in enumerate(ctx):
        for t in range(c):
            used[bt[r, t // 16], t % 16] = True
    nan = 0x7FC0
    kc, vc = kc.copy(), vc.copy()
    nb, slot = np.nonzero(~used)
    kc[:, nb, :, slot, :] = nan
    vc[:, nb, :, slot, :] = nan
    bad = bt.copy()
    bad[1, 8] = -5
    status = status_tensor()
    got = _run_prefill(kc, vc, bad, seq, pos, q, dt, theta, 600, status=status)
    assert status.item() == K.ST_BAD_BLOCK
    assert np.isfinite(got).all()
    keep = seq != 1
    want, st = oracle.paged_prefill(kc, vc, 1, q[keep], seq[keep], pos[keep], bt, theta, dt,
                                    n_threads=16)
    assert st == 0
    assert_decode_close(got[keep], want, "prefill with NaN rows outside the contexts")


def test_paged_prefill_all_tokens_invalid():
    # no valid token: every row zero, no tile, no unit; the tensor-core pass does nothing
    D, G, Hkv, dt, theta = 128, 4, 8, W.BF16, 5e5
    kc, vc, bt, seq, pos, q = _prefill_grouped(D, G, dt, [50, 20], [3, 2], Hkv, seed=350)
    seq = np.array([5, -1, 2, 9, 7], np.int32)
    status = status_tensor()
    got = _run_prefill(kc, vc, bt, seq, pos, q, dt, theta, 100, status=status)
    assert status.item() & K.ST_BAD_SEQ
    assert not got.any()


# ---------------------------------------------------------------------------
# append + decode in one call
# ---------------------------------------------------------------------------
def _fused_case(D, G, dt, ctx, Hkv, seed, rotate=True):
    kc, vc, q, bt = _decode_case(D, G, dt, ctx, Hkv=Hkv, L=2, seed=seed)
    batch = len(ctx)
    kn = gen_bits(seed + 5, (batch, Hkv, D), dt)
    vn = gen_bits(seed + 6, (batch, Hkv, D), dt)
    ctx = np.asarray(ctx, np.int32)
    pos = ctx - 1  # the new token is the newest one of the context
    slots = bt[np.arange(batch), pos // 16].astype(np.int64) * 16 + pos % 16
    theta = 5e5
    ek, ev = kc.copy(), vc.copy()
    oracle.append(ek, ev, 1, kn, vn, pos, slots, theta, dt, rotate=rotate)
    want, st = oracle.paged_decode(ek, ev, 1, q, pos, bt, ctx, theta, dt, rotate_q=rotate)
    assert st == 0
    return kc, vc, q, bt, kn, vn, ctx, pos, slots, theta, ek, ev, want


def _run_fused(kc, vc, q, bt, kn, vn, ctx, pos, dt, theta, variant, ctas, rotate=True,
               status=None):
    tdt = torch_dtype(dt)
    D = kc.shape[-1]
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(theta, D, int(ctx.max()) + 4) if rotate else None
    batch, Hq, _ = q.shape
    ws = K.make_decode_workspace(batch, Hq, kc.shape[2], D)
    out = torch.full((batch, Hq, D), float("nan"), dtype=tdt, device="cuda")
    K.kvinj_append_paged_decode(cache, rope, 1, from_bits(q, tdt), from_bits(kn, tdt),
                                from_bits(vn, tdt), i32(pos), i32(bt), i32(ctx), out, ws, 0.0,
                                status, None, variant, ctas)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), bits(cache.k), bits(cache.v)


@pytest.mark.parametrize("variant", [1, 2, 3])
@pytest.mark.parametrize("ctas", [0, 1, 5, 37])
@pytest.mark.parametrize("G,Hkv", [(4, 8), (1, 16), (8, 8)])
def test_append_paged_decode_matches_oracle(variant, ctas, G, Hkv):
    D, dt = 128, W.BF16
    ctx = [1, 16, 17, 250, 611, 33]
    kc, vc, q, bt, kn, vn, ctx, pos, slots, theta, ek, ev, want = _fused_case(
        D, G, dt, ctx, Hkv, seed=90 + G + Hkv)
    status = status_tensor()
    got, gk, gv = _run_fused(kc, vc, q, bt, kn, vn, ctx, pos, dt, theta, variant, ctas,
                             status=status)
    assert status.item() == 0
    assert np.array_equal(gv, ev)
    assert ulp_distance(gk, ek).max() <= 1
    assert_decode_close(got, want, f"fused variant{variant} ctas{ctas} G{G} Hkv{Hkv}")


@pytest.mark.parametrize("G", [4, 8])
def test_append_paged_decode_equals_separate_calls_bitwise(G):
    D, dt, Hkv = 128, W.BF16, 8
    ctx = [700, 33, 1500, 16, 2048, 5]
    kc, vc, q, bt, kn, vn, ctx, pos, slots, theta, ek, ev, want = _fused_case(
        D, G, dt, ctx, Hkv, seed=97)
    got, gk, gv = _run_fused(kc, vc, q, bt, kn, vn, ctx, pos, dt, theta, 3, 0)
    tdt = torch_dtype(dt)
    cache = K.Cache(from_bits(kc, tdt), from_bits(vc, tdt))
    rope = K.make_rope(theta, D, int(ctx.max()) + 4)
    K.kvinj_append(cache, rope, 1, from_bits(kn, tdt), from_bits(vn, tdt), i32(pos),
                   torch.from_numpy(slots).cuda())
    ws = K.make_decode_workspace(len(ctx), Hkv * G, Hkv, D)
    out = torch.empty((len(ctx), Hkv * G, D), dtype=tdt, device="cuda")
    K.kvinj_paged_decode_ex(cache, rope, 1, from_bits(q, tdt), i32(pos), i32(bt), i32(ctx), out,
                            ws, 0.0, None, None, 3, 0)
    torch.cuda.synchronize()
    assert np.array_equal(bits(cache.k), gk) and np.array_equal(bits(cache.v), gv)
    assert np.array_equal(out.float().cpu().numpy().astype(np.float64), got)


@pytest.mark.parametrize("variant", [2, 3])
def test_append_paged_decode_unrotated_and_bad_block(variant):
    D, G, dt, Hkv = 128, 4, W.BF16, 8
    ctx = [40, 300, 17]
    kc, vc, q, bt, kn, vn, ctx, pos, slots, theta, ek, ev, want = _fused_case(
        D, G, dt, ctx, Hkv, seed=98, rotate=False)
    got, gk, gv = _run_fused(kc, vc, q, bt, kn, vn, ctx, pos, dt, theta, variant, 0, rotate=False)
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)
    assert_decode_close(got, want, f"fused unrotated variant{variant}")
    # the new token's page outside the cache: flagged, other requests intact
    bt2 = bt.copy()
    bt2[0, pos[0] // 16] = kc.shape[1] + 3
    status = status_tensor()
    got, gk, gv = _run_fused(kc, vc, q, bt2, kn, vn, ctx, pos, dt, theta, variant, 0,
                             rotate=False, status=status)
    assert status.item() & K.ST_BAD_BLOCK
    assert_decode_close(got[1:], want[1:], f"fused bad block variant{variant}")
