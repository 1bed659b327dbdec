"""int8 KV cache on the GPU ("Latency Optimization > KV Cache Management", KV
cache quantization) against the fp64 oracle, through the C ABI:

- inject and append store, for every written row, the oracle's codes and scale
  bit for bit: keys rotated and rounded once to 16 bits as the oracle's fp64
  rotation is, then quantized as orc_quantize_rows_i8 does (values: quantized
  as stored); rows not written keep their sentinels;
- paged decode over an int8 cache matches orc_paged_decode_i8 within the
  decode tolerance, for G 1/2/4/8, bf16 and fp16 queries, cut segments (1, 5
  and 37 CTAs and the default grid), ragged tails, rows past the context that
  hold garbage codes and NaN scales, invalid contexts and blocks;
- the fused append writes the oracle's codes and scales and is attended to.

Caches for the decode tests are built from the oracle's own quantization of
seeded 16-bit rows; no expectation comes from the CUDA path."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from paged_kv_cache_inject_gb300 import kvinj as K
from tests.gpu_helpers import assert_decode_close, bits, from_bits, torch_dtype, ulp_distance

pytestmark = pytest.mark.gpu

SENT_CODE = 0x5A
SENT_SCALE = -7.25


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


def dev_cache(kq, ks, vq, vs):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return K.CacheI8(t(kq), t(vq), t(ks), t(vs))


def sentinel_cache(L, NB, Hkv, D=128, B=16):
    kq = np.full((L, NB, Hkv, B, D), SENT_CODE, np.int8)
    ks = np.full((L, NB, Hkv, B), SENT_SCALE, np.float32)
    return kq, ks, kq.copy(), ks.copy()


def host(cache: K.CacheI8):
    return (cache.k.cpu().numpy(), cache.k_scale.cpu().numpy(), cache.v.cpu().numpy(),
            cache.v_scale.cpu().numpy())


def expected_rows(kc16, vc16, dt, written):
    """The oracle's codes and scales of the written rows of 16-bit caches."""
    kq, ks = oracle.quantize_rows_i8(kc16[written], dt)
    vq, vs = oracle.quantize_rows_i8(vc16[written], dt)
    return kq, ks, vq, vs


# ---------------------------------------------------------------------------
# inject / append
# ---------------------------------------------------------------------------
def _inject_case(dt, seed, L=2, Hkv=8, c=32, n_chunks=9, NB=70):
    rng = np.random.default_rng(seed)
    D, B = 128, 16
    pool = gen_bits(seed, (n_chunks, L, 2, c, Hkv, D), dt)
    bt = rng.permutation(NB).astype(np.int32)[:64].reshape(2, 32)
    ids = np.array([3, 0, 8, 3, 5], np.int32)
    req = np.array([0, 0, 1, 1, 1], np.int32)
    start = np.array([0, 45, 7, 130, 480], np.int32)  # straddling blocks, ending the table
    seq = np.repeat(req, c).astype(np.int32)
    pos = (start[:, None] + np.arange(c)).reshape(-1).astype(np.int32)
    slots, st = oracle.slot_mapping(bt, seq, pos, B, NB)
    assert st == 0
    return dict(L=L, Hkv=Hkv, c=c, NB=NB, pool=pool, bt=bt, ids=ids, start=start, seq=seq,
                pos=pos, slots=slots)


@pytest.mark.parametrize("dt", [W.BF16, W.FP16])
def test_inject_i8_codes_and_scales_bit_exact(dt):
    cs = _inject_case(dt, seed=21 + dt)
    L, Hkv, NB = cs["L"], cs["Hkv"], cs["NB"]
    tdt = torch_dtype(dt)
    theta = 5e5
    # the oracle's 16-bit inject (keys rotated, rounded once), then its quantization
    SENT16 = 0x7FC1
    kc16 = np.full((L, NB, Hkv, 16, 128), SENT16, np.uint16)
    vc16 = kc16.copy()
    assert oracle.inject(cs["pool"], cs["ids"], cs["start"], cs["slots"], theta, dt, kc16,
                         vc16) == 0
    written = (kc16 != SENT16).any(axis=-1)
    ekq, eks, evq, evs = expected_rows(kc16, vc16, dt, written)

    cache = dev_cache(*sentinel_cache(L, NB, Hkv))
    pool = K.Pool(from_bits(cs["pool"], tdt))
    rope = K.make_rope(theta, 128, 600)
    status = status_tensor()
    slots = torch.from_numpy(cs["slots"]).cuda()
    K.kvinj_inject_i8(pool, cache, rope, i32(cs["ids"]), i32(cs["start"]), slots, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kq, ks, vq, vs = host(cache)
    assert np.array_equal(kq[written], ekq) and np.array_equal(ks[written], eks)
    assert np.array_equal(vq[written], evq) and np.array_equal(vs[written], evs)
    assert (kq[~written] == SENT_CODE).all() and (ks[~written] == SENT_SCALE).all()
    assert (vq[~written] == SENT_CODE).all() and (vs[~written] == SENT_SCALE).all()

    # the rows include keys whose fast rotation lands within its error of a 16-bit rounding
    # boundary: the 16-bit inject (fast rotation only) is one ulp off there, the int8 inject
    # still stores the oracle's codes
    c16 = K.Cache(from_bits(np.full_like(kc16, SENT16), tdt), from_bits(np.full_like(kc16, SENT16), tdt))
    K.kvinj_inject(pool, c16, rope, i32(cs["ids"]), i32(cs["start"]), slots, status=status)
    torch.cuda.synchronize()
    off = ulp_distance(bits(c16.k), kc16) > 0
    assert off.any(), "no key near a rounding boundary in this case: enlarge it"


@pytest.mark.parametrize("dt,rotate", [(W.BF16, True), (W.FP16, True), (W.BF16, False)])
def test_append_i8_codes_and_scales_bit_exact(dt, rotate):
    rng = np.random.default_rng(33)
    L, NB, Hkv, n = 2, 40, 8, 300
    tdt = torch_dtype(dt)
    theta = 1e4
    kn = gen_bits(34, (n, Hkv, 128), dt)
    vn = gen_bits(35, (n, Hkv, 128), dt)
    slots = rng.permutation(NB * 16)[:n].astype(np.int64)
    pos = rng.integers(0, 9000, n).astype(np.int32)
    SENT16 = 0x7FC1
    kc16 = np.full((L, NB, Hkv, 16, 128), SENT16, np.uint16)
    vc16 = kc16.copy()
    assert oracle.append(kc16, vc16, 1, kn, vn, pos, slots, theta, dt, rotate=rotate) == 0
    written = (kc16 != SENT16).any(axis=-1)
    ekq, eks, evq, evs = expected_rows(kc16, vc16, dt, written)
    cache = dev_cache(*sentinel_cache(L, NB, Hkv))
    rope = K.make_rope(theta, 128, 9000) if rotate else None
    status = status_tensor()
    K.kvinj_append_i8(cache, rope, 1, from_bits(kn, tdt), from_bits(vn, tdt), i32(pos),
                      torch.from_numpy(slots).cuda(), status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    kq, ks, vq, vs = host(cache)
    assert np.array_equal(kq[written], ekq) and np.array_equal(ks[written], eks)
    assert np.array_equal(vq[written], evq) and np.array_equal(vs[written], evs)
    assert (kq[~written] == SENT_CODE).all() and (vs[~written] == SENT_SCALE).all()


def test_inject_i8_refusals_and_bad_indices():
    cs = _inject_case(W.BF16, seed=40)
    L, Hkv, NB = cs["L"], cs["Hkv"], cs["NB"]
    cache = dev_cache(*sentinel_cache(L, NB, Hkv))
    pool = K.Pool(from_bits(cs["pool"], torch.bfloat16))
    rope = K.make_rope(5e5, 128, 600)
    slots = torch.from_numpy(cs["slots"]).cuda()
    # no fp64 table: refused
    bare = K.Rope(rope.table, 128)
    with pytest.raises(K.KvinjError) as e:
        K.kvinj_inject_i8(pool, cache, bare, i32(cs["ids"]), i32(cs["start"]), slots)
    assert e.value.code == K.KVINJ_EINVAL
    # a chunk id outside the pool and a position beyond the table: skipped and flagged
    ids = cs["ids"].copy()
    ids[1] = 99
    start = cs["start"].copy()
    start[4] = 590
    status = status_tensor()
    K.kvinj_inject_i8(pool, cache, rope, i32(ids), i32(start), slots, status=status)
    torch.cuda.synchronize()
    assert status.item() & K.ST_BAD_CHUNK and status.item() & K.ST_BAD_POS
    kq = cache.k.cpu().numpy()
    c = cs["c"]
    s1 = cs["slots"][c:2 * c]  # chunk 1's slots stay untouched
    assert (kq[:, s1 // 16, :, s1 % 16] == SENT_CODE).all()


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------
def _decode_i8_case(G, dt, ctx, Hkv=8, L=2, seed=50, spare=3):
    """An int8 cache quantized by the oracle from seeded 16-bit rows; the rows past each
    context in its last block hold garbage codes and NaN scales."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    pages = -(-ctx // 16)
    NB = int(pages.sum()) + spare
    max_blocks = int(pages.max()) + 2
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((ctx.size, max_blocks), -1, np.int32)
    o = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[o:o + p]
        o += p
    k16 = gen_bits(seed, (L, NB, Hkv, 16, 128), dt)
    v16 = gen_bits(seed + 1, (L, NB, Hkv, 16, 128), dt)
    kq, ks = oracle.quantize_rows_i8(k16, dt)
    vq, vs = oracle.quantize_rows_i8(v16, dt)
    for r, c in enumerate(ctx):
        if c % 16:
            blk = bt[r, c // 16]
            kq[:, blk, :, c % 16:] = rng.integers(-128, 128, kq[:, blk, :, c % 16:].shape)
            vq[:, blk, :, c % 16:] = rng.integers(-128, 128, vq[:, blk, :, c % 16:].shape)
            ks[:, blk, :, c % 16:] = np.nan
            vs[:, blk, :, c % 16:] = np.nan
    q = gen_bits(seed + 2, (ctx.size, Hkv * G, 128), dt)
    return kq, ks, vq, vs, q, bt, ctx


def _run_decode_i8(kq, ks, vq, vs, q, bt, ctx, q_pos, dt, theta, rope_max, ctas=0, layer=1,
                   kn=None, vn=None, status=None, rotate=True):
    tdt = torch_dtype(dt)
    cache = dev_cache(kq, ks, vq, vs)
    rope = K.make_rope(theta, 128, rope_max) if rotate else None
    batch, Hq, _ = q.shape
    ws = K.make_decode_workspace(batch, Hq, kq.shape[2], 128)
    out = torch.full((batch, Hq, 128), float("nan"), dtype=tdt, device="cuda")
    K.kvinj_paged_decode_i8(cache, rope, layer, from_bits(q, tdt), i32(q_pos), i32(bt), i32(ctx),
                            out, ws, k_new=None if kn is None else from_bits(kn, tdt),
                            v_new=None if vn is None else from_bits(vn, tdt), status=status,
                            ctas=ctas)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), cache


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("dt", [W.BF16, W.FP16])
@pytest.mark.parametrize("ctas", [0, 1, 5, 37])
def test_decode_i8_matches_oracle(G, dt, ctas):
    ctx = [1, 16, 17, 250, 611, 33, 1000]
    kq, ks, vq, vs, q, bt, ctx = _decode_i8_case(G, dt, ctx, seed=50 + G + 10 * dt)
    theta = 5e5
    q_pos = ctx - 1
    want, st = oracle.paged_decode_i8(kq, ks, vq, vs, 1, q, q_pos, bt, ctx, theta, dt)
    assert st == 0
    status = status_tensor()
    got, _ = _run_decode_i8(kq, ks, vq, vs, q, bt, ctx, q_pos, dt, theta, int(ctx.max()) + 4,
                            ctas=ctas, status=status)
    assert status.item() == 0
    assert_decode_close(got, want, f"int8 decode G{G} dt{dt} ctas{ctas}")


@pytest.mark.parametrize("G,Hkv", [(4, 16), (8, 8), (1, 8)])
def test_decode_i8_long_contexts_and_unrotated_query(G, Hkv):
    ctx = [4100, 9000, 2, 3333]
    kq, ks, vq, vs, q, bt, ctx = _decode_i8_case(G, W.BF16, ctx, Hkv=Hkv, seed=70 + G)
    want, st = oracle.paged_decode_i8(kq, ks, vq, vs, 0, q, ctx - 1, bt, ctx, 1e4, W.BF16,
                                      rotate_q=False)
    assert st == 0
    got, _ = _run_decode_i8(kq, ks, vq, vs, q, bt, ctx, ctx - 1, W.BF16, 1e4, 10, layer=0,
                            rotate=False)
    assert_decode_close(got, want, f"int8 decode long G{G}")


@pytest.mark.parametrize("G", [4, 8])
def test_decode_i8_invalid_context_and_block(G):
    ctx = [300, 0, 77, 5000]
    kq, ks, vq, vs, q, bt, ctx = _decode_i8_case(G, W.BF16, [300, 1, 77, 5000], seed=80 + G)
    ctx = np.array([300, 0, 77, 5000], np.int32)
    bad_bt = bt.copy()
    bad_bt[2, 3] = 10 ** 6  # a block outside the cache: its tokens are masked
    theta = 5e5
    status = status_tensor()
    got, _ = _run_decode_i8(kq, ks, vq, vs, q, bad_bt, ctx, np.maximum(ctx - 1, 0), W.BF16,
                            theta, 5010, status=status)
    st = status.item()
    assert st & K.ST_BAD_CTX and st & K.ST_BAD_BLOCK
    assert np.all(got[1] == 0.0)  # invalid context: zero output
    # the request with the bad block: attention over its other tokens
    keep = np.ones(int(ctx[2]), bool)
    keep[48:64] = False
    kr = np.stack([kq[1, bt[2, p // 16], :, p % 16] for p in np.nonzero(keep)[0]], 1)
    vr = np.stack([vq[1, bt[2, p // 16], :, p % 16] for p in np.nonzero(keep)[0]], 1)
    ksr = np.stack([ks[1, bt[2, p // 16], :, p % 16] for p in np.nonzero(keep)[0]], 1)
    vsr = np.stack([vs[1, bt[2, p // 16], :, p % 16] for p in np.nonzero(keep)[0]], 1)
    n = kr.shape[1]
    # contiguous single-request cache holding only the kept tokens, as a block table over them
    pages = -(-n // 16)
    kc = np.zeros((2, pages, kq.shape[2], 16, 128), np.int8)
    vc = np.zeros_like(kc)
    ksc = np.zeros((2, pages, kq.shape[2], 16), np.float32)
    vsc = np.zeros_like(ksc)
    for j in range(n):
        kc[1, j // 16, :, j % 16] = kr[:, j]
        vc[1, j // 16, :, j % 16] = vr[:, j]
        ksc[1, j // 16, :, j % 16] = ksr[:, j]
        vsc[1, j // 16, :, j % 16] = vsr[:, j]
    want2, st2 = oracle.paged_decode_i8(kc, ksc, vc, vsc, 1, q[2:3], np.array([ctx[2] - 1]),
                                        np.arange(pages, dtype=np.int32)[None], np.array([n]),
                                        theta, W.BF16)
    assert st2 == 0
    assert_decode_close(got[2:3], want2, "int8 decode with a masked block")
    # the other requests are unaffected
    want, _ = oracle.paged_decode_i8(kq, ks, vq, vs, 1, q[[0, 3]], ctx[[0, 3]] - 1, bt[[0, 3]],
                                     ctx[[0, 3]], theta, W.BF16)
    assert_decode_close(got[[0, 3]], want, "int8 decode beside invalid requests")


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("ctas", [0, 5, 37])
def test_decode_i8_fused_append_matches_oracle(G, ctas):
    dt = W.BF16
    ctx = [1, 16, 17, 250, 611, 33]
    kq, ks, vq, vs, q, bt, ctx = _decode_i8_case(G, dt, ctx, seed=90 + G)
    batch, Hkv = len(ctx), kq.shape[2]
    kn = gen_bits(95 + G, (batch, Hkv, 128), dt)
    vn = gen_bits(96 + G, (batch, Hkv, 128), dt)
    pos = ctx - 1
    theta = 5e5
    # the oracle's codes of the appended rows (key rotated at its position, rounded once)
    k_rot = oracle.rope_round_rows(kn.reshape(-1, 128), np.repeat(pos, Hkv), theta, dt)
    akq, aks = oracle.quantize_rows_i8(k_rot, dt)
    avq, avs = oracle.quantize_rows_i8(vn.reshape(-1, 128), dt)
    ekq, eks, evq, evs = kq.copy(), ks.copy(), vq.copy(), vs.copy()
    for r in range(batch):
        blk, off = bt[r, pos[r] // 16], pos[r] % 16
        ekq[1, blk, :, off] = akq[r * Hkv:(r + 1) * Hkv]
        eks[1, blk, :, off] = aks[r * Hkv:(r + 1) * Hkv]
        evq[1, blk, :, off] = avq[r * Hkv:(r + 1) * Hkv]
        evs[1, blk, :, off] = avs[r * Hkv:(r + 1) * Hkv]
    want, st = oracle.paged_decode_i8(ekq, eks, evq, evs, 1, q, pos, bt, ctx, theta, dt)
    assert st == 0
    status = status_tensor()
    got, cache = _run_decode_i8(kq, ks, vq, vs, q, bt, ctx, pos, dt, theta, int(ctx.max()) + 4,
                                ctas=ctas, kn=kn, vn=vn, status=status)
    assert status.item() == 0
    gkq, gks, gvq, gvs = host(cache)
    for r in range(batch):
        blk, off = bt[r, pos[r] // 16], pos[r] % 16
        assert np.array_equal(gkq[1, blk, :, off], ekq[1, blk, :, off])
        assert np.array_equal(gks[1, blk, :, off], eks[1, blk, :, off])
        assert np.array_equal(gvq[1, blk, :, off], evq[1, blk, :, off])
        assert np.array_equal(gvs[1, blk, :, off], evs[1, blk, :, off])
    assert_decode_close(got, want, f"int8 fused append G{G} ctas{ctas}")


def test_decode_i8_refusals():
    kq, ks, vq, vs, q, bt, ctx = _decode_i8_case(4, W.BF16, [40, 50], Hkv=8, seed=99)
    cache = dev_cache(kq, ks, vq, vs)
    rope = K.make_rope(5e5, 128, 60)
    qd = from_bits(q, torch.bfloat16)
    out = torch.empty_like(qd)
    ws = K.make_decode_workspace(2, 32, 8, 128)
    # a fused append needs the fp64 table
    with pytest.raises(K.KvinjError) as e:
        K.kvinj_paged_decode_i8(cache, K.Rope(rope.table, 128), 1, qd, i32(ctx - 1), i32(bt),
                                i32(ctx), out, ws, k_new=qd[:, :8], v_new=qd[:, :8])
    assert e.value.code == K.KVINJ_EINVAL
    # kv heads not a multiple of 8: no kernel
    kq4, ks4, vq4, vs4, q4, bt4, _ = _decode_i8_case(4, W.BF16, [40, 50], Hkv=4, seed=98)
    q4d = from_bits(q4, torch.bfloat16)
    with pytest.raises(K.KvinjError) as e:
        K.kvinj_paged_decode_i8(dev_cache(kq4, ks4, vq4, vs4), rope, 1, q4d, i32(ctx - 1),
                                i32(bt4), i32(ctx), torch.empty_like(q4d),
                                K.make_decode_workspace(2, 16, 4, 128))
    assert e.value.code == K.KVINJ_EUNSUPPORTED
