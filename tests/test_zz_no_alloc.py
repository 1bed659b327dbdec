"""kvinj_paged_decode_static: paged decode for callers that cannot allocate.

Some callers cannot hand the library a workspace: code running inside an
engine hook or plugin that must not call cudaMalloc, or in a process whose
device memory is already handed out. This entry point keeps its scratch in a
fixed device array of the library instead. It runs the same kernels as the
workspace entry point, so on the same inputs its output must be the same bit
for bit, call after call: the array keeps the previous call's contents, and
none of them may leak into the next result. The calls run from the largest
shape the array admits down to smaller ones, so a smaller call always finds
the partial states of a larger one under it.
The file sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
from paged_kv_cache_inject_gb300 import kvinj as K
from tests.gpu_helpers import assert_decode_close, bits, from_bits

pytestmark = pytest.mark.gpu

THETA, MAX_POS = 5e5, 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()


def _case(seed, ctx, Hkv=8, G=4, D=128, L=2):
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx, np.int32)
    pages = -(-ctx // 16)
    NB = int(pages.sum()) + 5
    max_blocks = int(pages.max()) + 1
    perm = rng.permutation(NB).astype(np.int32)
    bt = np.full((ctx.size, max_blocks), -1, np.int32)
    o = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[o:o + p]
        o += p
    key = W.stream_key(seed, W.STREAM_POOL)

    def gen(shape, off):
        n = int(np.prod(shape))
        return W.normal_bits(key, off + np.arange(n, dtype=np.uint64), W.BF16).reshape(shape)

    host = {"k": gen((L, NB, Hkv, 16, D), 0), "v": gen((L, NB, Hkv, 16, D), 1 << 32),
            "q": gen((ctx.size, Hkv * G, D), 1 << 33), "bt": bt, "ctx": ctx}
    cache = K.Cache(from_bits(host["k"], torch.bfloat16), from_bits(host["v"], torch.bfloat16))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return (cache, from_bits(host["q"], torch.bfloat16), dev(ctx - 1), dev(bt), dev(ctx)), host


def _static_and_workspace(case, rope, layer=1):
    cache, q, q_pos, bt, ctx = case
    batch, Hq, D = q.shape
    need = K.kvinj_decode_workspace_size(batch, Hq, cache.num_kv_heads, D)
    assert need <= K.KVINJ_STATIC_SCRATCH_BYTES, "the case must fit the fixed array"
    ref = torch.empty_like(q)
    ws = K.make_decode_workspace(batch, Hq, cache.num_kv_heads, D)
    K.kvinj_paged_decode(cache, rope, layer, q, q_pos, bt, ctx, ref, ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = torch.full_like(q, float("nan"))
    K.kvinj_paged_decode_static(cache, rope, layer, q, q_pos, bt, ctx, got, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return got, ref


def test_static_scratch_matches_workspace_entry_point_call_after_call():
    rope = K.make_rope(THETA, 128, MAX_POS)
    # largest shape the array admits on this GPU first (64 q / 8 kv heads: G = 8, about
    # 19 MiB of partial states on 152 SMs), then smaller ones over its leftovers
    cases = [
        _case(30, [4000, 33, 2500, 16, 3000, 5, 1024, 700], Hkv=8, G=8),
        _case(31, [700, 33, 1500, 16, 2048, 5]),
        _case(32, [100, 3000, 17, 900], G=1),
        _case(33, [2049, 1, 640], Hkv=8, G=8),
    ]
    for i, (case, host) in enumerate(cases):
        got, ref = _static_and_workspace(case, rope)
        assert np.array_equal(bits(got), bits(ref)), f"case {i}: static != workspace, bitwise"
        if i == 1:
            # and one of them against the fp64 oracle, at the decode tolerance
            want, st = oracle.paged_decode(host["k"], host["v"], 1, host["q"], host["ctx"] - 1,
                                           host["bt"], host["ctx"], THETA, W.BF16)
            assert st == 0
            assert_decode_close(got.float().cpu().numpy().astype(np.float64), want,
                                "static vs oracle")


def test_static_scratch_rejects_shapes_beyond_its_size():
    # 16 query heads per kv head over 8 kv heads needs more partial state than the
    # fixed array holds: refused on the host, nothing launched
    (cache, q, q_pos, bt, ctx), _ = _case(34, [40, 50], Hkv=8, G=2)
    need = K.kvinj_decode_workspace_size(2, 8 * 16, 8, 128)
    assert need > K.KVINJ_STATIC_SCRATCH_BYTES
    q16 = torch.zeros((2, 8 * 16, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q16)
    with pytest.raises(K.KvinjError) as e:
        K.kvinj_paged_decode_static(cache, None, 0, q16, q_pos, bt, ctx, out)
    assert e.value.code == K.KVINJ_EWORKSPACE
