"""kvinj_paged_decode_static: paged decode for callers that cannot allocate.

Some callers cannot hand the library a workspace: code running inside an
engine hook or plugin that must not call cudaMalloc, or in a process whose
device memory is already handed out. This entry point keeps its scratch in a
fixed device array of the library instead. Its results must match the
workspace entry point's on the same inputs, call after call (the array keeps
the previous call's contents, which must not leak into the next result).
The file sorts last so that a run stopping at the first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import workload as W
from paged_kv_cache_inject_gb300 import kvinj as K
from tests.gpu_helpers import assert_decode_close, from_bits

pytestmark = pytest.mark.gpu


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
    def bits(shape, off):
        n = int(np.prod(shape))
        return W.normal_bits(key, off + np.arange(n, dtype=np.uint64), W.BF16).reshape(shape)
    kc = bits((L, NB, Hkv, 16, D), 0)
    vc = bits((L, NB, Hkv, 16, D), 1 << 32)
    q = bits((ctx.size, Hkv * G, D), 1 << 33)
    cache = K.Cache(from_bits(kc, torch.bfloat16), from_bits(vc, torch.bfloat16))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return cache, from_bits(q, torch.bfloat16), dev(ctx - 1), dev(bt), dev(ctx)


def test_static_scratch_matches_workspace_entry_point_two_calls_in_a_row():
    rope = K.make_rope(5e5, 128, 4096)
    cases = [_case(31, [700, 33, 1500, 16, 2048, 5]), _case(32, [100, 3000, 17, 900])]
    for cache, q, q_pos, bt, ctx in cases:
        batch, Hq, D = q.shape
        ref = torch.empty_like(q)
        ws = K.make_decode_workspace(batch, Hq, cache.num_kv_heads, D)
        K.kvinj_paged_decode(cache, rope, 1, q, q_pos, bt, ctx, ref, ws)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = torch.full_like(q, float("nan"))
        K.kvinj_paged_decode_static(cache, rope, 1, q, q_pos, bt, ctx, got, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        assert_decode_close(got.float().cpu().numpy().astype(np.float64),
                            ref.float().cpu().numpy().astype(np.float64), "static vs workspace")


def test_static_scratch_rejects_shapes_beyond_its_size():
    # 16 query heads per kv head over 8 kv heads needs more partial state than the
    # fixed array holds: refused on the host, nothing launched
    cache, q, q_pos, bt, ctx = _case(33, [40, 50], Hkv=8, G=2)
    need = K.kvinj_decode_workspace_size(2, 8 * 16, 8, 128)
    assert need > (24 << 20)
    q16 = torch.zeros((2, 8 * 16, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q16)
    with pytest.raises(K.KvinjError) as e:
        K.kvinj_paged_decode_static(cache, None, 0, q16, q_pos, bt, ctx, out)
    assert e.value.code == K.KVINJ_EWORKSPACE
