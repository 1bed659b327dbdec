"""GB300-native (sm_103a) paged KV-cache injection and paged GQA decode.

The compute path is libkvinj.so (hand-written CUDA, C ABI in include/kvinj.h);
``kvinj`` is its thin ctypes binding and ``build`` compiles it in-tree.
"""
from . import kvinj  # noqa: F401
from .kvinj import (  # noqa: F401
    Cache, KvinjError, Pool, Rope, kvinj_append, kvinj_append_paged_decode, kvinj_copy_blocks,
    kvinj_decode_workspace_init,
    kvinj_decode_workspace_size, kvinj_inject, kvinj_kv_bytes, kvinj_paged_decode,
    kvinj_paged_decode_ex, kvinj_paged_decode_static, kvinj_paged_decode_window,
    kvinj_paged_prefill, kvinj_prefill_workspace_size, make_prefill_workspace, kvinj_rope_table_bytes, kvinj_rope_table_host, kvinj_slot_mapping,
    kvinj_strerror, make_decode_workspace, make_rope,
)
