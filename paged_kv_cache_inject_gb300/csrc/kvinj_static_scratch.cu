// kvinj_static_scratch.cu -- kvinj_paged_decode_static: paged decode whose
// scratch lives in a fixed device array of this library instead of a
// caller-provided workspace.
//
// Why: kvinj_paged_decode needs a workspace (cut-segment descriptors and the
// partial softmax states of the split context). Some callers cannot obtain
// one: code that runs where allocation is not allowed or not safe -- an
// engine's enqueue hook or plugin that must not call cudaMalloc (which can
// implicitly synchronize the device), a serving process whose memory pool has
// already been carved up, or a path that must not fail on memory pressure in
// the middle of a request. This entry point allocates nothing. Its scratch is
// the array below: KVINJ_STATIC_SCRATCH_BYTES of device memory that every GPU
// which loads this library holds until the process exits.
//
// Set-up: every call looks up the array's device address on the current
// device with cudaGetSymbolAddress (a host-side lookup, no stream work) and
// passes that address to the kernels; host code never hands the array's name
// itself to a kernel (in host code it is only a stand-in for the device
// symbol). The address is not cached: after a cudaDeviceReset, or when the
// device's primary context is destroyed and recreated, the module is loaded
// again and the array may sit elsewhere, and a cached address would point at
// freed memory. The first call on a device loads this library's device code
// there if nothing else has.
//
// Sharing: every call on a device uses the same array and leaves the last
// call's contents there. Nothing in it needs to start at zero (each call
// writes every descriptor and partial state before reading it), but two calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on the array and may corrupt each other's results.
#include "kvinj.h"
#include "kvinj_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[KVINJ_STATIC_SCRATCH_BYTES];

// device address of g_decode_scratch in the current device's context
int scratch_address(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess || !p) {
    if (e != cudaSuccess) cudaGetLastError();  // not sticky: clear it
    return KVINJ_ECUDA;
  }
  *out = p;
  return KVINJ_OK;
}

}  // namespace

extern "C" int kvinj_paged_decode_static(const kvinj_cache *cache, const kvinj_rope *rope,
                                         int32_t layer, int32_t num_q_heads, const void *q,
                                         const int32_t *q_pos, const int32_t *block_tables,
                                         int32_t max_blocks, const int32_t *context_lens,
                                         int32_t batch, float scale, void *out,
                                         int32_t *dev_status, kvinj_stream_t stream) {
  if (!cache || num_q_heads <= 0 || cache->num_kv_heads <= 0) return KVINJ_EINVAL;
  const size_t need = kvinj_decode_workspace_size(batch, num_q_heads, cache->num_kv_heads,
                                                  cache->head_dim);
  if (need > (size_t)KVINJ_STATIC_SCRATCH_BYTES) return KVINJ_EWORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc) return rc;
  return kvinj_paged_decode(cache, rope, layer, num_q_heads, q, q_pos, block_tables, max_blocks,
                            context_lens, batch, scale, out, scratch,
                            (size_t)KVINJ_STATIC_SCRATCH_BYTES, dev_status, stream);
}
