// kvinj_decode_umma_early.cu -- the tcgen05 paged decode for calls with
// KVINJ_DECODE_KV_READY: the split-K pass reads the context lengths, q
// positions and block tables, and issues its first stages of K/V pages, before
// it waits for the kernel ahead of it (the kernel template is in
// kvinj_decode_umma.cuh; its own translation unit so that the two
// instantiations compile in parallel).
#include "kvinj_decode_umma.cuh"

namespace kvinj {

cudaError_t launch_decode_umma_early(const DecodeArgs &a, const CUtensorMap &tmK,
                                     const CUtensorMap &tmV, int G, int dtype, int ctas,
                                     cudaStream_t s) {
  return launch_decode_umma_t<true>(a, tmK, tmV, G, dtype, ctas, s);
}

}  // namespace kvinj
