// kvinj_decode_umma.cu -- the tcgen05 paged decode for calls that wait for the
// kernel ahead of them before any read (the kernel template is in
// kvinj_decode_umma.cuh), and the dispatch to the early-reading instantiation
// of kvinj_decode_umma_early.cu.
#include "kvinj_decode_umma.cuh"

namespace kvinj {

cudaError_t launch_decode_umma_early(const DecodeArgs &a, const CUtensorMap &tmK,
                                     const CUtensorMap &tmV, int G, int dtype, int ctas,
                                     cudaStream_t s);

cudaError_t launch_decode_umma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int D, int G, int HG, int dtype, int ctas,
                               cudaStream_t s) {
  if (D != 128 || HG != 8) return cudaErrorInvalidValue;
  if (a.early) return launch_decode_umma_early(a, tmK, tmV, G, dtype, ctas, s);
  return launch_decode_umma_t<false>(a, tmK, tmV, G, dtype, ctas, s);
}

}  // namespace kvinj
