// tq_decode_mma_d96.cu -- tensor-core decode-attention instantiations for head dim 96
// (one translation unit per head dim so they compile in parallel).
#include "tq_decode_mma.cuh"

namespace tq {

template <int D>
cudaError_t launch_mma_d_extern(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt, cudaStream_t st);

template <>
cudaError_t launch_mma_d_extern<96>(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt,
                                     cudaStream_t st) {
    return mma_detail::launch_mma_d<96>(a, p, kb, vb, nt, st);
}

}  // namespace tq
