// tq_decode_mma_d64_stream.cu -- tensor-core decode-attention instantiations of the
// token-balanced schedule for head dim 64 (own translation unit: compiled in parallel).
#include "tq_decode_mma.cuh"

namespace tq {

template <int D>
cudaError_t launch_mma_d_stream_extern(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt, cudaStream_t st);

template <>
cudaError_t launch_mma_d_stream_extern<64>(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt,
                                           cudaStream_t st) {
    return mma_detail::launch_mma_d_stream<64>(a, p, kb, vb, nt, st);
}

}  // namespace tq
