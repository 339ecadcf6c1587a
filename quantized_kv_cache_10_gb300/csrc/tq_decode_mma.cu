// tq_decode_mma.cu -- tensor-core fused decode attention (filled in below).
#include "tq_decode_common.cuh"

namespace tq {

void build_decode_tables(const tq_codec& c, std::vector<uint32_t>& ktab, std::vector<uint32_t>& vtab) {
    (void)c;
    ktab.clear();
    vtab.clear();
}

bool decode_mma_supported(const tq_codec* ck, const tq_codec* cv, int G) {
    (void)ck;
    (void)cv;
    (void)G;
    return false;
}

cudaError_t launch_decode_mma(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    (void)a;
    (void)p;
    (void)st;
    return cudaErrorNotSupported;
}

}  // namespace tq
