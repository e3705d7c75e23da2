// Instantiations of the bf16 decode kernel for 16-token pages.
#include "decode_impl.cuh"

namespace pkv {

cudaError_t launch_bf16_p16(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    if (p.y.d == 128) return launch_bf16<16, 128, 0, 0>(p, total_pages, max_pages, num_sms, st);
    if (p.y.d == 64) return launch_bf16<16, 64, 0, 0>(p, total_pages, max_pages, num_sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
