// Instantiations of the bf16 decode kernel for INT4 factor stores.
#include "decode_impl.cuh"

namespace pkv {

cudaError_t launch_bf16_q4(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    const int P = p.y.P, d = p.y.d;
    if (P == 64 && d == 128 && p.y.rkp == 16 && p.y.rvp == 24)
        return launch_bf16<64, 128, 2, 3, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 32 && d == 128 && p.y.rkp == 16 && p.y.rvp == 16)  // the pages' own (16, 14)
        return launch_bf16<32, 128, 2, 2, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 64 && d == 128) return launch_bf16<64, 128, 0, 0, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 64 && d == 64) return launch_bf16<64, 64, 0, 0, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 32 && d == 128) return launch_bf16<32, 128, 0, 0, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 32 && d == 64) return launch_bf16<32, 64, 0, 0, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 16 && d == 128) return launch_bf16<16, 128, 0, 0, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 16 && d == 64) return launch_bf16<16, 64, 0, 0, true>(p, total_pages, max_pages, num_sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
