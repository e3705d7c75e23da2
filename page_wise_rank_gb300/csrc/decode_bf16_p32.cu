// Instantiations of the bf16 decode kernel for 32-token pages.
#include "decode_impl.cuh"

namespace pkv {

cudaError_t launch_bf16_p32(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    const int rkt = p.y.rkp / 8, rvt = p.y.rvp / 8;
    if (p.y.d == 128 && rkt <= 4 && rvt <= 4) {
        switch (rkt * 8 + rvt) {
            case 9: return launch_bf16<32, 128, 1, 1>(p, total_pages, max_pages, num_sms, st);
            case 10: return launch_bf16<32, 128, 1, 2>(p, total_pages, max_pages, num_sms, st);
            case 11: return launch_bf16<32, 128, 1, 3>(p, total_pages, max_pages, num_sms, st);
            case 12: return launch_bf16<32, 128, 1, 4>(p, total_pages, max_pages, num_sms, st);
            case 17: return launch_bf16<32, 128, 2, 1>(p, total_pages, max_pages, num_sms, st);
            case 18: return launch_bf16<32, 128, 2, 2>(p, total_pages, max_pages, num_sms, st);
            case 19: return launch_bf16<32, 128, 2, 3>(p, total_pages, max_pages, num_sms, st);
            case 20: return launch_bf16<32, 128, 2, 4>(p, total_pages, max_pages, num_sms, st);
            case 25: return launch_bf16<32, 128, 3, 1>(p, total_pages, max_pages, num_sms, st);
            case 26: return launch_bf16<32, 128, 3, 2>(p, total_pages, max_pages, num_sms, st);
            case 27: return launch_bf16<32, 128, 3, 3>(p, total_pages, max_pages, num_sms, st);
            case 28: return launch_bf16<32, 128, 3, 4>(p, total_pages, max_pages, num_sms, st);
            case 33: return launch_bf16<32, 128, 4, 1>(p, total_pages, max_pages, num_sms, st);
            case 34: return launch_bf16<32, 128, 4, 2>(p, total_pages, max_pages, num_sms, st);
            case 35: return launch_bf16<32, 128, 4, 3>(p, total_pages, max_pages, num_sms, st);
            case 36: return launch_bf16<32, 128, 4, 4>(p, total_pages, max_pages, num_sms, st);
            default: break;
        }
    }
    if (p.y.d == 128) return launch_bf16<32, 128, 0, 0>(p, total_pages, max_pages, num_sms, st);
    if (p.y.d == 64) return launch_bf16<32, 64, 0, 0>(p, total_pages, max_pages, num_sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
