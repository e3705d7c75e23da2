// Instantiations of the bf16 decode kernel for stores whose keys precede
// RoPE [PuzzleKV §4.1, Appendix D.3]: P = 32 and 64, d = 64 and 128.
#include "decode_impl.cuh"

namespace pkv {

cudaError_t launch_bf16_rope(DecodeParams &p, long total_pages, int max_pages, int num_sms, cudaStream_t st) {
    const int P = p.y.P, d = p.y.d;
    if (P == 64 && d == 128 && p.y.rkp == 16 && p.y.rvp == 24)
        return launch_bf16<64, 128, 2, 3, false, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 64 && d == 128) return launch_bf16<64, 128, 0, 0, false, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 64 && d == 64) return launch_bf16<64, 64, 0, 0, false, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 32 && d == 128) return launch_bf16<32, 128, 0, 0, false, true>(p, total_pages, max_pages, num_sms, st);
    if (P == 32 && d == 64) return launch_bf16<32, 64, 0, 0, false, true>(p, total_pages, max_pages, num_sms, st);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
