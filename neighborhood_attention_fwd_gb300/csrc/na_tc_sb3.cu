// na_tc_sb3.cu -- the forward tensor-core kernels with three score buffers (D <= 32, bf16 and fp16),
// for plans whose tiles walk many chunks.  They sit in a translation unit of their own so that the
// two-buffer kernels' code is laid out as without them.
#include "na_tc_impl.cuh"

namespace na {

int launch_fwd_tc_sb3(const TcParams& p, cudaStream_t s) {
    switch (p.D * 2 + (p.f16 ? 1 : 0)) {
        case 32: return launch_tc_sb<16, 0, false, 3>(p, s);
        case 33: return launch_tc_sb<16, 0, true, 3>(p, s);
        case 64: return launch_tc_sb<32, 0, false, 3>(p, s);
        case 65: return launch_tc_sb<32, 0, true, 3>(p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}

}  // namespace na
