// na_tc_f16.cu -- fp16 instantiations of the tensor-core kernels (na_tc_impl.cuh), compiled in a
// translation unit of their own so that the two element types build in parallel.
#include "na_tc_impl.cuh"

namespace na {

namespace {
template <int WHICH>
int launch_f16(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_tc<16, WHICH, true>(p, s);
        case 32: return launch_tc<32, WHICH, true>(p, s);
        case 64: return launch_tc<64, WHICH, true>(p, s);
        case 128: return launch_tc<128, WHICH, true>(p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}
}  // namespace

int launch_fwd_tc_f16(const TcParams& p, cudaStream_t s) { return launch_f16<0>(p, s); }
int launch_dq_tc_f16(const TcParams& p, cudaStream_t s) { return launch_f16<1>(p, s); }
int launch_dkdv_tc_f16(const TcParams& p, cudaStream_t s) { return launch_f16<2>(p, s); }

}  // namespace na
