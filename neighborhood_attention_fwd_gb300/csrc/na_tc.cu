// na_tc.cu -- bf16 instantiations of the tensor-core kernels (na_tc_impl.cuh) and the plan
// quantities the host planner needs.
#include "na_tc_impl.cuh"

namespace na {

uint32_t tc_smem_bytes(int which, const TilePlan& pl, int D) { return tc_layout(which, pl, D).total + 1024u; }

int tc_tmem_cols(int which, int D) { return tmem_cols_of(which, D); }

int tc_max_nc(int which, int D, int sbufs) {
    // the score accumulators (the backward's double-buffered with their dP beside them, the forward's
    // two or three) plus the tile accumulators; the forward's P overwrites its scores, and its softmax
    // takes a run of at most six groups (96 columns)
    const int cols = tc_tmem_cols(which, D);
    const int acc = (which == 2 ? 2 : 1) * abufs_of(which, D) * D;
    const int nc = which == 0 ? (cols - acc) / sbufs : (cols - acc) / 4;
    const int cap = which == 0 ? 96 : 128;
    return (nc < cap ? nc : cap) / 16 * 16;
}

namespace {
template <int WHICH>
int launch_bf16(const TcParams& p, cudaStream_t s) {
    switch (p.D) {
        case 16: return launch_tc<16, WHICH, false>(p, s);
        case 32: return launch_tc<32, WHICH, false>(p, s);
        case 64: return launch_tc<64, WHICH, false>(p, s);
        case 128: return launch_tc<128, WHICH, false>(p, s);
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
}
}  // namespace

int launch_fwd_tc(const TcParams& p, cudaStream_t s) { return p.f16 ? launch_fwd_tc_f16(p, s) : launch_bf16<0>(p, s); }
int launch_dq_tc(const TcParams& p, cudaStream_t s) { return p.f16 ? launch_dq_tc_f16(p, s) : launch_bf16<1>(p, s); }
int launch_dkdv_tc(const TcParams& p, cudaStream_t s) {
    return p.f16 ? launch_dkdv_tc_f16(p, s) : launch_bf16<2>(p, s);
}

}  // namespace na
