// kq_inst_tc.cu -- the tensor-core kernels (kq_tc.cuh) for one and two
// octets of tokens, and their ntok-dispatching entry points.
#include "kq_launch.cuh"

namespace kqlaunch {

cudaError_t direct_tc(int noct, const kq::SetParams &p, int grid, size_t smem, cudaStream_t s) {
    return noct == 1 ? launch_direct<8, true>(p, grid, smem, s)
                     : launch_direct<16, true>(p, grid, smem, s);
}

cudaError_t stream_tc(int noct, const kq::StreamParams &p, int grid, size_t smem,
                      cudaStream_t s) {
    return noct == 1 ? launch_stream<8, false, true>(p, grid, smem, s)
                     : launch_stream<16, false, true>(p, grid, smem, s);
}

}  // namespace kqlaunch
