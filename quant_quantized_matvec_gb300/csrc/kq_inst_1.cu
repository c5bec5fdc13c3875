// kq_inst_1.cu -- kernels for ntok = 1 (see kq_launch.cuh).
#include "kq_launch.cuh"

KQ_DEFINE_INSTANCES(1)

namespace kqlaunch {
template cudaError_t launch_stream<1, true, false, kq::kStreamConsumersTall>(
    const kq::StreamParams &, int, size_t, cudaStream_t);
template cudaError_t launch_stream<1, true, false, kq::kStreamConsumersTall, 1>(
    const kq::StreamParams &, int, size_t, cudaStream_t);
}
