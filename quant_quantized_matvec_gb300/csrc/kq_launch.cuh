// kq_launch.cuh -- kernel launch entry points, one set per token count.
// Each kq_inst_<n>.cu instantiates them for ntok = n so that the kernels
// compile in parallel translation units; kq_api.cu calls them through
// kq_launch_direct / kq_launch_stream.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "kq_kernel_direct.cuh"
#include "kq_kernel_stream.cuh"

namespace kqlaunch {

constexpr int kDirectSmemLimit = 200 * 1024;

template <int NTOK, bool TC = false>
cudaError_t launch_direct(const kq::SetParams &p, int grid, size_t smem,
                          cudaStream_t stream) {
    static std::mutex mu;
    static size_t configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    if (smem > 48 * 1024) {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev] < smem) {
            e = cudaFuncSetAttribute(kq::kq_set_direct<NTOK, TC>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kDirectSmemLimit);
            if (e != cudaSuccess) return e;
            configured[dev] = kDirectSmemLimit;
        }
    }
    kq::kq_set_direct<NTOK, TC><<<grid, kq::kDirectThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int NTOK, bool XSMEM, bool TC = false, int NCW = kq::kStreamConsumers, int RPT = 2>
cudaError_t launch_stream(const kq::StreamParams &p, int grid, size_t smem, cudaStream_t s) {
    static std::mutex mu;
    static size_t configured[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) dev = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (configured[dev] < smem) {
            e = cudaFuncSetAttribute(kq::kq_set_stream<NTOK, XSMEM, TC, NCW, RPT>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            configured[dev] = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(32 * (NCW + 1));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (p.overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kq::kq_set_stream<NTOK, XSMEM, TC, NCW, RPT>, p);
}

// Row gather + dequantization (kq_rows.cu).
cudaError_t rows(int fmt, const uint8_t *W, int64_t rows, int nb, const int32_t *ids, int64_t n,
                 float *out, cudaStream_t s);

// ntok-dispatching entry points (defined in kq_api.cu from the instances)
cudaError_t direct(int ntok, const kq::SetParams &p, int grid, size_t smem, cudaStream_t s);
// (tall: a one-column launch of Q6_K members whose CTAs stream many
// stages, run with kq::kStreamConsumersTall consumer warps; rpt: rows a
// lane-task, 2, or 1 for tall sets staged in row segments)
cudaError_t stream(int ntok, bool xsmem, const kq::StreamParams &p, int grid, size_t smem,
                   cudaStream_t s, bool tall, int rpt);
// tensor-core launches of noct octets of tokens (kq_inst_tc.cu)
cudaError_t direct_tc(int noct, const kq::SetParams &p, int grid, size_t smem, cudaStream_t s);
cudaError_t stream_tc(int noct, const kq::StreamParams &p, int grid, size_t smem,
                      cudaStream_t s);

}  // namespace kqlaunch

#define KQ_DECLARE_INSTANCES(N)                                                            \
    namespace kqlaunch {                                                                   \
    extern template cudaError_t launch_direct<N, false>(const kq::SetParams &, int,        \
                                                        size_t, cudaStream_t);             \
    extern template cudaError_t launch_stream<N, true, false>(const kq::StreamParams &,    \
                                                              int, size_t, cudaStream_t);  \
    extern template cudaError_t launch_stream<N, false, false>(const kq::StreamParams &,   \
                                                               int, size_t, cudaStream_t); \
    }
#define KQ_DEFINE_INSTANCES(N)                                                             \
    namespace kqlaunch {                                                                   \
    template cudaError_t launch_direct<N, false>(const kq::SetParams &, int, size_t,       \
                                                 cudaStream_t);                            \
    template cudaError_t launch_stream<N, true, false>(const kq::StreamParams &, int,      \
                                                       size_t, cudaStream_t);              \
    template cudaError_t launch_stream<N, false, false>(const kq::StreamParams &, int,     \
                                                        size_t, cudaStream_t);             \
    }
