// kq_api.cu -- the C ABI of libkq (include/kq.h): argument validation,
// launch planning and the kernel launch.  Validation is pure host logic and
// runs before any CUDA call, so a rejected call enqueues nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "kq.h"
#include "kq_kernel_direct.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

int64_t block_bytes_of(int fmt) {
    switch (fmt) {
    case KQ_Q4_K: return 144;
    case KQ_Q5_K: return 176;
    case KQ_Q6_K: return 210;
    default: return -1;
    }
}

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
bool overlaps(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

kq_status check_member(const kq_mat &m, int ntok) {
    if (block_bytes_of(m.fmt) < 0) return KQ_ERR_FORMAT;
    if (m.rows < 1 || m.rows > KQ_MAX_ROWS || m.cols < 256 ||
        m.cols % 256 != 0 || m.cols > KQ_MAX_COLS)
        return KQ_ERR_SHAPE;
    if (m.reserved != 0) return KQ_ERR_SHAPE;
    if (!m.W || !m.x || !m.y) return KQ_ERR_NULL;
    if (((uintptr_t)m.W & 15u) || ((uintptr_t)m.x & 15u) ||
        ((uintptr_t)m.y & 3u))
        return KQ_ERR_ALIGN;
    (void)ntok;
    return KQ_OK;
}

Range w_range(const kq_mat &m) {
    const uintptr_t lo = (uintptr_t)m.W;
    return {lo, lo + (uintptr_t)(m.rows * (m.cols / 256) * block_bytes_of(m.fmt))};
}
Range x_range(const kq_mat &m, int ntok) {
    const uintptr_t lo = (uintptr_t)m.x;
    return {lo, lo + (uintptr_t)(m.cols * ntok * (int64_t)sizeof(float))};
}
Range y_range(const kq_mat &m, int ntok) {
    const uintptr_t lo = (uintptr_t)m.y;
    return {lo, lo + (uintptr_t)(m.rows * ntok * (int64_t)sizeof(float))};
}

kq_status validate_set(const kq_mat *mats, int n, int ntok) {
    if (n < 1 || n > KQ_MAX_SET) return KQ_ERR_COUNT;
    if (!mats) return KQ_ERR_NULL;
    if (ntok < 1 || ntok > KQ_MAX_NTOK) return KQ_ERR_NTOK;
    for (int i = 0; i < n; ++i) {
        const kq_status s = check_member(mats[i], ntok);
        if (s != KQ_OK) return s;
    }
    for (int i = 0; i < n; ++i) {
        const Range yi = y_range(mats[i], ntok);
        for (int j = 0; j < n; ++j) {
            if (overlaps(yi, w_range(mats[j])) ||
                overlaps(yi, x_range(mats[j], ntok)))
                return KQ_ERR_ALIAS;
            if (j != i && overlaps(yi, y_range(mats[j], ntok)))
                return KQ_ERR_ALIAS;
        }
    }
    return KQ_OK;
}

// ---------------------------------------------------------------- device
struct DeviceInfo {
    int sms = 0;
};

DeviceInfo device_info(int dev) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) dev = 0;
    if (cache[dev].sms == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                cudaSuccess ||
            sms <= 0)
            sms = 148;
        cache[dev].sms = sms;
    }
    return cache[dev];
}

constexpr int kSmemLimit = 200 * 1024;

template <int NTOK>
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
            e = cudaFuncSetAttribute(kq::kq_set_direct<NTOK>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemLimit);
            if (e != cudaSuccess) return e;
            configured[dev] = kSmemLimit;
        }
    }
    kq::kq_set_direct<NTOK><<<grid, kq::kDirectThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

kq_status run_set(const kq_mat *mats, int n, int ntok, void *stream) {
    const kq_status v = validate_set(mats, n, ntok);
    if (v != KQ_OK) return v;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    const DeviceInfo info = device_info(dev);

    kq::SetParams p{};
    p.n = n;
    int64_t grid = 0;
    size_t smem = 0;
    for (int i = 0; i < n; ++i) {
        const kq_mat &m = mats[i];
        const int nb = (int)(m.cols / 256);
        // Rows per CTA: about one (row, block) pair per thread, at most 32,
        // fewer when the matrix would otherwise not reach every SM, and few
        // enough that the per-block partials fit in shared memory.
        int64_t rpc = std::max<int64_t>(1, kq::kDirectThreads / nb);
        rpc = std::min<int64_t>(rpc, 32);
        rpc = std::min<int64_t>(rpc, std::max<int64_t>(1, (m.rows + info.sms - 1) / info.sms));
        const int64_t per_row = (int64_t)nb * ntok * (int64_t)sizeof(float);
        rpc = std::min<int64_t>(rpc, std::max<int64_t>(1, kSmemLimit / per_row));
        if (per_row * rpc > kSmemLimit) return KQ_ERR_SHAPE;
        p.m[i].W = (const uint8_t *)m.W;
        p.m[i].x = m.x;
        p.m[i].y = m.y;
        p.m[i].rows = m.rows;
        p.m[i].nb = nb;
        p.m[i].fmt = m.fmt;
        p.m[i].cta_begin = (int32_t)grid;
        p.m[i].rpc = (int32_t)rpc;
        grid += (m.rows + rpc - 1) / rpc;
        smem = std::max<size_t>(smem, (size_t)(per_row * rpc));
        if (grid > 0x7FFFFFFF) return KQ_ERR_SHAPE;
    }

    cudaStream_t s = (cudaStream_t)stream;
    switch (ntok) {
    case 1: e = launch_direct<1>(p, (int)grid, smem, s); break;
    case 2: e = launch_direct<2>(p, (int)grid, smem, s); break;
    case 3: e = launch_direct<3>(p, (int)grid, smem, s); break;
    case 4: e = launch_direct<4>(p, (int)grid, smem, s); break;
    case 5: e = launch_direct<5>(p, (int)grid, smem, s); break;
    case 6: e = launch_direct<6>(p, (int)grid, smem, s); break;
    case 7: e = launch_direct<7>(p, (int)grid, smem, s); break;
    default: e = launch_direct<8>(p, (int)grid, smem, s); break;
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    return KQ_OK;
}

}  // namespace

extern "C" {

int64_t kq_block_bytes(int fmt) { return block_bytes_of(fmt); }

int64_t kq_matrix_bytes(int fmt, int64_t rows, int64_t cols) {
    const int64_t bb = block_bytes_of(fmt);
    if (bb < 0 || rows < 1 || rows > KQ_MAX_ROWS || cols < 256 ||
        cols % 256 != 0 || cols > KQ_MAX_COLS)
        return -1;
    return rows * (cols / 256) * bb;
}

kq_status kq_matvec(int fmt, const void *W, int64_t rows, int64_t cols,
                    const float *x, float *y, int ntok, void *stream) {
    kq_mat m;
    m.fmt = fmt;
    m.reserved = 0;
    m.W = W;
    m.rows = rows;
    m.cols = cols;
    m.x = x;
    m.y = y;
    return run_set(&m, 1, ntok, stream);
}

kq_status kq_matvec_set(const kq_mat *mats, int n, int ntok, void *stream) {
    return run_set(mats, n, ntok, stream);
}

const char *kq_status_str(int status) {
    switch (status) {
    case KQ_OK: return "ok";
    case KQ_ERR_FORMAT: return "unknown block format";
    case KQ_ERR_SHAPE: return "invalid or unsupported rows/cols";
    case KQ_ERR_NTOK: return "ntok outside 1..8";
    case KQ_ERR_NULL: return "null pointer";
    case KQ_ERR_ALIGN: return "misaligned pointer (W, x: 16 bytes; y: 4 bytes)";
    case KQ_ERR_ALIAS: return "an output overlaps an input or another output";
    case KQ_ERR_COUNT: return "set size outside 1..16";
    case KQ_ERR_CUDA: return "CUDA launch failed";
    case KQ_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
    }
}

int kq_last_cuda_error(void) { return g_last_cuda_error; }

int kq_version(void) { return (1 << 16) | 0; }

}  // extern "C"
