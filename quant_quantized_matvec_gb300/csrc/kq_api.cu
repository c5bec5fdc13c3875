// kq_api.cu -- the C ABI of libkq (include/kq.h): argument validation,
// launch planning and the kernel launch.  Validation is pure host logic and
// runs before any CUDA call, so a rejected call enqueues nothing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "kq.h"
#include "kq_internal.h"
#include "kq_launch.cuh"
#include "kq_plan.h"

KQ_DECLARE_INSTANCES(1)
KQ_DECLARE_INSTANCES(2)
KQ_DECLARE_INSTANCES(3)
KQ_DECLARE_INSTANCES(4)
KQ_DECLARE_INSTANCES(5)
KQ_DECLARE_INSTANCES(6)
KQ_DECLARE_INSTANCES(7)
KQ_DECLARE_INSTANCES(8)
namespace kqlaunch {
extern template cudaError_t launch_stream<1, true, false, kq::kStreamConsumersTall>(
    const kq::StreamParams &, int, size_t, cudaStream_t);
extern template cudaError_t launch_stream<1, true, false, kq::kStreamConsumersTall, 1>(
    const kq::StreamParams &, int, size_t, cudaStream_t);
}

namespace kqlaunch {
cudaError_t direct(int ntok, const kq::SetParams &p, int grid, size_t smem, cudaStream_t s) {
    switch (ntok) {
    case 1: return launch_direct<1>(p, grid, smem, s);
    case 2: return launch_direct<2>(p, grid, smem, s);
    case 3: return launch_direct<3>(p, grid, smem, s);
    case 4: return launch_direct<4>(p, grid, smem, s);
    case 5: return launch_direct<5>(p, grid, smem, s);
    case 6: return launch_direct<6>(p, grid, smem, s);
    case 7: return launch_direct<7>(p, grid, smem, s);
    default: return launch_direct<8>(p, grid, smem, s);
    }
}
cudaError_t stream(int ntok, bool xsmem, const kq::StreamParams &p, int grid, size_t smem,
                   cudaStream_t s, bool tall, int rpt) {
    switch (ntok * 2 + (xsmem ? 1 : 0)) {
    case 3:
        if (tall && rpt == 1)
            return launch_stream<1, true, false, kq::kStreamConsumersTall, 1>(p, grid, smem, s);
        return tall ? launch_stream<1, true, false, kq::kStreamConsumersTall>(p, grid, smem, s)
                    : launch_stream<1, true>(p, grid, smem, s);
    case 2: return launch_stream<1, false>(p, grid, smem, s);
    case 5: return launch_stream<2, true>(p, grid, smem, s);
    case 4: return launch_stream<2, false>(p, grid, smem, s);
    case 7: return launch_stream<3, true>(p, grid, smem, s);
    case 6: return launch_stream<3, false>(p, grid, smem, s);
    case 9: return launch_stream<4, true>(p, grid, smem, s);
    case 8: return launch_stream<4, false>(p, grid, smem, s);
    case 11: return launch_stream<5, true>(p, grid, smem, s);
    case 10: return launch_stream<5, false>(p, grid, smem, s);
    case 13: return launch_stream<6, true>(p, grid, smem, s);
    case 12: return launch_stream<6, false>(p, grid, smem, s);
    case 15: return launch_stream<7, true>(p, grid, smem, s);
    case 14: return launch_stream<7, false>(p, grid, smem, s);
    case 17: return launch_stream<8, true>(p, grid, smem, s);
    default: return launch_stream<8, false>(p, grid, smem, s);
    }
}
}  // namespace kqlaunch

// Device error word: set by a kernel whose bounded wait expired.
__device__ unsigned int g_kq_device_error;

namespace kq {
// Input records of every member, written to global memory (kq_xrec.cuh).
__global__ void __launch_bounds__(kPrepThreads) kq_xprep(const __grid_constant__ PrepParams p) {
    const int64_t w = ((int64_t)blockIdx.x * kPrepThreads + threadIdx.x) >> 5;
    if (w >= p.first_warp[p.n]) return;
    int mi = 0;
#pragma unroll 1
    for (int i = 1; i < p.n; ++i)
        if (w >= p.first_warp[i]) mi = i;
    const int i = (int)(w - p.first_warp[mi]);
    const int nb = p.nb[mi];
    const bool q6 = p.q6[mi] != 0;
    const int lane = threadIdx.x & 31;
    const int t = (i >> 1) / nb, ih = i - 2 * nb * t;  // token, half within the token
    const float4 v = record_inputs(p.x[mi], (int64_t)nb * 256, t, ih, lane);
    build_record_half(v, p.rec[mi] + (int64_t)(i >> 1) * rec_bytes(q6), i & 1, q6, lane);
}

// Input planes that live in host memory, copied once into device memory:
// one float4 per thread.  It lets the next kernel on the stream launch at
// once, so that kernel streams its weights while this copy runs.
struct StageParams {
    const float4 *src[KQ_MAX_SET];
    float4 *dst[KQ_MAX_SET];
    int64_t first[KQ_MAX_SET + 1];  // first float4 of each plane; first[n] = total
    int n;
};
constexpr int kStageThreads = 256;

__global__ void __launch_bounds__(kStageThreads) kq_xstage(const __grid_constant__ StageParams p) {
    // the matvec after this copy may start at once (it streams its weights
    // and waits for the copy before reading x); with launch overlap on this
    // copy itself is launched while the kernel before it still runs, and
    // waits for it before reading x or writing anything (a no-op otherwise)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t i = (int64_t)blockIdx.x * kStageThreads + threadIdx.x;
    if (i >= p.first[p.n]) return;
    int k = 0;
#pragma unroll 1
    for (int j = 1; j < p.n; ++j)
        if (i >= p.first[j]) k = j;
    const int64_t o = i - p.first[k];
    p.dst[k][o] = p.src[k][o];
}

// Input fragments of the tensor-core launches (kq_xtc.cuh): kTcPrepSplit
// warps per (plane, octet, column); planes are the distinct (x, cols) of a
// set.
struct TcPrepParams {
    const float *x[KQ_MAX_SET];
    uint8_t *rec[KQ_MAX_SET];
    int32_t nb[KQ_MAX_SET];
    int64_t first_warp[KQ_MAX_SET + 1];
    int32_t n, ntok;
};
constexpr int kTcPrepThreads = 128;

__global__ void __launch_bounds__(kTcPrepThreads) kq_xprep_tc(const __grid_constant__ TcPrepParams p) {
    // the matvec launched after this pass overlaps it (streaming its
    // weights) and waits for it before reading the fragments; this pass,
    // when launched to overlap the kernel before it, waits for that kernel
    // before reading x (a no-op otherwise)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ uint32_t smax[kTcPrepSplit * 8];
    static_assert(kTcPrepThreads == 32 * kTcPrepSplit, "one block per (plane, octet, column)");
    // every plane's warps start at a multiple of kTcPrepSplit, so a block's
    // warps all work or all return (build_tc_record holds a block barrier)
    const int64_t w = ((int64_t)blockIdx.x * kTcPrepThreads + threadIdx.x) >> 5;
    if ((int64_t)blockIdx.x * kTcPrepSplit >= p.first_warp[p.n]) return;
    int k = 0;
#pragma unroll 1
    for (int i = 1; i < p.n; ++i)
        if (w >= p.first_warp[i]) k = i;
    const int i = (int)(w - p.first_warp[k]);
    const int nb = p.nb[k];
    const int noct = (p.ntok + 7) / 8;
    const int q = i % kTcPrepSplit, oj = i / kTcPrepSplit;
    const int o = oj / nb, j = oj - o * nb;
    uint8_t *col = p.rec[k] + (int64_t)j * tc_col_bytes(noct);
    build_tc_record(p.x[k], p.ntok, nb, o, j, q, col + o * kTcFragOctBytes,
                    reinterpret_cast<float *>(col + noct * kTcFragOctBytes), threadIdx.x & 31,
                    smax);
}

}  // namespace kq

namespace {

thread_local int g_last_cuda_error = 0;
thread_local int g_last_kernels = 0;   // kq_last_kernels
thread_local int g_last_launches = 0;  // kq_last_launch_count

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

// ---------------------------------------------------------------- memory
// Where each pointer may point: W into device memory of the current device
// (the weight stream uses TMA); x and y into device memory of the current
// device, managed memory, or host memory mapped into the device's address
// space (pinned: cudaHostAlloc / cudaHostRegister), which the kernels read
// and write in place over the host link.  `alias` is the address the device
// uses.  A failed query is KQ_ERR_CUDA; anything else is KQ_ERR_MEMORY.
kq_status device_address(const void *p, int dev, bool host_ok, const void **alias,
                         bool *in_host) {
    *in_host = false;
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
        if (a.device != dev) return KQ_ERR_MEMORY;
        *alias = p;
        return KQ_OK;
    case cudaMemoryTypeManaged:
        *alias = p;
        return KQ_OK;
    case cudaMemoryTypeHost:
        if (!host_ok || !a.devicePointer) return KQ_ERR_MEMORY;
        *alias = a.devicePointer;
        *in_host = true;
        return KQ_OK;
    default:
        return KQ_ERR_MEMORY;
    }
}

// The set with every pointer checked and replaced by its device address;
// a pointer that repeats (a shared x) is looked up once.  x_host[i]: member
// i's x is in host memory.
kq_status resolve_set(const kq_mat *mats, int n, int dev, kq_mat *out, bool *x_host) {
    for (int i = 0; i < n; ++i) {
        out[i] = mats[i];
        x_host[i] = false;
        for (int k = 0; k < 3; ++k) {
            const void *p = k == 0 ? mats[i].W : k == 1 ? (const void *)mats[i].x : (const void *)mats[i].y;
            const void *q = nullptr;
            bool host = false;
            for (int j = 0; j < i && !q; ++j) {
                if (mats[j].W == p) q = out[j].W;
                else if ((const void *)mats[j].x == p) q = out[j].x, host = x_host[j];
                else if ((const void *)mats[j].y == p) q = out[j].y;
            }
            if (!q) {
                const kq_status st = device_address(p, dev, k != 0, &q, &host);
                if (st != KQ_OK) return st;
            }
            if (k == 1) x_host[i] = host;
            if (k == 0) out[i].W = q;
            else if (k == 1) out[i].x = static_cast<const float *>(q);
            else out[i].y = static_cast<float *>(const_cast<void *>(q));
        }
    }
    return KQ_OK;
}

// ---------------------------------------------------------------- device
struct DeviceInfo {
    int sms = 0;
    int smem_optin = 0;       // dynamic shared memory a CTA may opt into
    unsigned int *err = nullptr;  // device address of g_kq_device_error
    bool ok = false;
};

// Per-device facts, looked up on the first call made with that device
// current (that first call should come before any stream capture).
cudaError_t device_info(int dev, DeviceInfo &out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    DeviceInfo &d = cache[dev];
    if (!d.ok) {
        cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaGetSymbolAddress((void **)&d.err, g_kq_device_error);
        if (e != cudaSuccess) return e;
        d.ok = true;
    }
    out = d;
    return cudaSuccess;
}

constexpr int kSmemLimit = kqlaunch::kDirectSmemLimit;

// Input records of each member in global memory, for the kernels that do
// not build them in shared memory: one stream-ordered allocation, written
// by kq_xprep and released (in stream order) after the kernel that reads
// them.
// ------------------------------------------------------------ workspace
// The caller's device workspace of one kq_matvec_set_ws call: the call's
// temporaries are carved from it instead of allocated.  Regions, in the
// order the call takes them: staged host inputs, tensor-core fragments,
// then the dp4a input records, whose region each token chunk reuses (a
// chunk's record pass is an ordinary launch, so it starts only after the
// kernel before it -- the previous chunk's matvec -- has finished).
struct Arena {
    uint8_t *base = nullptr;
    int64_t size = 0, used = 0, chunk_mark = 0;
};
thread_local Arena *g_arena = nullptr;

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

// `bytes` of device memory for the current call: from the caller's
// workspace when one is active (*owned = false), else a stream-ordered
// temporary (*owned = true; the caller frees it on `s`).
cudaError_t call_alloc(void **p, int64_t bytes, cudaStream_t s, bool *owned) {
    *owned = false;
    if (g_arena) {
        const int64_t b = round256(bytes);
        // kq_matvec_set_ws checked the size against kq_workspace_bytes, an
        // upper bound of what a call takes: this does not fail
        if (g_arena->used + b > g_arena->size) return cudaErrorMemoryAllocation;
        *p = g_arena->base + g_arena->used;
        g_arena->used += b;
        return cudaSuccess;
    }
    const cudaError_t e = cudaMallocAsync(p, (size_t)bytes, s);
    *owned = e == cudaSuccess;
    return e;
}

struct GlobalRecords {
    uint8_t *buf = nullptr;
    bool owned = false;  // a stream-ordered temporary (else the workspace's)
    const uint8_t *rec[KQ_MAX_SET] = {};
};

cudaError_t prepare_records(const kq_mat *mats, int n, int ntok, cudaStream_t s,
                            GlobalRecords &out) {
    kq::PrepParams p{};
    p.n = n;
    p.ntok = ntok;
    int64_t off[KQ_MAX_SET], total = 0, warps = 0;
    for (int i = 0; i < n; ++i) {
        const int nb = (int)(mats[i].cols / 256);
        const bool q6 = mats[i].fmt == KQ_Q6_K;
        off[i] = total;
        total += ((int64_t)ntok * nb * kq::rec_bytes(q6) + 255) / 256 * 256;
        p.x[i] = mats[i].x;
        p.nb[i] = nb;
        p.q6[i] = q6 ? 1 : 0;
        p.first_warp[i] = warps;
        warps += (int64_t)ntok * nb * 2;
    }
    p.first_warp[n] = warps;
    cudaError_t e = call_alloc((void **)&out.buf, total, s, &out.owned);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < n; ++i) {
        p.rec[i] = out.buf + off[i];
        out.rec[i] = p.rec[i];
    }
    const int64_t blocks = (warps * 32 + kq::kPrepThreads - 1) / kq::kPrepThreads;
    kq::kq_xprep<<<(unsigned)blocks, kq::kPrepThreads, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        if (out.owned) cudaFreeAsync(out.buf, s);
        out.buf = nullptr;
    }
    return e;
}

// Plan and launch the direct-load kernel (any shape).
kq_status run_direct(const kq_mat *mats, int n, int ntok, cudaStream_t s,
                     const DeviceInfo &info) {
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
    GlobalRecords gr;
    cudaError_t e = prepare_records(mats, n, ntok, s, gr);
    if (e == cudaSuccess) {
        for (int i = 0; i < n; ++i) p.m[i].rec = gr.rec[i];
        e = kqlaunch::direct(ntok, p, (int)grid, smem, s);
        const cudaError_t ef = gr.owned ? cudaFreeAsync(gr.buf, s) : cudaSuccess;
        if (e == cudaSuccess) e = ef;
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    g_last_kernels = 1 | 4;
    g_last_launches = 2;
    return KQ_OK;
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
    });
    return fn;
}

struct MapKey {
    uintptr_t W;
    int64_t rows, row_bytes;
    int box_w, box_h;
    bool operator==(const MapKey &o) const {
        return W == o.W && rows == o.rows && row_bytes == o.row_bytes && box_w == o.box_w &&
               box_h == o.box_h;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const {
        size_t h = (size_t)k.W * 0x9E3779B97F4A7C15ull;
        h ^= (size_t)k.rows + 0x1234567 + (h << 6) + (h >> 2);
        h ^= (size_t)k.row_bytes + (h << 6) + (h >> 2);
        h ^= (size_t)(k.box_w * 977 + k.box_h) + (h << 6) + (h >> 2);
        return h;
    }
};

// A 2-D map over a row-major byte matrix viewed as [rows][row_bytes/8] u64,
// box [box_h rows][box_w u64]; boxes past the last column are zero-filled.
// Encoded maps are cached by (W, shape, box): encoding is a host-only call.
bool tensor_map(const void *W, int64_t rows, int64_t row_bytes, int box_w, int box_h,
                CUtensorMap *out) {
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    const MapKey key{(uintptr_t)W, rows, row_bytes, box_w, box_h};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            return true;
        }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    CUtensorMap m;
    cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / 8), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_h};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(W), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, m);
    *out = m;
    return true;
}

// Launch overlap with the preceding kernel (kq_set_overlap).
std::atomic<int> g_overlap{0};
// Wall-time limit of the streaming kernel's waits (kq_set_wait_limit_ns;
// 0: the default).
std::atomic<unsigned long long> g_wait_ns{0};

// Plan the streaming kernel.  Returns KQ_OK after launching, or
// KQ_ERR_SHAPE when the shapes cannot be staged (caller falls back).
kq_status run_stream(const kq_mat *mats, int n, int ntok, cudaStream_t s,
                     const DeviceInfo &info, bool after_stage, bool *launched) {
    *launched = false;
    static kq::StreamParams p;  // ~10 KB: kept off the stack
    static std::mutex pmu;
    std::lock_guard<std::mutex> plock(pmu);
    memset(&p, 0, sizeof(p));
    p.n = n;

    // launch geometry (kq_plan.cu)
    kqplan::Plan P;
    const kq_status ps = kqplan::plan_stream(mats, n, ntok, info.sms, info.smem_optin, &P);
    if (ps != KQ_OK) return ps;
    for (int i = 0; i < n; ++i) {
        const kq_mat &m = mats[i];
        const kqplan::Member &Q = P.m[i];
        kq::StreamMember &M = p.m[i];
        M.W = (const uint8_t *)m.W;
        M.x = m.x;
        M.rec = nullptr;
        M.y = m.y;
        M.rows = m.rows;
        M.nb = (int)(m.cols / 256);
        M.fmt = m.fmt;
        M.cta_begin = Q.cta_begin;
        M.ncta = Q.ncta;
        M.rows_q = Q.rows_q;
        M.rows_r = Q.rows_r;
        for (int big = 0; big < 2; ++big) {
            M.ng[big] = Q.ng[big];
            M.gq[big] = Q.gq[big];
            M.gr[big] = Q.gr[big];
        }
        M.rmax = Q.rmax;
        M.kb = Q.kb;
        M.seg = Q.seg;
        M.q6_whole = Q.whole;
        M.nmaps = m.fmt == KQ_Q6_K ? 0 : Q.nh;
        if (m.fmt != KQ_Q6_K) {
            // one tensor map per group height: boxes [h][kb * BB / 8] of u64
            const int box_w = (int)(Q.kb * block_bytes_of(m.fmt) / 8);
            for (int j = 0; j < Q.nh; ++j) {
                M.map_h[j] = Q.hs[j];
                if (!tensor_map(m.W, m.rows, Q.row_bytes, box_w, Q.hs[j], &p.maps[i][j]))
                    return KQ_ERR_SHAPE;
            }
        }
    }
    const bool xsmem = P.xsmem;
    const int cta = P.grid;
    p.nslot = (int)P.nslot;
    p.slot_bytes = (int)P.slot_bytes;
    p.x_bytes = (int)P.x_bytes;
    p.part_bytes = (int)P.part_bytes;
    p.part_bufs = P.part_bufs;
    // Launch overlap: as set by kq_set_overlap, and always right after the
    // staging kernel, which writes nothing this launch reads before its
    // griddepcontrol.wait.
    p.overlap = (g_overlap.load() || after_stage) ? 1 : 0;
    for (int hp = 1; hp <= kq::kMaxHinv; ++hp) p.hinv[hp] = ((1u << 20) + hp - 1) / hp;
    p.hinv[0] = 1u << 20;
    p.err = info.err;
    const unsigned long long wl = g_wait_ns.load();
    p.wait_ns = wl ? wl : kq::kWaitLimitNs;
    const size_t smem = (size_t)P.smem;
    // 15 consumer warps for tall Q6_K sets at one token column, one row a
    // lane-task when they are staged in row segments
    const bool tall = kqplan::stream_consumers(P, mats, n) == kq::kStreamConsumersTall;
    const int rpt = kqplan::stream_rows_per_lane(P, mats, n);
    *launched = true;
    GlobalRecords gr;
    cudaError_t e = cudaSuccess;
    if (!xsmem) {
        e = prepare_records(mats, n, ntok, s, gr);
        for (int i = 0; i < n; ++i) p.m[i].rec = gr.rec[i];
    }
    if (e == cudaSuccess) {
        e = kqlaunch::stream(ntok, xsmem, p, cta, smem, s, tall, rpt);
        if (gr.owned) {
            const cudaError_t ef = cudaFreeAsync(gr.buf, s);
            if (e == cudaSuccess) e = ef;
        }
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    g_last_kernels = xsmem ? 2 : (2 | 4);
    g_last_launches = xsmem ? 1 : 2;
    return KQ_OK;
}

// ------------------------------------------------------- tensor-core path
// Calls of kq::kTcMinNtok or more token columns (at most 16) run as one
// tensor-core launch (kq_tc.cuh): one pass builds the input fragments of
// each distinct input plane into global memory (kq_xprep_tc), and the
// streaming (or direct-load) kernel reads W once for all the columns.
// KQ_TC=off keeps such calls on the dp4a kernels (measurement only).
int tc_enabled() {
    static std::atomic<int> v{-1};
    int c = v.load();
    if (c < 0) {
        const char *e = getenv("KQ_TC");
        c = (e && !strcmp(e, "off")) ? 0 : 1;
        v.store(c);
    }
    return c;
}

// The arithmetic of a member: the tensor cores for kq::kTcMinNtok or more
// token columns, and for 2 or 3 when the member's dp4a input records
// (ntok x nb x record bytes) would pass kTcRecordBytes and so not stay in
// shared memory (wide matrices: FFN down, draft fc); else dp4a.  A function
// of the format, the columns and ntok alone, so that a set and separate
// calls, or row shards and the whole matrix, choose alike.
constexpr int64_t kTcRecordBytes = 140 * 1024;
bool member_tc(const kq_mat &m, int ntok) {
    if (!tc_enabled()) return false;
    if (ntok >= kq::kTcMinNtok) return true;
    return ntok >= 2 &&
           (int64_t)ntok * (m.cols / 256) * kq::rec_bytes(m.fmt == KQ_Q6_K) > kTcRecordBytes;
}

// Tensor-core records (kq_xtc.cuh) of every member in `buf` (caller-
// provided, or a stream-ordered temporary when buf is null: *owned is then
// set), one per distinct input plane; rec[i]: member i's records.
int64_t tc_records_bytes(const kq_mat *mats, int n, int ntok) {
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        bool seen = false;
        for (int j = 0; j < i && !seen; ++j)
            seen = mats[j].x == mats[i].x && mats[j].cols == mats[i].cols;
        if (!seen) total += (kq::tc_record_bytes(ntok, (int)(mats[i].cols / 256)) + 255) / 256 * 256;
    }
    return total;
}

cudaError_t prepare_tc_records(const kq_mat *mats, int n, int ntok, cudaStream_t s, uint8_t *buf,
                               uint8_t **owned, const uint8_t **rec, bool overlap) {
    *owned = nullptr;
    const int64_t total = tc_records_bytes(mats, n, ntok);
    if (!buf) {
        bool own = false;
        const cudaError_t e = call_alloc((void **)&buf, total, s, &own);
        if (e != cudaSuccess) return e;
        if (own) *owned = buf;
    }
    kq::TcPrepParams p{};
    p.ntok = ntok;
    const int noct = (ntok + 7) / 8;
    int plane_of[KQ_MAX_SET];
    int64_t off = 0, warps = 0;
    for (int i = 0; i < n; ++i) {
        plane_of[i] = -1;
        for (int k = 0; k < p.n && plane_of[i] < 0; ++k)
            if (p.x[k] == mats[i].x && p.nb[k] == (int)(mats[i].cols / 256)) plane_of[i] = k;
        if (plane_of[i] < 0) {
            const int k = p.n++;
            const int nb = (int)(mats[i].cols / 256);
            p.x[k] = mats[i].x;
            p.nb[k] = nb;
            p.rec[k] = buf + off;
            off += (kq::tc_record_bytes(ntok, nb) + 255) / 256 * 256;
            p.first_warp[k] = warps;
            warps += (int64_t)noct * nb * kq::kTcPrepSplit;
            plane_of[i] = k;
        }
        rec[i] = p.rec[plane_of[i]];
    }
    p.first_warp[p.n] = warps;
    const int64_t blocks = (warps * 32 + kq::kTcPrepThreads - 1) / kq::kTcPrepThreads;
    // With `overlap`, the pass is scheduled while the kernel before it
    // still runs and waits for it on the GPU (it writes nothing before that
    // wait), so the launch latency is hidden.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kq::kTcPrepThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kq::kq_xprep_tc, p);
    if (e != cudaSuccess && *owned) {
        cudaFreeAsync(*owned, s);
        *owned = nullptr;
    }
    return e;
}

// Rows per CTA of the direct-load kernel in a tensor-core launch: one
// 16-row tile, fewer when the matrix would not reach every SM or the
// partials would not fit; 0 if not even one row fits.
int64_t direct_tc_rows_per_cta(const kq_mat &m, int ntok, int sms) {
    const int nb = (int)(m.cols / 256);
    const int nt = 8 * ((ntok + 7) / 8);
    int64_t rpc = std::min<int64_t>(16, std::max<int64_t>(1, (m.rows + sms - 1) / sms));
    while (rpc > 0 && kq::direct_smem_bytes(nb, (int)rpc, nt, true) > kSmemLimit) --rpc;
    return rpc;
}

kq_status run_direct_tc(const kq_mat *mats, int n, int ntok, cudaStream_t s,
                        const DeviceInfo &info, const uint8_t *const *rec) {
    kq::SetParams p{};
    p.n = n;
    p.ntok = ntok;
    const int noct = (ntok + 7) / 8;
    int64_t grid = 0;
    size_t smem = 0;
    for (int i = 0; i < n; ++i) {
        const kq_mat &m = mats[i];
        const int nb = (int)(m.cols / 256);
        const int64_t rpc = direct_tc_rows_per_cta(m, ntok, info.sms);
        if (rpc < 1) return KQ_ERR_SHAPE;
        p.m[i].W = (const uint8_t *)m.W;
        p.m[i].x = m.x;
        p.m[i].rec = rec[i];
        p.m[i].y = m.y;
        p.m[i].rows = m.rows;
        p.m[i].nb = nb;
        p.m[i].fmt = m.fmt;
        p.m[i].cta_begin = (int32_t)grid;
        p.m[i].rpc = (int32_t)rpc;
        grid += (m.rows + rpc - 1) / rpc;
        smem = std::max<size_t>(smem, (size_t)kq::direct_smem_bytes(nb, (int)rpc, 8 * noct, true));
        if (grid > 0x7FFFFFFF) return KQ_ERR_SHAPE;
    }
    const cudaError_t e = kqlaunch::direct_tc(noct, p, (int)grid, smem, s);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    g_last_kernels = 1 | 4 | 8;
    g_last_launches = 2;
    return KQ_OK;
}

// The tensor-core streaming launch; with `automatic` (no kernel forced) it
// declines plans where the direct-load kernel is expected to be faster
// (kqplan::tc_stream_preferred), launching nothing.
kq_status run_stream_tc(const kq_mat *mats, int n, int ntok, cudaStream_t s,
                        const DeviceInfo &info, const uint8_t *const *rec, bool automatic,
                        bool *launched) {
    *launched = false;
    static kq::StreamParams p;  // ~10 KB: kept off the stack
    static std::mutex pmu;
    std::lock_guard<std::mutex> plock(pmu);
    memset(&p, 0, sizeof(p));
    p.n = n;
    const int noct = (ntok + 7) / 8;
    kqplan::Plan P;
    const kq_status ps = kqplan::plan_stream(mats, n, ntok, info.sms, info.smem_optin, &P, noct);
    if (ps != KQ_OK) return ps;
    if (automatic && !kqplan::tc_stream_preferred(P)) return KQ_ERR_SHAPE;
    for (int i = 0; i < n; ++i) {
        const kq_mat &m = mats[i];
        const kqplan::Member &Q = P.m[i];
        kq::StreamMember &M = p.m[i];
        M.W = (const uint8_t *)m.W;
        M.x = m.x;
        M.rec = rec[i];
        M.y = m.y;
        M.rows = m.rows;
        M.nb = (int)(m.cols / 256);
        M.fmt = m.fmt;
        M.cta_begin = Q.cta_begin;
        M.ncta = Q.ncta;
        M.rows_q = Q.rows_q;
        M.rows_r = Q.rows_r;
        for (int big = 0; big < 2; ++big) {
            M.ng[big] = Q.ng[big];
            M.gq[big] = Q.gq[big];
            M.gr[big] = Q.gr[big];
        }
        M.rmax = Q.rmax;
        M.kb = Q.kb;
        M.seg = Q.seg;
        M.q6_whole = Q.whole;
        M.nmaps = m.fmt == KQ_Q6_K ? 0 : Q.nh;
        if (m.fmt != KQ_Q6_K) {
            const int box_w = (int)(Q.kb * block_bytes_of(m.fmt) / 8);
            for (int j = 0; j < Q.nh; ++j) {
                M.map_h[j] = Q.hs[j];
                if (!tensor_map(m.W, m.rows, Q.row_bytes, box_w, Q.hs[j], &p.maps[i][j]))
                    return KQ_ERR_SHAPE;
            }
        }
    }
    p.nslot = (int)P.nslot;
    p.slot_bytes = (int)P.slot_bytes;
    p.x_bytes = 0;
    p.part_bytes = (int)P.part_bytes;
    p.part_bufs = P.part_bufs;
    p.scr_bytes = (int)P.scr_bytes;
    p.ntok = ntok;
    // always after the fragment pass, which it overlaps
    p.overlap = 1;
    for (int hp = 1; hp <= kq::kMaxHinv; ++hp) p.hinv[hp] = ((1u << 20) + hp - 1) / hp;
    p.hinv[0] = 1u << 20;
    p.err = info.err;
    const unsigned long long wl = g_wait_ns.load();
    p.wait_ns = wl ? wl : kq::kWaitLimitNs;
    *launched = true;
    const cudaError_t e = kqlaunch::stream_tc(noct, p, P.grid, (size_t)P.smem, s);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    g_last_kernels = 2 | 4 | 8;
    g_last_launches = 2;
    return KQ_OK;
}

// Kernel choice: the streaming kernel when the shapes can be staged, else
// the direct-load kernel.  KQ_KERNEL=direct|stream forces one (testing and
// measurement only; both give bitwise identical results).
std::atomic<int> g_choice{-1};

int kernel_choice() {
    int c = g_choice.load();
    if (c < 0) {
        const char *e = getenv("KQ_KERNEL");
        c = (e && !strcmp(e, "direct")) ? 1 : (e && !strcmp(e, "stream")) ? 2 : 0;
        int expected = -1;
        g_choice.compare_exchange_strong(expected, c);
        c = g_choice.load();
    }
    return c;
}

// Token columns per launch.  A token's result depends on its own input
// plane alone (every kernel treats the ntok columns independently), so a
// call with more columns runs as launches of at most this many, with the
// same results as one launch would give.
constexpr int kLaunchNtok = 8;
// Token columns per launch of kq_matvec / kq_matvec_set, at most: a call
// with more runs as ceil(ntok / limit) launches of near-equal size.  The
// kernels' cost per token column is lowest at 3..5 columns (block sums
// grow with the columns while the unrolled code and its registers grow
// too); on GB300, 4096x6656 matrices, ntok = 8 took 29-39 us as 4 + 4 and
// 40-50 us as one launch.  KQ_LAUNCH_NTOK=1..8 overrides the limit
// (measurement only; the results are the same for every value).
constexpr int kDefaultLaunchNtok = 5;
std::atomic<int> g_launch_ntok{0};

int launch_ntok() {
    int c = g_launch_ntok.load();
    if (c == 0) {
        const char *e = getenv("KQ_LAUNCH_NTOK");
        const int v = e ? atoi(e) : 0;
        c = (v >= 1 && v <= kLaunchNtok) ? v : kDefaultLaunchNtok;
        g_launch_ntok.store(c);
    }
    return c;
}

// The members of a set restricted to token columns [t0, t0 + nt).
void token_chunk(const kq_mat *mats, int n, int t0, kq_mat *out) {
    for (int i = 0; i < n; ++i) {
        out[i] = mats[i];
        out[i].x = mats[i].x + (int64_t)t0 * mats[i].cols;
        out[i].y = mats[i].y + (int64_t)t0 * mats[i].rows;
    }
}

kq_status run_chunk(const kq_mat *mats, int n, int ntok, void *stream, bool after_stage);

// Inputs in host memory: every distinct such x plane (all ntok columns) is
// copied once into one stream-ordered device temporary by kq_xstage, and
// the members read it there instead of across the host link from every CTA.
// *buf is the temporary (nullptr: nothing to stage).
cudaError_t stage_inputs(kq_mat *mats, int n, int ntok, const bool *x_host, cudaStream_t s,
                         void **buf, bool *owned) {
    *buf = nullptr;
    *owned = false;
    kq::StageParams p{};
    const float *planes[KQ_MAX_SET];
    int64_t off[KQ_MAX_SET], total = 0;
    int of[KQ_MAX_SET];  // plane of each member (-1: not staged)
    for (int i = 0; i < n; ++i) {
        of[i] = -1;
        if (!x_host[i]) continue;
        for (int k = 0; k < p.n && of[i] < 0; ++k)
            if (planes[k] == mats[i].x) of[i] = k;
        if (of[i] >= 0) continue;
        of[i] = p.n;
        planes[p.n] = mats[i].x;
        const int64_t n4 = (int64_t)ntok * mats[i].cols / 4;
        p.src[p.n] = reinterpret_cast<const float4 *>(mats[i].x);
        off[p.n] = total;
        total += (n4 * 16 + 255) / 256 * 256;
        p.first[p.n + 1] = p.first[p.n] + n4;
        ++p.n;
    }
    if (p.n == 0) return cudaSuccess;
    cudaError_t e = call_alloc(buf, total, s, owned);
    if (e != cudaSuccess) {
        *buf = nullptr;
        return e;
    }
    for (int k = 0; k < p.n; ++k)
        p.dst[k] = reinterpret_cast<float4 *>(static_cast<uint8_t *>(*buf) + off[k]);
    const int64_t blocks = (p.first[p.n] + kq::kStageThreads - 1) / kq::kStageThreads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kq::kStageThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (g_overlap.load()) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, kq::kq_xstage, p);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    for (int i = 0; i < n; ++i)
        if (of[i] >= 0) mats[i].x = reinterpret_cast<const float *>(p.dst[of[i]]);
    return cudaSuccess;
}

// A validated set with ntok >= kq::kTcMinNtok (device pointers): the
// fragment pass, then one tensor-core launch -- the streaming kernel when
// it can be staged (unless the direct kernel is selected), else the
// direct-load kernel.
kq_status run_tc(const kq_mat *mats, int n, int ntok, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    DeviceInfo info;
    if (e == cudaSuccess) e = device_info(dev, info);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    // the streaming kernel, when forced but unable to take the call, fails
    // before anything is enqueued
    const int choice = kernel_choice();
    bool streamed = false;
    kqplan::Plan PS;
    if (choice != 1) {
        const kq_status ps =
            kqplan::plan_stream(mats, n, ntok, info.sms, info.smem_optin, &PS, (ntok + 7) / 8);
        if (choice == 2 && ps != KQ_OK) return ps;
        streamed = ps == KQ_OK && (choice == 2 || kqplan::tc_stream_preferred(PS));
    }
    // With launch overlap on, the fragment pass overlaps the kernel before
    // it -- except before a streaming launch whose CTAs cycle their ring
    // (more stages than slots): there the early start of this call's CTAs
    // competed with the previous call's last ones (the QKV set at 4-16
    // columns, FFN gate/up and down and draft fc at 8: 2-5% slower), while
    // launches whose whole weight share is in flight at once gained (Q4_K
    // 4096x6656 at ntok 8: 12.96 -> 11.82 us per call).
    const bool overlap = g_overlap.load() && (!streamed || PS.stages <= PS.nslot);
    const uint8_t *rec[KQ_MAX_SET];
    uint8_t *owned = nullptr;
    e = prepare_tc_records(mats, n, ntok, s, nullptr, &owned, rec, overlap);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    kq_status st = KQ_ERR_SHAPE;
    bool launched = false;
    if (choice != 1) st = run_stream_tc(mats, n, ntok, s, info, rec, choice == 0, &launched);
    if (!launched && choice != 2) st = run_direct_tc(mats, n, ntok, s, info, rec);
    e = owned ? cudaFreeAsync(owned, s) : cudaSuccess;
    if (st == KQ_OK && e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        st = KQ_ERR_CUDA;
    }
    return st;
}

kq_status run_set(const kq_mat *in, int n, int ntok, void *stream) {
    const kq_status v = validate_set(in, n, ntok);
    if (v != KQ_OK) return v;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    kq_mat mats[KQ_MAX_SET];
    bool x_host[KQ_MAX_SET];
    const kq_status r = resolve_set(in, n, dev, mats, x_host);
    if (r != KQ_OK) return r;
    cudaStream_t s = (cudaStream_t)stream;
    void *staged = nullptr;
    bool staged_owned = false;
    cudaError_t se = stage_inputs(mats, n, ntok, x_host, s, &staged, &staged_owned);
    if (se != cudaSuccess) {
        if (staged_owned) cudaFreeAsync(staged, s);
        g_last_cuda_error = (int)se;
        return KQ_ERR_CUDA;
    }
    const bool after = staged != nullptr;
    int kernels = 0, launches = after ? 1 : 0;
    kq_status st = KQ_OK;
    // members by arithmetic: normally all alike (one launch); a set that
    // mixes them runs as one launch per arithmetic
    kq_mat tcm[KQ_MAX_SET], dpm[KQ_MAX_SET];
    int ntc = 0, ndp = 0;
    for (int i = 0; i < n; ++i) (member_tc(mats[i], ntok) ? tcm[ntc++] : dpm[ndp++]) = mats[i];
    if (ntc > 0) {
        st = run_tc(tcm, ntc, ntok, s);
        kernels = g_last_kernels;
        launches += g_last_launches;
    }
    if (g_arena) g_arena->chunk_mark = g_arena->used;
    const int cn = launch_ntok();
    // dp4a: near-equal chunks, the first `rem` taking one column more
    const int nch = ndp > 0 ? (ntok + cn - 1) / cn : 0;
    const int base = nch ? ntok / nch : 0, rem = nch ? ntok % nch : 0;
    kq_mat part[KQ_MAX_SET];
    for (int ci = 0, t0 = 0; ci < nch && st == KQ_OK; ++ci) {
        const int nt = base + (ci < rem ? 1 : 0);
        if (g_arena) g_arena->used = g_arena->chunk_mark;  // the chunks share one region
        token_chunk(dpm, ndp, t0, part);
        t0 += nt;
        st = run_chunk(part, ndp, nt, stream, after);
        kernels |= g_last_kernels;
        launches += g_last_launches;
    }
    if (staged_owned) {
        se = cudaFreeAsync(staged, s);
        if (st == KQ_OK && se != cudaSuccess) {
            g_last_cuda_error = (int)se;
            st = KQ_ERR_CUDA;
        }
    }
    if (st != KQ_OK) return st;
    g_last_kernels = kernels;
    g_last_launches = launches;
    return KQ_OK;
}

// One launch's worth (ntok <= kLaunchNtok) of a validated set.
// after_stage: the inputs were just staged by kq_xstage (kernels that can
// overlap it are launched to do so).
kq_status run_chunk(const kq_mat *mats, int n, int ntok, void *stream, bool after_stage) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    DeviceInfo info;
    if (e == cudaSuccess) e = device_info(dev, info);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    const int choice = kernel_choice();
    if (choice != 1) {
        bool launched = false;
        const kq_status st = run_stream(mats, n, ntok, s, info, after_stage, &launched);
        if (launched || choice == 2) return st;
    }
    return run_direct(mats, n, ntok, s, info);
}

// ------------------------------------------------------------ no-alloc path
// kq_matvec_noalloc: the direct-load path with its input records in one
// fixed file-scope device buffer (KQ_NOALLOC_RECORD_BYTES), so the call
// allocates nothing.  The buffer's address is looked up once per device.
static __device__ __align__(256) uint8_t g_kq_noalloc_records[KQ_NOALLOC_RECORD_BYTES];

cudaError_t noalloc_buffer(int dev, uint8_t **out) {
    static std::mutex mu;
    static uint8_t *addr[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_kq_noalloc_records);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<uint8_t *>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

kq_status run_noalloc_chunk(const kq_mat &m, int ntok, void *stream);

kq_status run_noalloc(const kq_mat &in, int ntok, void *stream) {
    const kq_status v = validate_set(&in, 1, ntok);
    if (v != KQ_OK) return v;
    // the records of one launch must fit: the tensor-core fragments of all
    // ntok columns, or the dp4a records of at most kLaunchNtok columns
    const int nb = (int)(in.cols / 256);
    const bool q6 = in.fmt == KQ_Q6_K;
    const bool tc = member_tc(in, ntok);
    const int64_t rec_total = tc ? tc_records_bytes(&in, 1, ntok)
                                 : (int64_t)std::min(ntok, kLaunchNtok) * nb * kq::rec_bytes(q6);
    if (rec_total > KQ_NOALLOC_RECORD_BYTES) return KQ_ERR_LIMIT;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    // host-memory inputs are read in place here: staging them would allocate
    kq_mat m;
    bool x_host = false;
    const kq_status r = resolve_set(&in, 1, dev, &m, &x_host);
    if (r != KQ_OK) return r;
    if (tc) {
        // the fragments into the fixed buffer, then the direct-load kernel
        DeviceInfo info;
        uint8_t *buf = nullptr;
        cudaError_t ce = device_info(dev, info);
        if (ce == cudaSuccess) ce = noalloc_buffer(dev, &buf);
        const uint8_t *rec[1];
        uint8_t *owned = nullptr;
        if (ce == cudaSuccess)
            ce = prepare_tc_records(&m, 1, ntok, (cudaStream_t)stream, buf, &owned, rec,
                                    g_overlap.load());
        if (ce != cudaSuccess) {
            g_last_cuda_error = (int)ce;
            return KQ_ERR_CUDA;
        }
        return run_direct_tc(&m, 1, ntok, (cudaStream_t)stream, info, rec);
    }
    int launches = 0;
    for (int t0 = 0; t0 < ntok; t0 += kLaunchNtok) {
        kq_mat part;
        token_chunk(&m, 1, t0, &part);
        // chunks run in stream order, so they reuse the one buffer in turn
        const kq_status st = run_noalloc_chunk(part, std::min(kLaunchNtok, ntok - t0), stream);
        if (st != KQ_OK) return st;
        launches += g_last_launches;
    }
    g_last_launches = launches;
    return KQ_OK;
}

kq_status run_noalloc_chunk(const kq_mat &m, int ntok, void *stream) {
    const int nb = (int)(m.cols / 256);
    const bool q6 = m.fmt == KQ_Q6_K;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    DeviceInfo info;
    if (e == cudaSuccess) e = device_info(dev, info);
    uint8_t *buf = nullptr;
    if (e == cudaSuccess) e = noalloc_buffer(dev, &buf);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;

    // the record pass, into the fixed buffer
    kq::PrepParams pp{};
    pp.n = 1;
    pp.ntok = ntok;
    pp.x[0] = m.x;
    pp.rec[0] = buf;
    pp.nb[0] = nb;
    pp.q6[0] = q6 ? 1 : 0;
    pp.first_warp[0] = 0;
    pp.first_warp[1] = (int64_t)ntok * nb * 2;
    const int64_t blocks = (pp.first_warp[1] * 32 + kq::kPrepThreads - 1) / kq::kPrepThreads;

    // the direct kernel's plan (rows per CTA as in run_direct)
    kq::SetParams p{};
    p.n = 1;
    int64_t rpc = std::max<int64_t>(1, kq::kDirectThreads / nb);
    rpc = std::min<int64_t>(rpc, 32);
    rpc = std::min<int64_t>(rpc, std::max<int64_t>(1, (m.rows + info.sms - 1) / info.sms));
    const int64_t per_row = (int64_t)nb * ntok * (int64_t)sizeof(float);
    rpc = std::min<int64_t>(rpc, std::max<int64_t>(1, kSmemLimit / per_row));
    if (per_row * rpc > kSmemLimit) return KQ_ERR_SHAPE;
    const int64_t grid = (m.rows + rpc - 1) / rpc;
    if (grid > 0x7FFFFFFF) return KQ_ERR_SHAPE;
    p.m[0].W = (const uint8_t *)m.W;
    p.m[0].x = m.x;
    p.m[0].rec = buf;
    p.m[0].y = m.y;
    p.m[0].rows = m.rows;
    p.m[0].nb = nb;
    p.m[0].fmt = m.fmt;
    p.m[0].cta_begin = 0;
    p.m[0].rpc = (int32_t)rpc;

    kq::kq_xprep<<<(unsigned)blocks, kq::kPrepThreads, 0, s>>>(pp);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = kqlaunch::direct(ntok, p, (int)grid, (size_t)(per_row * rpc), s);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    g_last_kernels = 1 | 4;
    g_last_launches = 2;
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

namespace {
// An upper bound of what run_set takes from a workspace: every member's x
// as if it were staged, the tensor-core members' fragments, and the dp4a
// members' input records for the largest token chunk.
int64_t workspace_need(const kq_mat *mats, int n, int ntok) {
    int64_t stage = 0, dp = 0;
    kq_mat tcm[KQ_MAX_SET];
    int ntc = 0;
    const int nt_chunk = std::min(ntok, kLaunchNtok);
    for (int i = 0; i < n; ++i) {
        const kq_mat &m = mats[i];
        stage += round256((int64_t)ntok * m.cols * (int64_t)sizeof(float));
        if (member_tc(m, ntok))
            tcm[ntc++] = m;
        else
            dp += round256((int64_t)nt_chunk * (m.cols / 256) * kq::rec_bytes(m.fmt == KQ_Q6_K));
    }
    return stage + (ntc ? tc_records_bytes(tcm, ntc, ntok) : 0) + dp;
}
}  // namespace

int64_t kq_workspace_bytes(const kq_mat *mats, int n, int ntok) {
    const kq_status v = validate_set(mats, n, ntok);
    if (v != KQ_OK) return -(int64_t)v;
    return workspace_need(mats, n, ntok);
}

kq_status kq_matvec_set_ws(const kq_mat *mats, int n, int ntok, void *stream, void *ws,
                           int64_t ws_bytes) {
    const kq_status v = validate_set(mats, n, ntok);
    if (v != KQ_OK) return v;
    if (ws_bytes < workspace_need(mats, n, ntok)) return KQ_ERR_LIMIT;
    if (!ws) return KQ_ERR_NULL;
    if ((uintptr_t)ws & 255u) return KQ_ERR_ALIGN;
    const Range rws{(uintptr_t)ws, (uintptr_t)ws + (uintptr_t)ws_bytes};
    for (int i = 0; i < n; ++i)
        if (overlaps(rws, w_range(mats[i])) || overlaps(rws, x_range(mats[i], ntok)) ||
            overlaps(rws, y_range(mats[i], ntok)))
            return KQ_ERR_ALIAS;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    const void *alias = nullptr;
    bool host = false;
    const kq_status wst = device_address(ws, dev, false, &alias, &host);
    if (wst != KQ_OK) return wst;
    Arena a;
    a.base = static_cast<uint8_t *>(ws);
    a.size = ws_bytes;
    g_arena = &a;
    const kq_status st = run_set(mats, n, ntok, stream);
    g_arena = nullptr;
    return st;
}

kq_status kq_dequant_rows(int fmt, const void *W, int64_t rows, int64_t cols,
                          const int32_t *ids, int64_t n, float *out, void *stream) {
    const int64_t bb = block_bytes_of(fmt);
    if (bb < 0) return KQ_ERR_FORMAT;
    if (rows < 1 || rows > KQ_MAX_ROWS || cols < 256 || cols % 256 != 0 || cols > KQ_MAX_COLS ||
        n < 0 || n > 0x7FFFFFFF)
        return KQ_ERR_SHAPE;
    if (n == 0) return KQ_OK;
    if (!W || !ids || !out) return KQ_ERR_NULL;
    if (((uintptr_t)W & 15u) || ((uintptr_t)out & 15u) || ((uintptr_t)ids & 3u))
        return KQ_ERR_ALIGN;
    const Range ro{(uintptr_t)out, (uintptr_t)out + (uintptr_t)(n * cols * (int64_t)sizeof(float))};
    const Range rw{(uintptr_t)W, (uintptr_t)W + (uintptr_t)(rows * (cols / 256) * bb)};
    const Range ri{(uintptr_t)ids, (uintptr_t)ids + (uintptr_t)(n * (int64_t)sizeof(int32_t))};
    if (overlaps(ro, rw) || overlaps(ro, ri)) return KQ_ERR_ALIAS;
    // the same memory rules as kq_matvec: W in this device's memory; ids
    // and out in device, managed or pinned host memory (read / written in
    // place through their device addresses)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    const void *Wd = nullptr, *idsd = nullptr, *outd = nullptr;
    bool host = false;
    kq_status st = device_address(W, dev, false, &Wd, &host);
    if (st == KQ_OK) st = device_address(ids, dev, true, &idsd, &host);
    if (st == KQ_OK) st = device_address(out, dev, true, &outd, &host);
    if (st != KQ_OK) return st;
    e = kqlaunch::rows(fmt, (const uint8_t *)Wd, rows, (int)(cols / 256),
                       static_cast<const int32_t *>(idsd), n,
                       static_cast<float *>(const_cast<void *>(outd)), (cudaStream_t)stream);
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    return KQ_OK;
}

kq_status kq_matvec_noalloc(int fmt, const void *W, int64_t rows, int64_t cols,
                            const float *x, float *y, int ntok, void *stream) {
    kq_mat m;
    m.fmt = fmt;
    m.reserved = 0;
    m.W = W;
    m.rows = rows;
    m.cols = cols;
    m.x = x;
    m.y = y;
    return run_noalloc(m, ntok, stream);
}

const char *kq_status_str(int status) {
    switch (status) {
    case KQ_OK: return "ok";
    case KQ_ERR_FORMAT: return "unknown block format";
    case KQ_ERR_SHAPE: return "invalid or unsupported rows/cols";
    case KQ_ERR_NTOK: return "ntok outside 1..16";
    case KQ_ERR_NULL: return "null pointer";
    case KQ_ERR_ALIGN: return "misaligned pointer (W, x: 16 bytes; y: 4 bytes)";
    case KQ_ERR_ALIAS: return "an output overlaps an input or another output";
    case KQ_ERR_COUNT: return "set size outside 1..16";
    case KQ_ERR_CUDA: return "a CUDA call failed (see kq_last_cuda_error)";
    case KQ_ERR_TIMEOUT: return "device-side wait timed out";
    case KQ_ERR_LIMIT: return "a fixed buffer is too small (kq_matvec_noalloc's, or a kq_matvec_set_ws workspace)";
    case KQ_ERR_MEMORY: return "a pointer addresses memory the device cannot use there";
    default: return "unknown status";
    }
}

int kq_last_cuda_error(void) { return g_last_cuda_error; }

kq_status kq_device_error(int clear) {
    int dev = 0;
    DeviceInfo info;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = device_info(dev, info);
    unsigned int v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, info.err, sizeof(v), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear && v) {
        const unsigned int zero = 0;
        e = cudaMemcpy(info.err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return KQ_ERR_CUDA;
    }
    return v ? KQ_ERR_TIMEOUT : KQ_OK;
}

int kq_select_kernel(int which) {
    const int prev = kernel_choice();
    if (which >= 0 && which <= 2) g_choice.store(which);
    return prev;
}

int kq_last_kernels(void) { return g_last_kernels; }
int kq_last_launch_count(void) { return g_last_launches; }

int kq_set_overlap(int enable) {
    const int prev = g_overlap.load();
    if (enable == 0 || enable == 1) g_overlap.store(enable);
    return prev;
}

int kq_version(void) { return (1 << 16) | 4; }

unsigned long long kq_set_wait_limit_ns(unsigned long long ns) {
    return g_wait_ns.exchange(ns);
}

}  // extern "C"
