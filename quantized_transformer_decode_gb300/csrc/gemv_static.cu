// Split-K GEMV over raw Q8_0 blocks whose scratch memory is a static device
// array: qw3_q8_0_gemv_splitk_noalloc.
//
// Why it exists: some callers must not allocate device memory during a call.
// A serving loop whose device memory is fully reserved by a caching
// allocator has none to give, and cudaMalloc/cudaFree cost latency and
// cudaFree synchronises the whole device, which stalls every other stream of
// the process. This entry needs no allocation: the partial sums and the
// per-row-group arrival counters live in g_splitk_scratch below, whose size
// is fixed when the module loads.
//
// What it computes is qw3_q8_0_gemv's y[b][r] = sum_k W[r][k] x[b][k] (the
// Q8_0 decode of "Model files and quantization", 11.7, dotted with x); only
// the order of the f32 additions differs. The K range of every 8-row group is
// split across CTAs so that matrices with few rows and long rows still fill
// the GPU; each CTA writes its partial sums to the scratch, and the last CTA
// to arrive at a row group (atomic counter) adds the partials in split order
// and writes y, so the result does not depend on CTA timing.
#include <algorithm>
#include <mutex>

#include "qw3_internal.cuh"

namespace qw3 {

namespace {

// Scratch layout: kSplitkMaxGroups u32 arrival counters, then
// kSplitkMaxPartials f32 partial sums. 256 KiB + 4 MiB.
constexpr int kSplitkMaxGroups = 1 << 16;     // 8-row groups: rows <= 524288
constexpr int kSplitkMaxPartials = 1 << 20;   // nsplit * B * rows <= 1048576
constexpr int kSplitkMaxSplit = 64;
constexpr size_t kSplitkCounterBytes = static_cast<size_t>(kSplitkMaxGroups) * 4;
constexpr size_t kSplitkScratchBytes = kSplitkCounterBytes + static_cast<size_t>(kSplitkMaxPartials) * 4;

// The counters must be zero when a call starts. Static device storage is
// zero-initialised when the module is loaded, and every call's last CTA of a
// row group puts that group's counter back to zero, so the invariant holds
// from call to call (a call that stopped part-way, e.g. after a device fault,
// would break it; the context is then unusable anyway).
static __device__ __align__(256) unsigned char g_splitk_scratch[kSplitkScratchBytes];

template <int B>
__global__ void __launch_bounds__(256) k_gemv_splitk(const uint8_t *__restrict__ W, int rows, int nbpr,
                                                     const float *__restrict__ x, float *__restrict__ y,
                                                     unsigned int *__restrict__ counters,
                                                     float *__restrict__ partials) {
    __shared__ int last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = blockIdx.x, split = blockIdx.y, nsplit = gridDim.y;
    const int row = group * 8 + warp;
    const int K = nbpr * 32;
    // this split's block range of every row
    const int per = (nbpr + nsplit - 1) / nsplit;
    const int kb0 = min(nbpr, split * per), kb1 = min(nbpr, kb0 + per);
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    if (row < rows) {
        for (int kb = kb0 + lane; kb < kb1; kb += 32) {
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(W + (static_cast<int64_t>(row) * nbpr + kb) * 34);
            const float d = __half2float(__ushort_as_half(blk[0]));
            float part[B];
#pragma unroll
            for (int b = 0; b < B; ++b) part[b] = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint16_t pair = blk[1 + k];
                const float q0 = static_cast<float>(static_cast<int8_t>(pair & 0xff));
                const float q1 = static_cast<float>(static_cast<int8_t>(pair >> 8));
#pragma unroll
                for (int b = 0; b < B; ++b) {
                    const float2 xv = *reinterpret_cast<const float2 *>(x + static_cast<int64_t>(b) * K + kb * 32 + 2 * k);
                    part[b] = fmaf(q0, xv.x, part[b]);
                    part[b] = fmaf(q1, xv.y, part[b]);
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) acc[b] = fmaf(d, part[b], acc[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float s = warp_sum(acc[b]);
        if (lane == 0 && row < rows) partials[(static_cast<size_t>(split) * B + b) * rows + row] = s;
    }
    // publish the partials, then count this CTA in
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = (atomicAdd(&counters[group], 1u) == static_cast<unsigned>(nsplit - 1));
    __syncthreads();
    if (!last) return;
    __threadfence();
    if (row < rows && lane < B) {
        float s = 0.0f;
        for (int sp = 0; sp < nsplit; ++sp) s += __ldcg(&partials[(static_cast<size_t>(sp) * B + lane) * rows + row]);
        y[static_cast<int64_t>(lane) * rows + row] = s;
    }
    if (threadIdx.x == 0) counters[group] = 0u;   // leave the counter at zero for the next call
}

// Device address of g_splitk_scratch, resolved once per device.
std::mutex g_splitk_mu;
void *g_splitk_addr[64] = {nullptr};

cudaError_t splitk_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_splitk_mu);
    if (!g_splitk_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_splitk_scratch);
        if (e != cudaSuccess) return e;
        g_splitk_addr[dev] = p;
    }
    *out = g_splitk_addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace qw3

using namespace qw3;

extern "C" int qw3_q8_0_gemv_splitk_noalloc(const void *W_dev, int32_t rows, int32_t cols, const float *x_dev,
                                            int32_t B, float *y_dev, void *stream) {
    if (!W_dev || !x_dev || !y_dev || rows < 0 || cols < 0 || B < 1 || B > 8) {
        set_thread_error("qw3_q8_0_gemv_splitk_noalloc: null pointer, negative size or B outside 1..8");
        return QW3_ERR_INVALID_ARG;
    }
    if (cols % 32) {
        set_thread_error("qw3_q8_0_gemv_splitk_noalloc: cols must be a multiple of 32");
        return QW3_ERR_SHAPE;
    }
    if ((reinterpret_cast<uintptr_t>(W_dev) & 1u) || (reinterpret_cast<uintptr_t>(x_dev) & 7u) ||
        (reinterpret_cast<uintptr_t>(y_dev) & 3u)) {
        set_thread_error("qw3_q8_0_gemv_splitk_noalloc: W must be 2-byte, x 8-byte and y 4-byte aligned");
        return QW3_ERR_INVALID_ARG;
    }
    const int64_t groups = (static_cast<int64_t>(rows) + 7) / 8;
    if (groups > kSplitkMaxGroups || static_cast<int64_t>(B) * rows > kSplitkMaxPartials) {
        set_thread_error("qw3_q8_0_gemv_splitk_noalloc: rows must be <= 524288 and B*rows <= 1048576 "
                         "(the fixed scratch holds 65536 row groups and 1048576 partial sums)");
        return QW3_ERR_SHAPE;
    }
    if (rows == 0 || cols == 0) {
        if (rows > 0 && cols == 0) {
            for (int b = 0; b < B; ++b)
                QW3_CUDA_TRY(cudaMemsetAsync(y_dev + static_cast<size_t>(b) * rows, 0, static_cast<size_t>(rows) * 4,
                                             static_cast<cudaStream_t>(stream)));
        }
        return QW3_OK;
    }
    void *scratch = nullptr;
    QW3_CUDA_TRY(splitk_scratch(&scratch));
    unsigned int *counters = static_cast<unsigned int *>(scratch);
    float *partials = reinterpret_cast<float *>(static_cast<unsigned char *>(scratch) + kSplitkCounterBytes);

    const int nbpr = cols / 32;
    const int64_t target = 2LL * num_sms();
    int64_t nsplit = (target + groups - 1) / groups;
    nsplit = std::min<int64_t>(nsplit, std::min(nbpr, kSplitkMaxSplit));
    nsplit = std::min<int64_t>(nsplit, kSplitkMaxPartials / (static_cast<int64_t>(B) * rows));
    if (nsplit < 1) nsplit = 1;
    const dim3 grid(static_cast<unsigned>(groups), static_cast<unsigned>(nsplit));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (B) {
        case 1: k_gemv_splitk<1><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        case 2: k_gemv_splitk<2><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        case 3: k_gemv_splitk<3><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        case 4: k_gemv_splitk<4><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        case 5: k_gemv_splitk<5><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        case 6: k_gemv_splitk<6><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        case 7: k_gemv_splitk<7><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
        default: k_gemv_splitk<8><<<grid, 256, 0, s>>>(static_cast<const uint8_t *>(W_dev), rows, nbpr, x_dev, y_dev, counters, partials); break;
    }
    QW3_CUDA_TRY(cudaGetLastError());
    return QW3_OK;
}
