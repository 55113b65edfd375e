// Q8_0 codec kernels ("Model files and quantization", section 11.7), the
// repack into the tiled device layout, and the standalone GEMV over raw GGUF
// blocks.
//
// Block wire format: f16 scale d (little endian) then 32 int8 codes, 34 bytes.
// Encoder: amax = max|v|; d = amax / 127 (f32, IEEE division); inv_d = 0 if
// d == 0 else 1 / d (IEEE division); q = clamp(round(v * inv_d), -127, 127)
// with the product rounded once (no FMA contraction) and halves rounded away
// from zero; d stored as an f16 rounded to nearest even. A 0 * inf product
// (d so small that 1/d overflows) encodes as 0; other products saturate.
#include "qw3_internal.cuh"

namespace qw3 {

namespace {

__global__ void k_quantize(const float *__restrict__ x, int64_t nb, uint8_t *__restrict__ out,
                           int32_t *status) {
    const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (blk >= nb) return;
    const float v = x[blk * 32 + lane];
    uint8_t *b = out + blk * 34;
    if (!__all_sync(0xffffffffu, isfinite(v))) {
        if (lane < 17) reinterpret_cast<uint16_t *>(b)[lane] = 0;
        if (lane == 0) record_status(status, QW3_ERR_NONFINITE);
        return;
    }
    const float amax = warp_max(fabsf(v));
    const float d = __fdiv_rn(amax, 127.0f);
    const float inv_d = (d == 0.0f) ? 0.0f : __fdiv_rn(1.0f, d);
    const float prod = __fmul_rn(v, inv_d);
    int q = 0;
    if (!isnan(prod)) q = static_cast<int>(fminf(fmaxf(roundf(prod), -127.0f), 127.0f));
    b[2 + lane] = static_cast<uint8_t>(static_cast<int8_t>(q));
    if (lane == 0) *reinterpret_cast<uint16_t *>(b) = __half_as_ushort(__float2half_rn(d));
}

__global__ void k_dequantize(const uint8_t *__restrict__ blocks, int64_t n, float *__restrict__ y) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint8_t *b = blocks + (i >> 5) * 34;
    const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(b)));
    y[i] = d * static_cast<float>(static_cast<int8_t>(b[2 + (i & 31)]));
}

// One thread per block: raw block (src row r, block j) -> the tiled layout,
// destination row dst_row0 + r * dst_row_stride.
__global__ void k_repack(const uint8_t *__restrict__ raw, int rows, int nbpr, QMat m, int dst_row0,
                         int dst_row_stride) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= static_cast<int64_t>(rows) * nbpr) return;
    const int r = static_cast<int>(t / nbpr);
    const int j = static_cast<int>(t % nbpr);
    const uint16_t *b = reinterpret_cast<const uint16_t *>(raw + t * 34);
    const int dst = dst_row0 + r * dst_row_stride;
    *const_cast<__half *>(qm_scale(m, dst, 32 * j)) = __ushort_as_half(b[0]);
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = static_cast<uint32_t>(b[1 + 2 * k]) | (static_cast<uint32_t>(b[2 + 2 * k]) << 16);
    uint4 *o = reinterpret_cast<uint4 *>(const_cast<int8_t *>(qm_codes(m, dst, 32 * j)));
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// Raw-block GEMV: a CTA takes 8 consecutive rows; their bytes are one
// contiguous range, staged through shared memory 32 blocks (1088 bytes) per
// row at a time with coalesced 2-byte loads; warp w then reduces row w.
template <int B>
__global__ void __launch_bounds__(256) k_gemv_raw(const uint8_t *__restrict__ W, int rows, int nbpr,
                                                  const float *__restrict__ x, float *__restrict__ y) {
    __shared__ uint16_t tile[8 * 32 * 17];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = blockIdx.x * 8;
    const int nrows = min(8, rows - row0);
    const int K = nbpr * 32;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    for (int c0 = 0; c0 < nbpr; c0 += 32) {
        const int nbc = min(32, nbpr - c0);
        const int seg = nbc * 17;  // u16 per row segment
        __syncthreads();
        for (int i = threadIdx.x; i < nrows * seg; i += 256) {
            const int r = i / seg, o = i % seg;
            const uint16_t *src = reinterpret_cast<const uint16_t *>(
                W + (static_cast<int64_t>(row0 + r) * nbpr + c0) * 34);
            tile[r * 32 * 17 + o] = src[o];
        }
        __syncthreads();
        if (warp < nrows && lane < nbc) {
            const uint16_t *blk = tile + warp * 32 * 17 + lane * 17;
            const float dsc = __half2float(__ushort_as_half(blk[0]));
            const int kb = (c0 + lane) * 32;
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
                    const float *xb = x + static_cast<int64_t>(b) * K + kb + 2 * k;
                    part[b] = fmaf(q0, xb[0], part[b]);
                    part[b] = fmaf(q1, xb[1], part[b]);
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) acc[b] = fmaf(dsc, part[b], acc[b]);
        }
    }
    if (warp < nrows) {
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const float s = warp_sum(acc[b]);
            if (lane == 0) y[static_cast<int64_t>(b) * rows + row0 + warp] = s;
        }
    }
}

}  // namespace

cudaError_t launch_quantize(const float *x, int64_t nblocks, uint8_t *out, int32_t *status, cudaStream_t s) {
    if (nblocks == 0) return cudaSuccess;
    const int64_t threads = nblocks * 32;
    const int64_t grid = (threads + 255) / 256;
    k_quantize<<<static_cast<unsigned>(grid), 256, 0, s>>>(x, nblocks, out, status);
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t *blocks, int64_t nblocks, float *y, cudaStream_t s) {
    const int64_t n = nblocks * 32;
    if (n == 0) return cudaSuccess;
    k_dequantize<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(blocks, n, y);
    return cudaGetLastError();
}

cudaError_t launch_repack(const uint8_t *raw, int rows, int cols, const QMat &dst, int dst_row0,
                          int dst_row_stride, cudaStream_t s) {
    const int nbpr = cols / 32;
    const int64_t n = static_cast<int64_t>(rows) * nbpr;
    if (n == 0) return cudaSuccess;
    k_repack<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(raw, rows, nbpr, dst, dst_row0,
                                                                     dst_row_stride);
    return cudaGetLastError();
}

cudaError_t launch_gemv_raw(const uint8_t *W, int rows, int cols, const float *x, int B, float *y,
                            cudaStream_t s) {
    const int nbpr = cols / 32;
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    if (grid == 0) return cudaSuccess;
    switch (B) {
        case 1: k_gemv_raw<1><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 2: k_gemv_raw<2><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 3: k_gemv_raw<3><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 4: k_gemv_raw<4><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 5: k_gemv_raw<5><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 6: k_gemv_raw<6><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 7: k_gemv_raw<7><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        case 8: k_gemv_raw<8><<<grid, 256, 0, s>>>(W, rows, nbpr, x, y); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qw3
