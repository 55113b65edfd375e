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

// Raw-block GEMV, the general path (any cols % 32 == 0, W 2-byte aligned):
// a CTA takes 8 consecutive rows; their bytes are one
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

// Raw-row GEMV, the fast path (cols % 256 == 0 and W 16-byte aligned, so
// every row starts 16-byte aligned: 8 blocks are 272 = 17 * 16 bytes). A
// CTA takes 8 rows, warp w row w. The warp streams its row 32 blocks (1088
// bytes, 68 uint4) per step with 128-bit loads, the next step's loads in
// flight while it computes, through a warp-private shared buffer; lane j
// takes block j of the step. f32 activations (Q8A false): the 32 codes times
// x in f32, times d. Q8A: x is first encoded per 32-block by every CTA into
// shared memory with the 11.7 encoder (codes and f32(f16(d))), and a block
// contributes (d_w * d_a) * i32 dot of the codes (four dp4a over 32 codes),
// "Model files and quantization", 11.9. A lane's blocks add up in f32, the
// lanes of a row in a fixed shuffle order.
template <int B, bool Q8A>
__global__ void __launch_bounds__(256) k_gemv_rows(const uint8_t *__restrict__ W, int rows, int nbpr,
                                                   const float *__restrict__ x, float *__restrict__ y) {
    extern __shared__ uint4 gsm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = nbpr * 32;
    uint4 *buf = gsm + warp * 68;                                   // [8][68] uint4
    uint32_t *xq = reinterpret_cast<uint32_t *>(gsm + 8 * 68);      // Q8A: [B][K / 4] code words
    float *xs = reinterpret_cast<float *>(xq + static_cast<size_t>(B) * K / 4);   // Q8A: [B][nbpr] scales
    if constexpr (Q8A) {
        const int n4 = B * K / 4;
        for (int base = 0; base < n4; base += 256) {   // uniform trip count: all lanes shuffle
            const int i = base + threadIdx.x;
            const bool act = i < n4;
            const float4 u = act ? reinterpret_cast<const float4 *>(x)[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            float amax = fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w)));
            bool bad = !(isfinite(u.x) && isfinite(u.y) && isfinite(u.z) && isfinite(u.w));
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {   // every lane shuffles (no short-circuit)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                const int ob = __shfl_xor_sync(0xffffffffu, static_cast<int>(bad), o);
                bad = bad || ob != 0;
            }
            const float d = __fdiv_rn(amax, 127.0f);
            const float inv = (d == 0.0f) ? 0.0f : __fdiv_rn(1.0f, d);
            auto code = [&](float v) {
                const float p = __fmul_rn(v, inv);
                return static_cast<int>(fminf(fmaxf(roundf(p), -127.0f), 127.0f));
            };
            if (act) {
                xq[i] = pack4_s8(code(u.x), code(u.y), code(u.z), code(u.w));
                if ((i & 7) == 0) xs[i >> 3] = bad ? __int_as_float(0x7fc00000) : __half2float(__float2half_rn(d));
            }
        }
        __syncthreads();
    }
    const int row = blockIdx.x * 8 + warp;
    if (row >= rows) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(W + static_cast<int64_t>(row) * nbpr * 34);
    const int nsteps = (nbpr + 31) / 32;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    uint4 r0, r1, r2;
    auto load = [&](int st) {
        const int nv = min(32, nbpr - st * 32) * 34 / 16;     // uint4 in this step (a multiple of 17)
        const uint4 *p = src + st * 68;
        if (lane < nv) r0 = __ldg(p + lane);
        if (lane + 32 < nv) r1 = __ldg(p + lane + 32);
        if (lane + 64 < nv) r2 = __ldg(p + lane + 64);
    };
    load(0);
    for (int st = 0; st < nsteps; ++st) {
        const int nb = min(32, nbpr - st * 32);
        const int nv = nb * 34 / 16;
        if (lane < nv) buf[lane] = r0;
        if (lane + 32 < nv) buf[lane + 32] = r1;
        if (lane + 64 < nv) buf[lane + 64] = r2;
        __syncwarp();
        if (st + 1 < nsteps) load(st + 1);
        if (lane < nb) {
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(buf) + lane * 17;
            const float dw = __half2float(__ushort_as_half(blk[0]));
            uint32_t wq[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) wq[k] = static_cast<uint32_t>(blk[1 + 2 * k]) | (static_cast<uint32_t>(blk[2 + 2 * k]) << 16);
            const int jb = st * 32 + lane;                        // block index within the row
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if constexpr (Q8A) {
                    const uint32_t *aq = xq + static_cast<size_t>(b) * K / 4 + jb * 8;
                    int dot = 0;
#pragma unroll
                    for (int k = 0; k < 8; ++k) dot = __dp4a(static_cast<int>(wq[k]), static_cast<int>(aq[k]), dot);
                    acc[b] += (dw * xs[b * nbpr + jb]) * static_cast<float>(dot);
                } else {
                    const float4 *xb = reinterpret_cast<const float4 *>(x + static_cast<int64_t>(b) * K + jb * 32);
                    float part = 0.0f;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float4 v = __ldg(xb + k);
                        const uint32_t w4 = wq[k];
                        part = fmaf(static_cast<float>(static_cast<int8_t>(w4 & 0xff)), v.x, part);
                        part = fmaf(static_cast<float>(static_cast<int8_t>((w4 >> 8) & 0xff)), v.y, part);
                        part = fmaf(static_cast<float>(static_cast<int8_t>((w4 >> 16) & 0xff)), v.z, part);
                        part = fmaf(static_cast<float>(static_cast<int8_t>(w4 >> 24)), v.w, part);
                    }
                    acc[b] = fmaf(dw, part, acc[b]);
                }
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const float t = warp_sum(acc[b]);
        if (lane == 0) y[static_cast<int64_t>(b) * rows + row] = t;
    }
}

template <bool Q8A>
cudaError_t launch_rows_t(const uint8_t *W, int rows, int nbpr, const float *x, int B, float *y, cudaStream_t s) {
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    const size_t smem = 8 * 68 * 16 + (Q8A ? static_cast<size_t>(B) * nbpr * (32 + 4) : 0);
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    switch (B) {
#define QW3_ROWS_CASE(n)                                                                              \
    case n:                                                                                           \
        if (smem > 48 * 1024) {                                                                       \
            cudaError_t e = cudaFuncSetAttribute(k_gemv_rows<n, Q8A>,                                 \
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,         \
                                                 static_cast<int>(smem));                             \
            if (e != cudaSuccess) return e;                                                           \
        }                                                                                             \
        k_gemv_rows<n, Q8A><<<grid, 256, smem, s>>>(W, rows, nbpr, x, y);                             \
        break;
        QW3_ROWS_CASE(1) QW3_ROWS_CASE(2) QW3_ROWS_CASE(3) QW3_ROWS_CASE(4)
        QW3_ROWS_CASE(5) QW3_ROWS_CASE(6) QW3_ROWS_CASE(7) QW3_ROWS_CASE(8)
#undef QW3_ROWS_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
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

cudaError_t launch_gemv_raw(const uint8_t *W, int rows, int cols, const float *x, int B, float *y, bool q8act,
                            cudaStream_t s) {
    const int nbpr = cols / 32;
    const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
    if (grid == 0) return cudaSuccess;
    const bool fast = cols % 256 == 0 && (reinterpret_cast<uintptr_t>(W) & 15) == 0 &&
                      (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    if (q8act) {
        if (!fast) return cudaErrorInvalidValue;
        return launch_rows_t<true>(W, rows, nbpr, x, B, y, s);
    }
    if (fast) return launch_rows_t<false>(W, rows, nbpr, x, B, y, s);
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
