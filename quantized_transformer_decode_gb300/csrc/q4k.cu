// Q4_K weights ("Model files and quantization", 11.8): the encoder, the
// decoder, the embedding gather and the decode GEMV over raw GGUF Q4_K rows.
//
// Block (144 bytes, 256 values): f16 d, f16 dmin, 12 bytes holding eight
// 6-bit sub-scales sc_j and eight 6-bit sub-mins m_j (bytes 0-3: sc_0..3 in
// the low six bits, the top two bits of sc_4..7 above them; bytes 4-7: the
// same for the mins; bytes 8-11: low nibble sc_4..7 & 15, high nibble
// m_4..7 & 15), then 128 bytes of 4-bit codes (byte 32c + l: value 64c + l in
// the low nibble, value 64c + 32 + l in the high one). Value i of sub-block
// j = i / 32: (d * sc_j) * q - dmin * m_j in f32 (both products exact, one
// rounding).
#include <algorithm>

#include "qw3_internal.cuh"

namespace qw3 {

namespace {

constexpr int kQK = 256;
constexpr int kQ4Bytes = 144;

// One warp per block: lane l holds values 8l .. 8l + 7 (sub-block l / 4).
// The encoder of the oracle, step for step in f32: per sub-block lo =
// min(0, min x), S = (max x - lo) / 15, O = 0 - lo; d = max S / 63, dmin =
// max O / 63 as f16; sc = round(S / d16), m = round(O / dmin16) in [0, 63]
// (0 when the stored scale is 0); q = round((x + dmin16 * m) / (d16 * sc)) in
// [0, 15] (0 when d16 * sc is 0); halves away from zero. A block holding NaN
// or inf is written as zero bytes and reported.
__global__ void __launch_bounds__(256) k_q4k_quantize(const float *__restrict__ x, int64_t nb,
                                                      uint8_t *__restrict__ out, int32_t *status) {
    const int64_t blk = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (blk >= nb) return;   // whole warps: blockDim is a multiple of 32
    uint8_t *b = out + blk * kQ4Bytes;
    float v[8];
    const float4 a0 = reinterpret_cast<const float4 *>(x + blk * kQK + 8 * lane)[0];
    const float4 a1 = reinterpret_cast<const float4 *>(x + blk * kQK + 8 * lane)[1];
    v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w; v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
    bool fin = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) fin = fin && isfinite(v[i]);
    if (!__all_sync(0xffffffffu, fin)) {
        reinterpret_cast<uint32_t *>(b)[lane] = 0;        // 128 of the 144 bytes
        if (lane < 4) reinterpret_cast<uint32_t *>(b)[32 + lane] = 0;
        if (lane == 0) record_status(status, QW3_ERR_NONFINITE);
        return;
    }
    float mn = v[0], mx = v[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        mn = fminf(mn, v[i]);
        mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float lo = fminf(0.0f, mn);
    const float S = __fdiv_rn(__fsub_rn(mx, lo), 15.0f);
    const float O = __fsub_rn(0.0f, lo);
    float smax = S, omax = O;
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        omax = fmaxf(omax, __shfl_xor_sync(0xffffffffu, omax, o));
    }
    const __half d16 = __float2half_rn(__fdiv_rn(smax, 63.0f));
    const __half m16 = __float2half_rn(__fdiv_rn(omax, 63.0f));
    const float d32 = __half2float(d16), m32 = __half2float(m16);
    const int sc = d32 > 0.0f ? static_cast<int>(fminf(fmaxf(roundf(__fdiv_rn(S, d32)), 0.0f), 63.0f)) : 0;
    const int mm = m32 > 0.0f ? static_cast<int>(fminf(fmaxf(roundf(__fdiv_rn(O, m32)), 0.0f), 63.0f)) : 0;
    const float Se = __fmul_rn(d32, static_cast<float>(sc));
    const float Oe = __fmul_rn(m32, static_cast<float>(mm));
    uint32_t qlo = 0, qhi = 0;   // the lane's 8 codes, 4 bits each
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = 0;
        if (Se > 0.0f) q = static_cast<int>(fminf(fmaxf(roundf(__fdiv_rn(__fadd_rn(v[i], Oe), Se)), 0.0f), 15.0f));
        if (i < 4) qlo |= static_cast<uint32_t>(q) << (8 * i);
        else qhi |= static_cast<uint32_t>(q) << (8 * (i - 4));
    }
    // lane l (l % 8 < 4) owns bytes 32 (l / 8) + 8 (l % 8) .. + 8: its codes in
    // the low nibbles, lane l + 4's in the high ones
    const uint32_t plo = __shfl_down_sync(0xffffffffu, qlo, 4);
    const uint32_t phi = __shfl_down_sync(0xffffffffu, qhi, 4);
    if ((lane & 7) < 4) {
        const uint2 w = make_uint2(qlo | (plo << 4), qhi | (phi << 4));
        *reinterpret_cast<uint2 *>(b + 16 + 32 * (lane >> 3) + 8 * (lane & 7)) = w;
    }
    int scs[8], ms[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        scs[j] = __shfl_sync(0xffffffffu, sc, 4 * j);
        ms[j] = __shfl_sync(0xffffffffu, mm, 4 * j);
    }
    if (lane == 0) {
        uint8_t s[12];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            s[j] = static_cast<uint8_t>(scs[j] | ((scs[j + 4] >> 4) << 6));
            s[j + 4] = static_cast<uint8_t>(ms[j] | ((ms[j + 4] >> 4) << 6));
            s[j + 8] = static_cast<uint8_t>((scs[j + 4] & 0xF) | ((ms[j + 4] & 0xF) << 4));
        }
        reinterpret_cast<uint16_t *>(b)[0] = __half_as_ushort(d16);
        reinterpret_cast<uint16_t *>(b)[1] = __half_as_ushort(m16);
#pragma unroll
        for (int w = 0; w < 3; ++w)
            reinterpret_cast<uint32_t *>(b + 4)[w] = static_cast<uint32_t>(s[4 * w]) |
                                                     (static_cast<uint32_t>(s[4 * w + 1]) << 8) |
                                                     (static_cast<uint32_t>(s[4 * w + 2]) << 16) |
                                                     (static_cast<uint32_t>(s[4 * w + 3]) << 24);
    }
}

__global__ void k_q4k_dequantize(const uint8_t *__restrict__ blocks, int64_t n, float *__restrict__ y) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n) return;
    y[i] = q4k_value(blocks + (i >> 8) * kQ4Bytes, static_cast<int>(i & 255));
}

// x[i][:] = the dequantised embedding row tokens[i].
__global__ void __launch_bounds__(256) k_embed_q4k(const int32_t *__restrict__ tokens, const uint8_t *__restrict__ E,
                                                   int H, int vocab, float *__restrict__ x) {
    const int i = blockIdx.x;
    int t = tokens[i];
    t = t < 0 ? 0 : (t >= vocab ? vocab - 1 : t);   // ids are validated on the host
    const uint8_t *row = E + static_cast<size_t>(t) * (H / kQK) * kQ4Bytes;
    for (int k = threadIdx.x; k < H; k += blockDim.x) x[static_cast<size_t>(i) * H + k] = q4k_value(row + (k >> 8) * kQ4Bytes, k & 255);
}

// GEMV over raw Q4_K rows: y[b][r] = sum_k W[r][k] xn[b][k], xn = x or its
// RMSNorm (norm_w). A CTA takes 8 rows, warp w row w. The B input rows are
// staged once per CTA in shared memory (normalised) with their per-32-value
// sums, so that a sub-block contributes d1 * sum(q x) - m1 * sum(x). A warp
// streams its row 8 blocks (1152 bytes, 72 uint4) per step with 128-bit
// loads through a warp buffer, the next step's loads in flight; lane p takes
// (block p / 8, sub-block p % 8) of the step and p + 32.
// Modes: 0 store, 1 add to y (residual), 2 SwiGLU over (gate, up) row pairs
// 2i, 2i + 1 into y[b][i], 3 argmax: y (nullable, or io->logits) stored and
// the packed (value, lowest index) key of each row max'ed into key[b].
template <int B, int MODE>
__global__ void __launch_bounds__(256) k_gemv_q4k(const uint8_t *__restrict__ W, int N, int K,
                                                  const float *__restrict__ x, const float *__restrict__ norm_w,
                                                  float eps, float *y, const DecodeIO *io,
                                                  unsigned long long *__restrict__ key, int R) {
    extern __shared__ __align__(16) float q4sm[];
    float *xs = q4sm;                              // [B][K]
    float *xsum = xs + B * K;                      // [B][K / 32]
    uint4 *wbuf = reinterpret_cast<uint4 *>(xsum + B * (K / 32));   // [8 warps][72]
    __shared__ float red[8][B];
    __shared__ float nsc[B];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nsb = K / kQK;
    // the weights do not depend on the previous kernel: warm L2 with this
    // warp's first row, let the next kernel launch, then wait for the inputs
    {
        const int row0 = blockIdx.x * R * 8 + warp;
        if (row0 < N)
            for (int o = lane * 128; o < nsb * kQ4Bytes; o += 32 * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(W + static_cast<size_t>(row0) * nsb * kQ4Bytes + o));
    }
    pdl_trigger();
    pdl_wait();
    if (MODE == 3 && io && io->logits) y = io->logits;
    // ---- stage the inputs (and their norm scale)
    if (norm_w) {
        for (int b = 0; b < B; ++b) {
            float ss = 0.0f;
            for (int k = tid; k < K; k += 256) ss = fmaf(x[static_cast<size_t>(b) * K + k], x[static_cast<size_t>(b) * K + k], ss);
            ss = warp_sum(ss);
            if (lane == 0) red[warp][b] = ss;
        }
        __syncthreads();
        if (tid < B) {
            float t = 0.0f;
            for (int w = 0; w < 8; ++w) t += red[w][tid];
            nsc[tid] = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
        }
        __syncthreads();
    }
    for (int base = 0; base < B * K / 4; base += 256) {   // uniform trip count: 8-lane sums below
        const int i4 = base + tid;
        const bool act = i4 < B * K / 4;
        float4 u = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (act) {
            const int b = (i4 * 4) / K, k = (i4 * 4) % K;
            u = *reinterpret_cast<const float4 *>(x + static_cast<size_t>(b) * K + k);
            if (norm_w) {
                const float r = nsc[b];
                const float4 w4 = *reinterpret_cast<const float4 *>(norm_w + k);
                u.x = u.x * r * w4.x;
                u.y = u.y * r * w4.y;
                u.z = u.z * r * w4.z;
                u.w = u.w * r * w4.w;
            }
            reinterpret_cast<float4 *>(xs)[i4] = u;
        }
        float s = (u.x + u.y) + (u.z + u.w);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        if (act && (i4 & 7) == 0) xsum[i4 >> 3] = s;
    }
    __syncthreads();
    // ---- the rows: R groups of 8, warp w row w of each
    for (int rg = 0; rg < R; ++rg) {
    const int grp = blockIdx.x * R + rg;
    const int row = grp * 8 + warp;
    float acc[B];
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = 0.0f;
    if (row < N) {
        const uint4 *src = reinterpret_cast<const uint4 *>(W + static_cast<size_t>(row) * nsb * kQ4Bytes);
        uint4 *buf = wbuf + warp * 72;
        const int nsteps = (nsb + 7) / 8;
        uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0, r2 = r0;
        auto load = [&](int st) {
            const int nv = min(8, nsb - st * 8) * 9;   // uint4 in this step
            const uint4 *p = src + st * 72;
            if (lane < nv) r0 = __ldg(p + lane);
            if (lane + 32 < nv) r1 = __ldg(p + lane + 32);
            if (lane + 64 < nv) r2 = __ldg(p + lane + 64);
        };
        load(0);
        for (int st = 0; st < nsteps; ++st) {
            const int nbk = min(8, nsb - st * 8);
            const int nv = nbk * 9;
            if (lane < nv) buf[lane] = r0;
            if (lane + 32 < nv) buf[lane + 32] = r1;
            if (lane + 64 < nv) buf[lane + 64] = r2;
            __syncwarp();
            if (st + 1 < nsteps) load(st + 1);
            const uint8_t *bb = reinterpret_cast<const uint8_t *>(buf);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int p = lane + 32 * h;
                const int sb = p >> 3, j = p & 7;
                if (sb < nbk) {
                    const uint8_t *blk = bb + sb * kQ4Bytes;
                    float d1, m1;
                    q4k_sub(blk, j, d1, m1);
                    const uint4 *cw = reinterpret_cast<const uint4 *>(blk + 16 + 32 * (j >> 1));   // 16-byte aligned
                    const uint4 c0 = cw[0], c1 = cw[1];
                    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    const int shift = (j & 1) * 4;
                    const int col = (st * 8 + sb) * kQK + j * 32;
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const float4 *xb = reinterpret_cast<const float4 *>(xs + b * K + col);
                        float dot = 0.0f;
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            const uint32_t q = words[w] >> shift;
                            const float4 xv = xb[w];
                            dot = fmaf(static_cast<float>(q & 0xF), xv.x, dot);
                            dot = fmaf(static_cast<float>((q >> 8) & 0xF), xv.y, dot);
                            dot = fmaf(static_cast<float>((q >> 16) & 0xF), xv.z, dot);
                            dot = fmaf(static_cast<float>((q >> 24) & 0xF), xv.w, dot);
                        }
                        acc[b] = fmaf(d1, dot, fmaf(-m1, xsum[b * (K / 32) + col / 32], acc[b]));
                    }
                }
            }
            __syncwarp();
        }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) acc[b] = warp_sum(acc[b]);
    if (MODE == 2) {
        __syncthreads();
        if (lane == 0)
#pragma unroll
            for (int b = 0; b < B; ++b) red[warp][b] = acc[b];
        __syncthreads();
        // rows 8c + 2i (gate) and 8c + 2i + 1 (up) -> y[b][4c + i]
        if (tid < 4 * B) {
            const int i = tid % 4, b = tid / 4;
            const int r = grp * 8 + 2 * i;
            if (r + 1 < N) {
                const float g = red[2 * i][b], u = red[2 * i + 1][b];
                y[static_cast<size_t>(b) * (N / 2) + r / 2] = g / (1.0f + expf(-g)) * u;
            }
        }
        continue;
    }
    if (lane == 0 && row < N) {
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float *o = y ? y + static_cast<size_t>(b) * N + row : nullptr;
            if (MODE == 0) *o = acc[b];
            else if (MODE == 1) *o += acc[b];
            else {
                if (o) *o = acc[b];
                atomicMax(&key[b], argmax_pack(acc[b], row));
            }
        }
    }
    }
}

template <int MODE>
cudaError_t gemv_q4k_mode(const uint8_t *W, int N, int K, int B, const float *x, const float *norm_w, float eps,
                          float *y, const DecodeIO *io, unsigned long long *key, bool pdl, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(B) * K * 4 + static_cast<size_t>(B) * (K / 32) * 4 + 8 * 72 * 16;
    // R groups of 8 rows per CTA (a warp's rows run one after the other, so
    // more CTAs of one group each keep more loads in flight: R = 1 measured
    // faster on the 0.6B lm_head than 16)
    const int groups = (N + 7) / 8;
    const int R = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>((groups + R - 1) / R));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (B) {
#define QW3_Q4_CASE(n)                                                                                       \
    case n:                                                                                                  \
        return cudaLaunchKernelEx(&cfg, k_gemv_q4k<n, MODE>, W, N, K, x, norm_w, eps, y, io, key, R);
        QW3_Q4_CASE(1) QW3_Q4_CASE(2) QW3_Q4_CASE(3) QW3_Q4_CASE(4)
        QW3_Q4_CASE(5) QW3_Q4_CASE(6) QW3_Q4_CASE(7) QW3_Q4_CASE(8)
#undef QW3_Q4_CASE
        default: return cudaErrorInvalidValue;
    }
}

template <int MODE>
cudaError_t configure_q4k_mode() {
    cudaError_t e = cudaSuccess;
#define QW3_Q4_CFG(n)                                                                                         \
    if (e == cudaSuccess)                                                                                     \
        e = cudaFuncSetAttribute(k_gemv_q4k<n, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    QW3_Q4_CFG(1) QW3_Q4_CFG(2) QW3_Q4_CFG(3) QW3_Q4_CFG(4) QW3_Q4_CFG(5) QW3_Q4_CFG(6) QW3_Q4_CFG(7) QW3_Q4_CFG(8)
#undef QW3_Q4_CFG
    return e;
}

}  // namespace

size_t q4k_row_bytes(int cols) { return static_cast<size_t>(cols / kQK) * kQ4Bytes; }

bool q4k_gemv_fits(int B, int K) { return B >= 1 && B <= 8 && K % kQK == 0 && static_cast<size_t>(B) * K <= 49152; }

cudaError_t configure_q4k() {
    cudaError_t e = configure_q4k_mode<0>();
    if (e == cudaSuccess) e = configure_q4k_mode<1>();
    if (e == cudaSuccess) e = configure_q4k_mode<2>();
    if (e == cudaSuccess) e = configure_q4k_mode<3>();
    return e;
}

cudaError_t launch_q4k_quantize(const float *x, int64_t nblocks, uint8_t *out, int32_t *status, cudaStream_t s) {
    if (nblocks == 0) return cudaSuccess;
    const int64_t threads = nblocks * 32;
    k_q4k_quantize<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, s>>>(x, nblocks, out, status);
    return cudaGetLastError();
}

cudaError_t launch_q4k_dequantize(const uint8_t *blocks, int64_t nblocks, float *y, cudaStream_t s) {
    const int64_t n = nblocks * kQK;
    if (n == 0) return cudaSuccess;
    k_q4k_dequantize<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(blocks, n, y);
    return cudaGetLastError();
}

cudaError_t launch_embed_q4k(const int32_t *tokens, int M, const uint8_t *E, int H, int vocab, float *x, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    k_embed_q4k<<<M, 256, 0, s>>>(tokens, E, H, vocab, x);
    return cudaGetLastError();
}

cudaError_t launch_gemv_q4k(const uint8_t *W, int N, int K, int B, const float *x, const float *norm_w, float eps,
                            float *y, int mode, const DecodeIO *io, unsigned long long *key, bool pdl,
                            cudaStream_t s) {
    if (!q4k_gemv_fits(B, K) || N <= 0) return cudaErrorInvalidValue;
    switch (mode) {
        case GEMV_STORE: return gemv_q4k_mode<0>(W, N, K, B, x, norm_w, eps, y, io, key, pdl, s);
        case GEMV_RESID: return gemv_q4k_mode<1>(W, N, K, B, x, norm_w, eps, y, io, key, pdl, s);
        case GEMV_SWIGLU: return gemv_q4k_mode<2>(W, N, K, B, x, norm_w, eps, y, io, key, pdl, s);
        case GEMV_ARGMAX: return gemv_q4k_mode<3>(W, N, K, B, x, norm_w, eps, y, io, key, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qw3
