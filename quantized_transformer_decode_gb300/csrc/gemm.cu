// Prefill / batched-decode linear layers: C[M][N] = A[M][K] . W[N][K]^T with
// W a repacked Q8_0 matrix ("A transformer from scratch", 12.5: prefill is
// the compute-bound regime where each weight is reused M times).
//
// SIMT f32 tiles of 64 x 64 x 32 (one Q8_0 block of K per step); the W tile
// is dequantised (d * q, exact in f32) into shared memory. Epilogues: store,
// residual add, SwiGLU over interleaved gate/up columns, and argmax over the
// vocabulary (packed (value, index) keys, lowest index on ties).
#include "qw3_internal.cuh"

namespace qw3 {

namespace {

constexpr int BM = 64, BN = 64, BK = 32;

template <int MODE>
__global__ void __launch_bounds__(256) k_gemm(const float *__restrict__ A, int M, int K, const QMat W,
                                              int N, int rows_pad, float *C,
                                              unsigned long long *__restrict__ argmax_key,
                                              const DecodeIO *io) {
    if (MODE == GEMV_ARGMAX && io) C = io->logits;
    __shared__ __align__(16) float As[BK][BM + 4];
    __shared__ __align__(16) float Ws[BK][BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    // loaders: A: row = tid / 4, k-part = (tid % 4) * 8 ; W: row = tid / 4, 8 codes
    const int lr = tid >> 2, lk = (tid & 3) * 8;
    for (int k0 = 0; k0 < K; k0 += BK) {
        float av[8];
        if (m0 + lr < M) {
            const float4 a0 = *reinterpret_cast<const float4 *>(A + static_cast<size_t>(m0 + lr) * K + k0 + lk);
            const float4 a1 = *reinterpret_cast<const float4 *>(A + static_cast<size_t>(m0 + lr) * K + k0 + lk + 4);
            av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w;
            av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = 0.0f;
        }
        float wv[8];
        const int wr = n0 + lr;
        if (wr < rows_pad) {
            const uint2 q = *reinterpret_cast<const uint2 *>(qm_codes(W, wr, k0 + lk));
            const float d = __half2float(*qm_scale(W, wr, k0));
            const uint32_t w0 = q.x, w1 = q.y;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wv[i] = d * static_cast<float>(static_cast<int8_t>((w0 >> (8 * i)) & 0xff));
                wv[4 + i] = d * static_cast<float>(static_cast<int8_t>((w1 >> (8 * i)) & 0xff));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) wv[i] = 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            As[lk + i][lr] = av[i];
            Ws[lk + i][lr] = wv[i];
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            const float4 a4 = *reinterpret_cast<const float4 *>(&As[k][ty * 4]);
            const float4 w4 = *reinterpret_cast<const float4 *>(&Ws[k][tx * 4]);
            const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
            const float wr4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], wr4[j], acc[i][j]);
        }
    }

    // ---- epilogue
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        const bool mrow = m < M;
        if (MODE == GEMV_ARGMAX) {
            unsigned long long key = 0ull;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (mrow && n < N) {
                    if (C) C[static_cast<size_t>(m) * N + n] = acc[i][j];
                    const unsigned long long kk = argmax_pack(acc[i][j], n);
                    key = kk > key ? kk : key;
                }
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
                key = other > key ? other : key;
            }
            if (tx == 0 && mrow && key) atomicMax(&argmax_key[m], key);
            continue;
        }
        if (!mrow) continue;
        if (MODE == GEMV_SWIGLU) {
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                const int n = n0 + tx * 4 + j;
                if (n < N) {
                    const float g = acc[i][j], u = acc[i][j + 1];
                    C[static_cast<size_t>(m) * (N / 2) + n / 2] = g / (1.0f + expf(-g)) * u;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (n < N) {
                    float *c = C + static_cast<size_t>(m) * N + n;
                    if (MODE == GEMV_RESID) *c += acc[i][j];
                    else *c = acc[i][j];
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_gemm(const float *A, int M, int K, const QMat &W, float *C, int mode,
                        unsigned long long *argmax_key, const DecodeIO *io, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    dim3 grid((W.rows + BN - 1) / BN, (M + BM - 1) / BM);
    switch (mode) {
        case GEMV_STORE: k_gemm<GEMV_STORE><<<grid, 256, 0, s>>>(A, M, K, W, W.rows, W.rows_pad, C, nullptr, nullptr); break;
        case GEMV_RESID: k_gemm<GEMV_RESID><<<grid, 256, 0, s>>>(A, M, K, W, W.rows, W.rows_pad, C, nullptr, nullptr); break;
        case GEMV_SWIGLU: k_gemm<GEMV_SWIGLU><<<grid, 256, 0, s>>>(A, M, K, W, W.rows, W.rows_pad, C, nullptr, nullptr); break;
        case GEMV_ARGMAX: k_gemm<GEMV_ARGMAX><<<grid, 256, 0, s>>>(A, M, K, W, W.rows, W.rows_pad, C, argmax_key, io); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qw3
