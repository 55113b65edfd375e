// Prefill / batched-decode linear layers: C[M][N] = A[M][K] . W[N][K]^T with
// W a repacked Q8_0 matrix ("A transformer from scratch", 12.5: prefill is
// the compute-bound regime where each weight is reused M times).
//
// SIMT f32 tiles of 64 x 64 x 32 (one Q8_0 block of K per step); the W tile
// is dequantised (d * q, exact in f32) into shared memory. Epilogues: store,
// residual add, SwiGLU over interleaved gate/up columns, and argmax over the
// vocabulary (packed (value, index) keys, lowest index on ties).
#include <cuda_bf16.h>

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
                        unsigned long long *argmax_key, const DecodeIO *io, cudaStream_t s, int32_t *status) {
    if (M <= 0) return cudaSuccess;
    if (gemm_tc_supported(M, K, W)) return launch_gemm_tc(A, M, K, W, C, mode, argmax_key, io, status, s);
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

// ===========================================================================
// Tensor-core path (tcgen05, sm_103a) for the dense contraction: prefill and
// large-batch decode, C[M][N] = A[M][K] . W[N][K]^T.
//
// Exactness plan: int8 codes times an f16 scale need 18 significant bits and
// activations are f32, so both operands are split into bf16 pairs, a = ah + al
// and w = wh + wl (w = d * q formed exactly in f32 first), and each 16-deep
// step issues three MMAs, ah.wh + ah.wl + al.wh, accumulated in f32 in tensor
// memory; the dropped al.wl term and the split residues are ~2^-17 of each
// product, the size of f32 rounding.
//
// CTA tile 128 (activation rows, TMEM lanes) x 128 (weight rows, TMEM
// columns), K steps of 64. Two shared-memory stages of four 128 x 64 bf16
// operands (A hi/lo, W hi/lo) in the no-swizzle K-major core-matrix layout:
// element (r, k) at (r / 8) * 1024 + (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2.
// All 256 threads build the next stage (loads, dequantisation, splits) while
// the tensor core consumes the current one; thread 0 issues the 12 MMAs of a
// step and commits them to the stage's mbarrier, which frees the stage. The
// epilogue reads the accumulator from tensor memory (32x32b loads: warp w
// reads TMEM lanes 32 (w % 4).., columns half (w / 4)).
// ===========================================================================
namespace {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 64;
constexpr int TC_THREADS = 256;
constexpr uint32_t TC_OPERAND = TC_BM * TC_BK * 2;          // 16 KB per bf16 operand
constexpr uint32_t TC_STAGE = 4 * TC_OPERAND;               // A hi, A lo, W hi, W lo
constexpr uint32_t TC_SMEM = 2 * TC_STAGE + 2048;           // + barriers, alignment slack

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
    // start >> 4; leading byte offset 128 (next 8-deep K core); stride byte
    // offset 1024 (next 8-row group); descriptor version 1; no swizzle
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46);
}

// kind::f16 instruction descriptor: f32 accumulator, bf16 A and B, both
// K-major, N = 128, M = 128.
constexpr uint32_t kTcIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((TC_BN >> 3) << 17) | ((TC_BM >> 4) << 24);

__device__ __forceinline__ uint32_t core_off(int r, int k) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// Split 8 consecutive values into their bf16 hi and lo parts, as two uint4.
__device__ __forceinline__ void split8(const float *v, uint4 &hi, uint4 &lo) {
    float h[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
        l[i] = v[i] - h[i];
    }
    hi = make_uint4(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]), pack_bf16(h[4], h[5]), pack_bf16(h[6], h[7]));
    lo = make_uint4(pack_bf16(l[0], l[1]), pack_bf16(l[2], l[3]), pack_bf16(l[4], l[5]), pack_bf16(l[6], l[7]));
}

__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity) { return mbar_wait_bounded(bar, parity); }

template <int MODE>
__global__ void __launch_bounds__(TC_THREADS, 1) k_gemm_tc(const float *__restrict__ A, int M, int K, const QMat W,
                                                           int N, float *C, unsigned long long *__restrict__ argmax_key,
                                                           const DecodeIO *io, int32_t *status) {
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + 2 * TC_STAGE);   // [2]
    uint32_t *tbase = reinterpret_cast<uint32_t *>(base + 2 * TC_STAGE + 64);
    int *err = reinterpret_cast<int *>(base + 2 * TC_STAGE + 128);
    if (MODE == GEMV_ARGMAX && io) C = io->logits;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * TC_BM, n0 = blockIdx.x * TC_BN;
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *err = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tbase)),
                     "r"(TC_BN) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tbase;

    // staging roles: thread t fills row t / 2, columns (t % 2) * 32 .. + 32 of
    // the 128 x 64 A tile and of the 128 x 64 W tile
    const int sr = tid >> 1, sh = (tid & 1) * 32;
    const int am = m0 + sr, wn = n0 + sr;
    const int nsteps = K / TC_BK;
    for (int ks = 0; ks < nsteps; ++ks) {
        const int st = ks & 1;
        uint8_t *sb = base + st * TC_STAGE;
        if (ks >= 2 && !*err && !tc_wait(&bars[st], static_cast<uint32_t>(((ks - 2) >> 1) & 1))) {
            *err = 1;
            record_status(status, QW3_ERR_TIMEOUT);
        }
        const int k0 = ks * TC_BK + sh;
        // activations
        {
            float v[32];
            if (am < M) {
                const float4 *src = reinterpret_cast<const float4 *>(A + static_cast<size_t>(am) * K + k0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 t = src[i];
                    v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 hi, lo;
                split8(v + 8 * j, hi, lo);
                *reinterpret_cast<uint4 *>(sb + core_off(sr, sh + 8 * j)) = hi;
                *reinterpret_cast<uint4 *>(sb + TC_OPERAND + core_off(sr, sh + 8 * j)) = lo;
            }
        }
        // weights: one Q8_0 block of row wn, dequantised exactly, split
        {
            float v[32];
            if (wn < W.rows_pad) {
                const uint4 *q = reinterpret_cast<const uint4 *>(qm_codes(W, wn, k0));
                const float d = __half2float(*qm_scale(W, wn, k0));
                const uint4 c0 = q[0], c1 = q[1];
                const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        v[4 * i + b] = d * static_cast<float>(static_cast<int8_t>((w[i] >> (8 * b)) & 0xffu));
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint4 hi, lo;
                split8(v + 8 * j, hi, lo);
                *reinterpret_cast<uint4 *>(sb + 2 * TC_OPERAND + core_off(sr, sh + 8 * j)) = hi;
                *reinterpret_cast<uint4 *>(sb + 3 * TC_OPERAND + core_off(sr, sh + 8 * j)) = lo;
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> tensor core reads
        __syncthreads();
        if (tid == 0 && !*err) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a_hi = smem_u32(sb), a_lo = a_hi + TC_OPERAND;
            const uint32_t w_hi = a_hi + 2 * TC_OPERAND, w_lo = a_hi + 3 * TC_OPERAND;
#pragma unroll
            for (int sub = 0; sub < TC_BK / 16; ++sub) {
                const uint32_t off = sub * 256;   // two 8-deep K cores per 16-deep step
                const uint32_t acc0 = (ks > 0 || sub > 0) ? 1u : 0u;
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %3, 1;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %2, %3, 1;\n\t}"
                    ::"r"(tmem), "l"(umma_desc(a_hi + off)), "l"(umma_desc(w_hi + off)), "r"(kTcIdesc), "r"(acc0),
                      "l"(umma_desc(w_lo + off)), "l"(umma_desc(a_lo + off))
                    : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&bars[st]))
                         : "memory");
        }
    }
    // the last commit covers every MMA issued before it
    if (nsteps > 0 && !*err) {
        const int last = nsteps - 1;
        if (!tc_wait(&bars[last & 1], static_cast<uint32_t>((last >> 1) & 1))) {
            *err = 1;
            record_status(status, QW3_ERR_TIMEOUT);
        }
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    __syncthreads();

    // ---- epilogue: row m0 + 32 (warp % 4) + lane, columns half (warp / 4)
    const int row = 32 * (warp & 3) + lane;
    const int m = m0 + row;
    const int cbase = (warp >> 2) * (TC_BN / 2);
    unsigned long long best = 0ull;
    for (int c0 = 0; c0 < TC_BN / 2; c0 += 16) {
        uint32_t r[16];
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + static_cast<uint32_t>(cbase + c0);
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
        if (m >= M || *err) continue;
        const int nb = n0 + cbase + c0;
        if (MODE == GEMV_SWIGLU) {
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
                const int n = nb + j;
                if (n < N) {
                    const float g = __uint_as_float(r[j]), u = __uint_as_float(r[j + 1]);
                    C[static_cast<size_t>(m) * (N / 2) + n / 2] = g / (1.0f + expf(-g)) * u;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int n = nb + j;
                if (n < N) {
                    const float y = __uint_as_float(r[j]);
                    float *c = C ? C + static_cast<size_t>(m) * N + n : nullptr;
                    if (MODE == GEMV_STORE) *c = y;
                    else if (MODE == GEMV_RESID) *c += y;
                    else {
                        if (c) *c = y;
                        const unsigned long long k = argmax_pack(y, n);
                        best = k > best ? k : best;
                    }
                }
            }
        }
    }
    if (MODE == GEMV_ARGMAX && m < M && best) atomicMax(&argmax_key[m], best);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_BN) : "memory");
}

template <int MODE>
cudaError_t launch_tc_mode(const float *A, int M, int K, const QMat &W, float *C, unsigned long long *argmax_key,
                           const DecodeIO *io, int32_t *status, cudaStream_t s) {
    const dim3 grid((W.rows + TC_BN - 1) / TC_BN, (M + TC_BM - 1) / TC_BM);
    k_gemm_tc<MODE><<<grid, TC_THREADS, TC_SMEM, s>>>(A, M, K, W, W.rows, C, argmax_key, io, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_gemm_tc() {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<GEMV_STORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<GEMV_RESID>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<GEMV_SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<GEMV_ARGMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    return e;
}

bool gemm_tc_supported(int M, int K, const QMat &W) {
    return M >= kGemmTcMinRows && K % TC_BK == 0 && W.kt % TC_BK == 0 && W.cols == K;
}

cudaError_t launch_gemm_tc(const float *A, int M, int K, const QMat &W, float *C, int mode,
                           unsigned long long *argmax_key, const DecodeIO *io, int32_t *status, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    switch (mode) {
        case GEMV_STORE: return launch_tc_mode<GEMV_STORE>(A, M, K, W, C, argmax_key, io, status, s);
        case GEMV_RESID: return launch_tc_mode<GEMV_RESID>(A, M, K, W, C, argmax_key, io, status, s);
        case GEMV_SWIGLU: return launch_tc_mode<GEMV_SWIGLU>(A, M, K, W, C, argmax_key, io, status, s);
        case GEMV_ARGMAX: return launch_tc_mode<GEMV_ARGMAX>(A, M, K, W, C, argmax_key, io, status, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qw3
