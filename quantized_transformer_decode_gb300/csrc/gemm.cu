// Prefill / batched-decode linear layers: C[M][N] = A[M][K] . W[N][K]^T with
// W a repacked Q8_0 matrix ("A transformer from scratch", 12.5: prefill is
// the compute-bound regime where each weight is reused M times).
//
// SIMT f32 tiles of 64 x 64 x 32 (one Q8_0 block of K per step); the W tile
// is dequantised (d * q, exact in f32) into shared memory. Epilogues: store,
// residual add, SwiGLU over interleaved gate/up columns, and argmax over the
// vocabulary (packed (value, index) keys, lowest index on ties).

#include <algorithm>

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
                        unsigned long long *argmax_key, const DecodeIO *io, cudaStream_t s, int32_t *status,
                        uint8_t *apack, const GemmSplitK *sk) {
    if (M <= 0) return cudaSuccess;
    if (apack && gemm_tc_supported(M, K, W))
        return launch_gemm_tc(A, M, K, W, C, mode, argmax_key, io, status, apack, s, sk);
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
// Exactness plan: int8 codes times an f16 scale need 19 significant bits and
// activations are f32, so both operands are split into fp16 pairs, a = ah + al
// and w = wh + wl, after each row of A and of W is multiplied by its own power
// of two 2^t (row maximum into [2^14, 2^15): no fp16 overflow, small values
// stay normal). d * q * 2^t is then exactly wh + wl; a * 2^t keeps 22 of its
// 24 bits. Each 16-deep step issues three MMAs, ah.wh + ah.wl + al.wh,
// accumulated in f32 in tensor memory (fp16 x fp16 products are exact in
// f32); the dropped al.wl term and the split residue are ~2^-22 of each
// product, the order of f32 rounding itself. The epilogue multiplies C[m][n]
// by 2^-t(m) and 2^-t(n) (exact).
//
// Operands are packed once into "UMMA tiles": 128 rows x 64 K of fp16 in the
// no-swizzle K-major core-matrix layout (element (r, k) at (r / 8) * 1024 +
// (k / 8) * 128 + (r % 8) * 16 + (k % 8) * 2, 16 KB), hi then lo (32 KB), tile
// (row tile t, K step s) at ((t * K / 64 + s) * 32 KB), then the row factors
// (2^t for each padded row, then 2^-t). Q4_K weights are packed at model
// creation (4 bytes per weight); each GEMM input is packed by k_pack_act
// (whose inverse row factors follow its tiles). The GEMM then streams 64 KB per K step (A and
// W, hi and lo) with two 1-D bulk copies into a 3-stage ring; one thread
// issues the 12 MMAs of a step and commits them to the stage's "empty"
// barrier. CTA tile 128 x 128, accumulated in short chains (the accumulator
// promotion below); the epilogue (store / residual / SwiGLU pairs / argmax
// keys) reads it with 32x32b loads. Where 128 x 256 tiles still fill the GPU
// (long prefills), a CTA takes two W tiles per K step against one A tile
// (96 KB per step, 2 stages): a CTA's bulk copies complete at a roughly
// fixed rate, so sharing A raises the work per byte copied. Where the tiles cannot fill the GPU
// (batched decode), K is split over several CTAs that write f32 partial tiles
// to a workspace; k_splitk_reduce sums them in split order and applies the
// epilogue.
// ===========================================================================
namespace {

constexpr int TC_BM = 128, TC_BN = 128, TC_BK = 64;
constexpr int TC_THREADS = 256;   // warp 0 producer, warp 1 MMA, warps 4-7 promotion + epilogue
constexpr uint32_t TC_OPERAND = 128 * TC_BK * 2;            // 16 KB: one fp16 operand tile
constexpr uint32_t TC_PAIR = 2 * TC_OPERAND;                // hi + lo
// NH = 128-column halves of the output tile (1: 128 x 128, 2: 128 x 256 with
// the A tile shared by two N=128 products): a stage holds the A pair and NH
// W pairs; three stages for NH = 1, two for NH = 2.
template <int NH> __host__ __device__ constexpr uint32_t tc_stage() { return (1 + NH) * TC_PAIR; }
template <int NH> __host__ __device__ constexpr int tc_stages() { return NH == 1 ? 3 : 2; }
template <int NH> __host__ __device__ constexpr uint32_t tc_smem() { return tc_stages<NH>() * tc_stage<NH>() + 2048; }

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
    // start >> 4; leading byte offset 128 (next 8-deep K core); stride byte
    // offset 1024 (next 8-row group); descriptor version 1; no swizzle
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46);
}

// kind::f16 instruction descriptor: f32 accumulator (bit 4), fp16 A and B
// (format fields 0), both K-major, N = 128, M = 128.
constexpr uint32_t kTcIdesc = (1u << 4) | ((TC_BN >> 3) << 17) | ((TC_BM >> 4) << 24);

__device__ __forceinline__ uint32_t core_off(int r, int k) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ size_t ut_tile(int t, int s, int ksteps) {
    return (static_cast<size_t>(t) * ksteps + s) * TC_PAIR;
}

__host__ __device__ inline int pad_rows(int rows) { return (rows + TC_BM - 1) / TC_BM * TC_BM; }
// bytes of the operand tiles alone (the row factors follow them)
__host__ __device__ inline size_t ut_tile_bytes(int rows, int K) {
    return static_cast<size_t>(pad_rows(rows)) * static_cast<size_t>(K) * 4;
}

// The row factors of a raw Q4_K matrix (one warp per padded row): row r's
// decoded maximum magnitude sets scale[r] = 2^t, scale[rows + r] = 2^-t
// (padding rows: 1, 1).
__global__ void k_row_exp_q4k(const uint8_t *__restrict__ W, int N, int K, float *__restrict__ scale) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int rows = pad_rows(N);
    if (r >= rows) return;
    float amax = 0.0f;
    if (r < N)
        for (int k = lane; k < K; k += 32)
            amax = fmaxf(amax, fabsf(q4k_value(W + (static_cast<size_t>(r) * (K / 256) + k / 256) * 144, k % 256)));
    amax = warp_max(amax);
    if (lane == 0) {
        const int t = f16_row_exp(amax);
        scale[r] = pow2_f32(t);
        scale[rows + r] = pow2_f32(-t);
    }
}

// One thread per (row, 8-column group): weights of a raw Q4_K matrix (rows of
// K / 256 blocks of 144 bytes), decoded exactly in f32, times the row's
// factor, then split.
__global__ void k_pack_w_q4k(const uint8_t *__restrict__ W, int N, int K, uint8_t *__restrict__ dst) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int groups = K / 8;
    const int rows = pad_rows(N);
    if (i >= static_cast<int64_t>(rows) * groups) return;
    const int r = static_cast<int>(i / groups), k = static_cast<int>(i % groups) * 8;
    const float sr = reinterpret_cast<const float *>(dst + ut_tile_bytes(N, K))[r];
    float v[8];
    if (r < N) {
        const uint8_t *blk = W + (static_cast<size_t>(r) * (K / 256) + k / 256) * 144;
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = q4k_value(blk, (k % 256) + j) * sr;
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    uint4 hi, lo;
    split8_f16(v, hi, lo);
    uint8_t *t = dst + ut_tile(r / TC_BM, k / TC_BK, K / TC_BK);
    *reinterpret_cast<uint4 *>(t + core_off(r % TC_BM, k % TC_BK)) = hi;
    *reinterpret_cast<uint4 *>(t + TC_OPERAND + core_off(r % TC_BM, k % TC_BK)) = lo;
}

// One 128-thread CTA per (padded) row of an f32 activation matrix: the
// row's maximum magnitude sets its factor 2^t; the scaled row is split into
// the fp16 hi/lo tiles and 2^-t goes to inv[row] (padding rows: zero,
// factor 1).
constexpr int kPackActThreads = 128;
__global__ void __launch_bounds__(kPackActThreads) k_pack_act(const float *__restrict__ A, int M, int K,
                                                              uint8_t *__restrict__ dst, float *__restrict__ inv) {
    __shared__ float red[kPackActThreads / 32];
    const int r = blockIdx.x, tid = threadIdx.x;
    const float *row = A + static_cast<size_t>(r) * K;
    float amax = 0.0f;
    if (r < M)
#pragma unroll 4
        for (int k = 4 * tid; k < K; k += 4 * kPackActThreads) {
            const float4 a = *reinterpret_cast<const float4 *>(row + k);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        }
    amax = warp_max(amax);
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const int t = f16_row_exp(amax);
    const float sr = pow2_f32(t);
    if (tid == 0) inv[r] = pow2_f32(-t);
    for (int k = 8 * tid; k < K; k += 8 * kPackActThreads) {
        float v[8];
        if (r < M) {
            const float4 a = *reinterpret_cast<const float4 *>(row + k);
            const float4 b = *reinterpret_cast<const float4 *>(row + k + 4);
            v[0] = a.x * sr; v[1] = a.y * sr; v[2] = a.z * sr; v[3] = a.w * sr;
            v[4] = b.x * sr; v[5] = b.y * sr; v[6] = b.z * sr; v[7] = b.w * sr;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = 0.0f;
        }
        uint4 hi, lo;
        split8_f16(v, hi, lo);
        uint8_t *t8 = dst + ut_tile(r / TC_BM, k / TC_BK, K / TC_BK);
        *reinterpret_cast<uint4 *>(t8 + core_off(r % TC_BM, k % TC_BK)) = hi;
        *reinterpret_cast<uint4 *>(t8 + TC_OPERAND + core_off(r % TC_BM, k % TC_BK)) = lo;
    }
}

// C[m][n] of an accumulator row times the inverse factors of A's row m and of
// W's rows n0 .. n0 + 15 (powers of two: exact unless the true value is out
// of f32 range).
__device__ __forceinline__ void unscale16(float (&v)[16], float am, const float *__restrict__ winv, int n0) {
    const float4 *w4 = reinterpret_cast<const float4 *>(winv + n0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 w = w4[j];
        v[4 * j] = (v[4 * j] * am) * w.x;
        v[4 * j + 1] = (v[4 * j + 1] * am) * w.y;
        v[4 * j + 2] = (v[4 * j + 2] * am) * w.z;
        v[4 * j + 3] = (v[4 * j + 3] * am) * w.w;
    }
}

// ---- Accumulator promotion. The tensor core adds each MMA's products into
// its f32 accumulator with the sum truncated toward zero, so a long chain of
// MMAs into one accumulator shrinks the result: about 1.6e-8 relative per
// MMA, -3.7e-5 over the 2304 MMAs of a 12288-deep product (3 per 16 K). So
// the products sum in short chains. Accumulator tile i (128 TMEM columns: an
// m-tile or an n-half of the CTA's output) takes its K steps in intervals of
// kPromo steps: interval 0 accumulates into the tile's master columns,
// interval j >= 1 into a partial buffer that four promotion warps add into
// the master on the CUDA cores (f32, round to nearest) while the MMAs go on;
// the epilogue adds the last interval's partial. With two tiles, tile 1's
// intervals start half an interval later than tile 0's, and the tile that
// starts an interval (and may wait for its buffer) is issued second, so one
// tile's promotion overlaps the other's MMAs. TMEM: the masters at column
// 128 i, the partial buffers after them (two for one tile, one each for two
// tiles); 512 columns.
constexpr int kPromo = 4;
constexpr uint32_t kPromoCols = 512;
template <int T>
struct PromoPlan {
    static constexpr int NB = T == 1 ? 2 : 1;   // partial buffers per tile
    __device__ static int off(int i) { return (T == 2 && i == 1) ? kPromo / 2 : 0; }
    __device__ static int interval(int i, int ks) { return (ks + off(i)) / kPromo; }
    __device__ static int first(int i, int j) { return max(0, j * kPromo - off(i)); }
    __device__ static int last(int i, int j, int ksteps) { return min(ksteps, (j + 1) * kPromo - off(i)) - 1; }
    __device__ static int count(int i, int ksteps) { return (ksteps - 1 + off(i)) / kPromo + 1; }
    __device__ static uint32_t master_col(int i) { return 128u * static_cast<uint32_t>(i); }
    __device__ static int buf(int i, int j) { return i * NB + (j - 1) % NB; }   // interval j >= 1
    __device__ static uint32_t partial_col(int i, int j) { return 128u * (T + static_cast<uint32_t>(buf(i, j))); }
    __device__ static uint32_t use(int j) { return static_cast<uint32_t>((j - 1) / NB); }   // earlier uses of j's buffer
    // the tile issued n-th at k-step ks
    __device__ static int order(int n, int ks, int ntiles) {
        return (T == 2 && ntiles == 2 && ks > 0 && first(0, interval(0, ks)) == ks) ? 1 - n : n;
    }
};

// master[lane][0..128) += partial[lane][0..128) for this warp's 32 TMEM lanes
// (taddr: lane field and column); completes its stores before returning.
__device__ __forceinline__ void tmem_add_rows(uint32_t master, uint32_t partial) {
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t a[16], b[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
              "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
              "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
              "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
            : "r"(master + c0), "r"(partial + c0)
            : "memory");
#pragma unroll
        for (int j = 0; j < 16; ++j) a[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(b[j]));
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
            ::"r"(master + c0), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]),
              "r"(a[7]), "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15])
            : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// v = master[lane][c .. c + 16) (+ partial[lane][c .. c + 16) when add).
__device__ __forceinline__ void tmem_ld_sum16(uint32_t master, uint32_t partial, bool add, float (&v)[16]) {
    if (add) {
        uint32_t a[16], b[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
              "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
              "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
              "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
            : "r"(master), "r"(partial)
            : "memory");
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(a[j]) + __uint_as_float(b[j]);
        return;
    }
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(master)
        : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

template <int MODE, int NH>
__global__ void __launch_bounds__(TC_THREADS, 1) k_gemm_tc(const uint8_t *__restrict__ Ap, int M, int K,
                                                           const uint8_t *__restrict__ Wp, int N, float *C,
                                                           unsigned long long *__restrict__ argmax_key,
                                                           const DecodeIO *io, int32_t *status, float *ws,
                                                           const float *__restrict__ ainv,
                                                           const float *__restrict__ winv) {
    using Plan = PromoPlan<NH>;
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int TC_STAGES = tc_stages<NH>();
    constexpr uint32_t TC_STAGE = tc_stage<NH>();
    constexpr int BNE = TC_BN * NH;                                                 // output columns per CTA
    uint64_t *full = reinterpret_cast<uint64_t *>(base + TC_STAGES * TC_STAGE);   // [TC_STAGES]
    uint64_t *empty = full + TC_STAGES;                                             // [TC_STAGES]
    uint64_t *pdone = empty + TC_STAGES;                                            // [2] partial complete
    uint64_t *pfree = pdone + 2;                                                    // [2] partial promoted
    uint64_t *done = pfree + 2;                                                     // [1]
    uint32_t *tbase = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *err = reinterpret_cast<volatile int *>(tbase + 1);
    if (MODE == GEMV_ARGMAX && io) C = io->logits;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.y, nt = blockIdx.x;
    // split K over gridDim.z CTAs (small M: too few output tiles to fill the
    // GPU); each takes a contiguous run of k-steps
    const int ksteps_all = K / TC_BK;
    const int kz = blockIdx.z, nks = gridDim.z;
    const int kb = static_cast<int>(static_cast<int64_t>(kz) * ksteps_all / nks);
    const int ksteps = static_cast<int>(static_cast<int64_t>(kz + 1) * ksteps_all / nks) - kb;
    if (tid == 0) {
        for (int i = 0; i < TC_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&pdone[i], 1);
            mbar_init(&pfree[i], 4);
        }
        mbar_init(done, 1);
        *err = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tbase)),
                     "r"(kPromoCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tbase;

    if (warp == 0 && lane == 0) {
        // producer: A tile pair and W tile pair of each K step
        for (int ks = 0; ks < ksteps; ++ks) {
            const int st = ks % TC_STAGES;
            if (ks >= TC_STAGES && !mbar_wait_bounded(&empty[st], static_cast<uint32_t>(((ks / TC_STAGES) - 1) & 1))) {
                *err = 1;
                record_status(status, QW3_ERR_TIMEOUT);
                break;
            }
            if (*err) break;
            uint8_t *sb = base + st * TC_STAGE;
            mbar_arrive_expect_tx(&full[st], TC_STAGE);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(smem_u32(sb)), "l"(Ap + ut_tile(mt, kb + ks, ksteps_all)), "r"(TC_PAIR),
                           "r"(smem_u32(&full[st]))
                         : "memory");
#pragma unroll
            for (int h = 0; h < NH; ++h)
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                             ::"r"(smem_u32(sb + (1 + h) * TC_PAIR)), "l"(Wp + ut_tile(nt * NH + h, kb + ks, ksteps_all)),
                               "r"(TC_PAIR), "r"(smem_u32(&full[st]))
                             : "memory");
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: n-half h's products in promotion intervals (PromoPlan)
        for (int ks = 0; ks < ksteps && !*err; ++ks) {
            const int st = ks % TC_STAGES;
            if (!mbar_wait_bounded(&full[st], static_cast<uint32_t>((ks / TC_STAGES) & 1)) || *err) {
                *err = 1;
                record_status(status, QW3_ERR_TIMEOUT);
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a_hi = smem_u32(base + st * TC_STAGE), a_lo = a_hi + TC_OPERAND;
            for (int n = 0; n < NH; ++n) {
                const int h = Plan::order(n, ks, NH);
                const int j = Plan::interval(h, ks);
                const bool first = Plan::first(h, j) == ks;
                if (first && j >= 1 && Plan::use(j) >= 1) {
                    if (!mbar_wait_bounded(&pfree[Plan::buf(h, j)], (Plan::use(j) - 1) & 1u)) {
                        *err = 1;
                        record_status(status, QW3_ERR_TIMEOUT);
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                }
                const uint32_t w_hi = a_hi + (1 + h) * TC_PAIR, w_lo = w_hi + TC_OPERAND;
                const uint32_t th = tmem + (j == 0 ? Plan::master_col(h) : Plan::partial_col(h, j));
#pragma unroll
                for (int sub = 0; sub < TC_BK / 16; ++sub) {
                    const uint32_t off = sub * 256;   // two 8-deep K cores per 16-deep step
                    const uint32_t acc0 = (!first || sub > 0) ? 1u : 0u;
                    asm volatile(
                        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %3, 1;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %2, %3, 1;\n\t}"
                        ::"r"(th), "l"(umma_desc(a_hi + off)), "l"(umma_desc(w_hi + off)), "r"(kTcIdesc), "r"(acc0),
                          "l"(umma_desc(w_lo + off)), "l"(umma_desc(a_lo + off))
                        : "memory");
                }
                if (j >= 1 && j < Plan::count(h, ksteps) - 1 && Plan::last(h, j, ksteps) == ks)
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     smem_u32(&pdone[Plan::buf(h, j)]))
                                 : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&empty[st]))
                         : "memory");
        }
        // completion of everything issued (commit tracks all prior MMAs)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(done))
                     : "memory");
    } else if (warp >= 4) {
        // promotion warps (TMEM lanes 32 (warp - 4) ..), as in k_gemm_tc_q8;
        // every branch warp-uniform
        const uint32_t lanes = static_cast<uint32_t>(32 * (warp - 4)) << 16;
        bool stop = false;
        for (int ks = 0; ks < ksteps && !stop; ++ks) {
            for (int n = 0; n < NH && !stop; ++n) {
                const int h = Plan::order(n, ks, NH);
                const int j = Plan::interval(h, ks);
                if (j < 1 || j >= Plan::count(h, ksteps) - 1 || Plan::last(h, j, ksteps) != ks) continue;
                const bool ok = !*err && mbar_wait_bounded(&pdone[Plan::buf(h, j)], Plan::use(j) & 1u);
                if (!__all_sync(0xffffffffu, ok)) {
                    *err = 1;
                    record_status(status, QW3_ERR_TIMEOUT);
                    stop = true;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                tmem_add_rows(tmem + lanes + Plan::master_col(h), tmem + lanes + Plan::partial_col(h, j));
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&pfree[Plan::buf(h, j)]);
            }
        }
    }
    __syncwarp();
    // all threads: wait for the accumulators (or give up after 1 s), then the
    // producer's copies must have landed before the CTA may exit
    if (!mbar_wait_bounded(done, 0u)) {
        *err = 1;
        record_status(status, QW3_ERR_TIMEOUT);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0 && *err) {
        // drain copies that may still be in flight (bounded)
        for (int ks = ksteps > TC_STAGES ? ksteps - TC_STAGES : 0; ks < ksteps; ++ks)
            (void)mbar_wait_bounded(&full[ks % TC_STAGES], static_cast<uint32_t>((ks / TC_STAGES) & 1));
    }

    if (warp >= 4) {
        // ---- epilogue: thread (warp, lane) owns row 32 (warp - 4) + lane, all
        // BNE columns: each half's master plus its last interval's partial
        const int row = 32 * (warp - 4) + lane;
        const int m = mt * TC_BM + row;
        const uint32_t lanes = static_cast<uint32_t>(32 * (warp - 4)) << 16;
        unsigned long long best = 0ull;
        auto emit = [&](const float (&v)[16], int c0) {
            if (m >= M || *err) return;
            const int nb = nt * BNE + c0;
            if (MODE == GEMV_SWIGLU) {
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const int n = nb + j;
                    if (n < N) C[static_cast<size_t>(m) * (N / 2) + n / 2] = v[j] / (1.0f + expf(-v[j])) * v[j + 1];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = nb + j;
                    if (n < N) {
                        const float y = v[j];
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
        };
        const int Np = gridDim.x * BNE;   // workspace row stride
        for (int c0 = 0; c0 < BNE; c0 += 16) {
            const int h = c0 / TC_BN, jl = Plan::count(h, ksteps) - 1;
            float v[16];
            tmem_ld_sum16(tmem + lanes + Plan::master_col(h) + (c0 % TC_BN),
                          jl >= 1 ? tmem + lanes + Plan::partial_col(h, jl) + (c0 % TC_BN) : 0u, jl >= 1, v);
            if (m >= M) continue;
            unscale16(v, ainv[m], winv, nt * BNE + c0);
            if (nks > 1) {
                // this split's partial tile (valid rows) to the workspace [z][m][n]
                float4 *w4 = reinterpret_cast<float4 *>(
                    ws + (static_cast<size_t>(kz) * gridDim.y * TC_BM + static_cast<size_t>(m)) * Np + nt * BNE + c0);
#pragma unroll
                for (int j = 0; j < 4; ++j) w4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            } else {
                emit(v, c0);
            }
        }
        if (MODE == GEMV_ARGMAX && m < M && best) atomicMax(&argmax_key[m], best);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPromoCols) : "memory");
}

// ---------------------------------------------------------------------------
// The same product with the weights streamed as Q8_0 (1.0625 bytes per
// weight instead of the 4 of pre-packed fp16 hi/lo tiles). Weights are
// laid out once per (128-row tile t, 64-column K step s) as one 8704-byte
// piece: the 128 x 64 int8 codes, then the 128 x 2 f16 scales; the row
// factors (2^t from 128 times the row's largest block scale) follow the
// pieces. Per K step the producer copies the A pair and that piece into a
// stage; eight converter warps turn the piece into the fp16 hi/lo operand
// pair (q * (d * 2^t) is exact in f32 and in the pair) in one of two operand
// buffers, fence it for the tensor core's async proxy and signal; the MMA
// thread then issues the step's 12 MMAs per m-tile. Stage free = MMA commit + converters done (2
// arrivals); operand buffer free = MMA commit. 512 threads: warp 0 producer,
// warp 1 MMA, warps 4-11 converters (thread c: row c % 128, Q8_0 block
// c / 128 of the step: one scale), warps 12-15 accumulator promotion and the
// epilogue (TMEM lanes 32 (warp - 12) ..).
constexpr uint32_t TQ_RAW = 128 * TC_BK + 128 * 4;              // 8704
// MT m-tiles per CTA share each converted W tile (MT = 2 halves the
// conversion per MMA where there are enough row tiles: prefill)
template <int MT> __host__ __device__ constexpr uint32_t tq_stage() { return (MT * TC_PAIR + TQ_RAW + 1023) / 1024 * 1024; }
template <int MT> __host__ __device__ constexpr int tq_stages() { return MT == 1 ? 3 : 2; }
constexpr int TQ_WBUF = 2;
constexpr int TQ_THREADS = 512;
constexpr int TQ_CONV = 256;   // converter threads
template <int MT>
__host__ __device__ constexpr uint32_t tq_smem() { return tq_stages<MT>() * tq_stage<MT>() + TQ_WBUF * TC_PAIR + 2048 + 1024; }

// The row factors of a repacked Q8_0 matrix (one warp per padded row): 2^t
// for a row bound of 128 times the largest block scale at scale[r], 2^-t at
// scale[rows + r] (padding rows: 1, 1).
__global__ void k_row_exp_q8(const QMat W, int N, int K, float *__restrict__ scale) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int rows = pad_rows(N);
    if (r >= rows) return;
    float dmax = 0.0f;
    if (r < N)
        for (int k = 32 * lane; k < K; k += 32 * 32) dmax = fmaxf(dmax, fabsf(__half2float(*qm_scale(W, r, k))));
    dmax = warp_max(dmax);
    if (lane == 0) {
        const int t = f16_row_exp(128.0f * dmax);
        scale[r] = pow2_f32(t);
        scale[rows + r] = pow2_f32(-t);
    }
}

// One thread per (row, 8-column group) of a repacked Q8_0 matrix -> the
// streamed layout above (rows past N are zero).
__global__ void k_pack_w_q8(const QMat W, int N, int K, uint8_t *__restrict__ dst) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int groups = K / 8;
    const int rows = (N + TC_BM - 1) / TC_BM * TC_BM;
    if (i >= static_cast<int64_t>(rows) * groups) return;
    const int r = static_cast<int>(i / groups), k = static_cast<int>(i % groups) * 8;
    uint8_t *piece = dst + (static_cast<size_t>(r / TC_BM) * (K / TC_BK) + k / TC_BK) * TQ_RAW;
    uint2 c = make_uint2(0, 0);
    if (r < N) c = *reinterpret_cast<const uint2 *>(qm_codes(W, r, k));
    *reinterpret_cast<uint2 *>(piece + (r % TC_BM) * TC_BK + (k % TC_BK)) = c;
    if (k % 32 == 0) {
        const __half sc = r < N ? *qm_scale(W, r, k) : __float2half(0.0f);
        *reinterpret_cast<__half *>(piece + 128 * TC_BK + (r % TC_BM) * 4 + ((k % TC_BK) / 32) * 2) = sc;
    }
}

// The same two steps from raw Q8_0 rows (blocks of 34 bytes: f16 scale, 32
// int8 codes; row r's block b at (r * K / 32 + b) * 34).
__global__ void k_row_exp_q8_raw(const uint8_t *__restrict__ W, int N, int K, float *__restrict__ scale) {
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int rows = pad_rows(N);
    if (r >= rows) return;
    float dmax = 0.0f;
    if (r < N)
        for (int b = lane; b < K / 32; b += 32)
            dmax = fmaxf(dmax, fabsf(__half2float(
                                   *reinterpret_cast<const __half *>(W + (static_cast<size_t>(r) * (K / 32) + b) * 34))));
    dmax = warp_max(dmax);
    if (lane == 0) {
        const int t = f16_row_exp(128.0f * dmax);
        scale[r] = pow2_f32(t);
        scale[rows + r] = pow2_f32(-t);
    }
}

__global__ void k_pack_w_q8_raw(const uint8_t *__restrict__ W, int N, int K, uint8_t *__restrict__ dst) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int groups = K / 8;
    const int rows = pad_rows(N);
    if (i >= static_cast<int64_t>(rows) * groups) return;
    const int r = static_cast<int>(i / groups), k = static_cast<int>(i % groups) * 8;
    uint8_t *piece = dst + (static_cast<size_t>(r / TC_BM) * (K / TC_BK) + k / TC_BK) * TQ_RAW;
    const uint8_t *blk = W + (static_cast<size_t>(r) * (K / 32) + k / 32) * 34;
    uint2 c = make_uint2(0, 0);
    if (r < N) {
        // codes k % 32 .. + 7 of the block, at an even offset: four 2-byte loads
        const uint16_t *cp = reinterpret_cast<const uint16_t *>(blk + 2 + (k % 32));
        c.x = static_cast<uint32_t>(cp[0]) | (static_cast<uint32_t>(cp[1]) << 16);
        c.y = static_cast<uint32_t>(cp[2]) | (static_cast<uint32_t>(cp[3]) << 16);
    }
    *reinterpret_cast<uint2 *>(piece + (r % TC_BM) * TC_BK + (k % TC_BK)) = c;
    if (k % 32 == 0) {
        const __half sc = r < N ? *reinterpret_cast<const __half *>(blk) : __float2half(0.0f);
        *reinterpret_cast<__half *>(piece + 128 * TC_BK + (r % TC_BM) * 4 + ((k % TC_BK) / 32) * 2) = sc;
    }
}

template <int MODE, int MT>
__global__ void __launch_bounds__(TQ_THREADS, 1) k_gemm_tc_q8(const uint8_t *__restrict__ Ap, int M, int K,
                                                             const uint8_t *__restrict__ Wq, int N, float *C,
                                                             unsigned long long *__restrict__ argmax_key,
                                                             const DecodeIO *io, int32_t *status, float *ws,
                                                             const float *__restrict__ ainv,
                                                             const float *__restrict__ wscale) {
    using Plan = PromoPlan<MT>;
    extern __shared__ __align__(1024) uint8_t tq_smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tq_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int TQ_STAGES = tq_stages<MT>();
    constexpr uint32_t TQ_STAGE = tq_stage<MT>();   // MT A pairs, then the Q8_0 piece
    uint8_t *wbuf = base + TQ_STAGES * TQ_STAGE;                                       // [TQ_WBUF] operand pairs
    uint64_t *full = reinterpret_cast<uint64_t *>(wbuf + TQ_WBUF * TC_PAIR);          // [TQ_STAGES]
    uint64_t *empty = full + TQ_STAGES;                                               // [TQ_STAGES]
    uint64_t *wready = empty + TQ_STAGES;                                             // [TQ_WBUF]
    uint64_t *wfree = wready + TQ_WBUF;                                               // [TQ_WBUF]
    uint64_t *wfull = wfree + TQ_WBUF;                                                // [TQ_STAGES] W piece landed
    uint64_t *pdone = wfull + TQ_STAGES;                                              // [2] partial complete
    uint64_t *pfree = pdone + 2;                                                      // [2] partial promoted
    uint64_t *done = pfree + 2;                                                       // [1]
    uint32_t *tbase = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *err = reinterpret_cast<volatile int *>(tbase + 1);
    volatile int *cvok = err + 1;
    if (MODE == GEMV_ARGMAX && io) C = io->logits;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = blockIdx.x;
    const int mtiles = (M + TC_BM - 1) / TC_BM;
    const int mt0 = blockIdx.y * MT;
    const int nmt = min(MT, mtiles - mt0);   // m-tiles this CTA computes
    const int ksteps_all = K / TC_BK;
    const int kz = blockIdx.z, nks = gridDim.z;
    const int kb = static_cast<int>(static_cast<int64_t>(kz) * ksteps_all / nks);
    const int ksteps = static_cast<int>(static_cast<int64_t>(kz + 1) * ksteps_all / nks) - kb;
    if (tid == 0) {
        for (int i = 0; i < TQ_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 2);
            mbar_init(&wfull[i], 1);
        }
        for (int i = 0; i < TQ_WBUF; ++i) {
            mbar_init(&wready[i], 1);
            mbar_init(&wfree[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&pdone[i], 1);
            mbar_init(&pfree[i], 4);
        }
        mbar_init(done, 1);
        *err = 0;
        *cvok = 1;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tbase)),
                     "r"(kPromoCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tbase;

    if (warp == 0 && lane == 0) {
        // producer: the A pairs and the Q8_0 piece of each K step
        for (int ks = 0; ks < ksteps; ++ks) {
            const int st = ks % TQ_STAGES;
            if (ks >= TQ_STAGES && !mbar_wait_bounded(&empty[st], static_cast<uint32_t>(((ks / TQ_STAGES) - 1) & 1))) {
                *err = 1;
                record_status(status, QW3_ERR_TIMEOUT);
                break;
            }
            if (*err) break;
            uint8_t *sb = base + st * TQ_STAGE;
            // the Q8_0 piece first, on its own barrier, so that the converters
            // start while the A pairs are still streaming
            mbar_arrive_expect_tx(&wfull[st], TQ_RAW);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                         ::"r"(smem_u32(sb + MT * TC_PAIR)),
                           "l"(Wq + (static_cast<size_t>(nt) * ksteps_all + kb + ks) * TQ_RAW), "r"(TQ_RAW),
                           "r"(smem_u32(&wfull[st]))
                         : "memory");
            mbar_arrive_expect_tx(&full[st], nmt * TC_PAIR);
            for (int i = 0; i < nmt; ++i)
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                             ::"r"(smem_u32(sb + i * TC_PAIR)), "l"(Ap + ut_tile(mt0 + i, kb + ks, ksteps_all)),
                               "r"(TC_PAIR), "r"(smem_u32(&full[st]))
                             : "memory");
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: m-tile i's products in promotion intervals (PromoPlan)
        for (int ks = 0; ks < ksteps && !*err; ++ks) {
            const int st = ks % TQ_STAGES, wb = ks % TQ_WBUF;
            if (!mbar_wait_bounded(&full[st], static_cast<uint32_t>((ks / TQ_STAGES) & 1)) ||
                !mbar_wait_bounded(&wready[wb], static_cast<uint32_t>((ks / TQ_WBUF) & 1)) || *err) {
                *err = 1;
                record_status(status, QW3_ERR_TIMEOUT);
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t w_hi = smem_u32(wbuf + wb * TC_PAIR), w_lo = w_hi + TC_OPERAND;
            for (int n = 0; n < nmt; ++n) {
                const int i = Plan::order(n, ks, nmt);
                const int j = Plan::interval(i, ks);
                const bool first = Plan::first(i, j) == ks;
                if (first && j >= 1 && Plan::use(j) >= 1) {
                    // the partial buffer must have been promoted
                    if (!mbar_wait_bounded(&pfree[Plan::buf(i, j)], (Plan::use(j) - 1) & 1u)) {
                        *err = 1;
                        record_status(status, QW3_ERR_TIMEOUT);
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                }
                const uint32_t a_hi = smem_u32(base + st * TQ_STAGE + i * TC_PAIR), a_lo = a_hi + TC_OPERAND;
                const uint32_t th = tmem + (j == 0 ? Plan::master_col(i) : Plan::partial_col(i, j));
#pragma unroll
                for (int sub = 0; sub < TC_BK / 16; ++sub) {
                    const uint32_t off = sub * 256;
                    const uint32_t acc0 = (!first || sub > 0) ? 1u : 0u;
                    asm volatile(
                        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %3, 1;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %2, %3, 1;\n\t}"
                        ::"r"(th), "l"(umma_desc(a_hi + off)), "l"(umma_desc(w_hi + off)), "r"(kTcIdesc), "r"(acc0),
                          "l"(umma_desc(w_lo + off)), "l"(umma_desc(a_lo + off))
                        : "memory");
                }
                // a partial interval other than the tile's last is promoted
                if (j >= 1 && j < Plan::count(i, ksteps) - 1 && Plan::last(i, j, ksteps) == ks)
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     smem_u32(&pdone[Plan::buf(i, j)]))
                                 : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&empty[st]))
                         : "memory");
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&wfree[wb]))
                         : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(done))
                     : "memory");
    } else if (warp >= 4 && warp < 12) {
        // converters: thread c converts the 32 codes of block c / 128 of row c % 128
        const int c = tid - 128;
        const int crow = c & 127, cblk = c >> 7;
        const float rs = wscale[nt * TC_BN + crow];   // this row's factor 2^t
        for (int ks = 0; ks < ksteps; ++ks) {
            const int st = ks % TQ_STAGES, wb = ks % TQ_WBUF;
            if (c == 0) {
                bool ok = !*err && mbar_wait_bounded(&wfull[st], static_cast<uint32_t>((ks / TQ_STAGES) & 1));
                if (ok && ks >= TQ_WBUF)
                    ok = mbar_wait_bounded(&wfree[wb], static_cast<uint32_t>(((ks / TQ_WBUF) - 1) & 1));
                if (!ok) {
                    *err = 1;
                    record_status(status, QW3_ERR_TIMEOUT);
                }
                *cvok = ok ? 1 : 0;
            }
            asm volatile("bar.sync 2, 256;" ::: "memory");
            if (!*cvok) break;
            const uint8_t *raw = base + st * TQ_STAGE + MT * TC_PAIR;
            const uint4 *cw = reinterpret_cast<const uint4 *>(raw + crow * TC_BK + cblk * 32);
            const float d = __half2float(*reinterpret_cast<const __half *>(raw + 128 * TC_BK + crow * 4 + cblk * 2)) * rs;
            uint8_t *wo = wbuf + wb * TC_PAIR;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const uint4 w16 = cw[q];   // codes 16q .. 16q + 15 of the block
                const uint32_t words[4] = {w16.x ^ 0x80808080u, w16.y ^ 0x80808080u, w16.z ^ 0x80808080u,
                                           w16.w ^ 0x80808080u};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // int8 -> f32: the biased byte in the mantissa of 2^23 (exact),
                    // times the scaled block scale (exact); then the fp16 hi/lo split
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int pr = 0; pr < 4; ++pr) {
                        const uint32_t wsrc = words[2 * h + pr / 2];
                        const int b0 = 2 * (pr % 2);
                        const float v0 = (__uint_as_float(__byte_perm(wsrc, 0x4B000000u, 0x7540u + b0)) - 8388736.0f) * d;
                        const float v1 =
                            (__uint_as_float(__byte_perm(wsrc, 0x4B000000u, 0x7540u + b0 + 1)) - 8388736.0f) * d;
                        const __half2 h2 = __floats2half2_rn(v0, v1);
                        const float2 hf = __half22float2(h2);
                        const __half2 l2 = __floats2half2_rn(v0 - hf.x, v1 - hf.y);
                        hw[pr] = *reinterpret_cast<const uint32_t *>(&h2);
                        lw[pr] = *reinterpret_cast<const uint32_t *>(&l2);
                    }
                    const int k = 32 * cblk + 16 * q + 8 * h;
                    *reinterpret_cast<uint4 *>(wo + core_off(crow, k)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(wo + TC_OPERAND + core_off(crow, k)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("bar.sync 2, 256;" ::: "memory");
            if (c == 0) {
                mbar_arrive(&wready[wb]);
                mbar_arrive(&empty[st]);
            }
        }
    } else if (warp >= 12) {
        // promotion warps (TMEM lanes 32 (warp - 12) ..): each finished partial
        // interval of a tile (not its last) into the tile's master, in the
        // order the MMA thread completes them
        // (every branch warp-uniform: the TMEM accesses are warp-collective)
        const uint32_t lanes = static_cast<uint32_t>(32 * (warp - 12)) << 16;
        bool stop = false;
        for (int ks = 0; ks < ksteps && !stop; ++ks) {
            for (int n = 0; n < nmt && !stop; ++n) {
                const int i = Plan::order(n, ks, nmt);
                const int j = Plan::interval(i, ks);
                if (j < 1 || j >= Plan::count(i, ksteps) - 1 || Plan::last(i, j, ksteps) != ks) continue;
                const bool ok = !*err && mbar_wait_bounded(&pdone[Plan::buf(i, j)], Plan::use(j) & 1u);
                if (!__all_sync(0xffffffffu, ok)) {
                    *err = 1;
                    record_status(status, QW3_ERR_TIMEOUT);
                    stop = true;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                tmem_add_rows(tmem + lanes + Plan::master_col(i), tmem + lanes + Plan::partial_col(i, j));
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&pfree[Plan::buf(i, j)]);
            }
        }
    }
    __syncwarp();
    // all threads: wait for the accumulators (or give up after 1 s), then the
    // producer's copies must have landed before the CTA may exit
    if (!mbar_wait_bounded(done, 0u)) {
        *err = 1;
        record_status(status, QW3_ERR_TIMEOUT);
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0 && *err) {
        for (int ks = ksteps > TQ_STAGES ? ksteps - TQ_STAGES : 0; ks < ksteps; ++ks) {
            (void)mbar_wait_bounded(&full[ks % TQ_STAGES], static_cast<uint32_t>((ks / TQ_STAGES) & 1));
            (void)mbar_wait_bounded(&wfull[ks % TQ_STAGES], static_cast<uint32_t>((ks / TQ_STAGES) & 1));
        }
    }
    for (int mi = 0; mi < nmt && warp >= 12; ++mi) {
        // ---- epilogue: thread (warp, lane) owns row 32 (warp - 12) + lane of
        // m-tile mi, all 128 columns: the master plus the last interval's partial
        const int mt = mt0 + mi;
        const int row = 32 * (warp - 12) + lane;
        const int m = mt * TC_BM + row;
        const int jl = Plan::count(mi, ksteps) - 1;
        const uint32_t lanes = static_cast<uint32_t>(32 * (warp - 12)) << 16;
        unsigned long long best = 0ull;
        const int Np = gridDim.x * TC_BN;   // workspace row stride
        for (int c0 = 0; c0 < TC_BN; c0 += 16) {
            float v[16];
            tmem_ld_sum16(tmem + lanes + Plan::master_col(mi) + c0,
                          jl >= 1 ? tmem + lanes + Plan::partial_col(mi, jl) + c0 : 0u, jl >= 1, v);
            if (m >= M || *err) continue;
            unscale16(v, ainv[m], wscale + gridDim.x * TC_BN, nt * TC_BN + c0);
            if (nks > 1) {
                float4 *w4 = reinterpret_cast<float4 *>(
                    ws + (static_cast<size_t>(kz) * mtiles * TC_BM + static_cast<size_t>(m)) * Np + nt * TC_BN + c0);
#pragma unroll
                for (int j = 0; j < 4; ++j) w4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                continue;
            }
            const int nb = nt * TC_BN + c0;
            if (MODE == GEMV_SWIGLU) {
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    const int n = nb + j;
                    if (n < N) C[static_cast<size_t>(m) * (N / 2) + n / 2] = v[j] / (1.0f + expf(-v[j])) * v[j + 1];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int n = nb + j;
                    if (n < N) {
                        const float y = v[j];
                        float *cp = C ? C + static_cast<size_t>(m) * N + n : nullptr;
                        if (MODE == GEMV_STORE) *cp = y;
                        else if (MODE == GEMV_RESID) *cp += y;
                        else {
                            if (cp) *cp = y;
                            const unsigned long long kk = argmax_pack(y, n);
                            best = kk > best ? kk : best;
                        }
                    }
                }
            }
        }
        if (MODE == GEMV_ARGMAX && m < M && best) atomicMax(&argmax_key[m], best);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPromoCols) : "memory");
}

// Sum of the K splits of a tensor-core GEMM in split order (deterministic),
// then the epilogue: thread = (row, 4 columns).
template <int MODE>
__global__ void k_splitk_reduce(const float *__restrict__ ws, int nks, int M, int N, int Np, int Mp, float *C) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int cols4 = N / 4;
    if (i >= static_cast<int64_t>(M) * cols4) return;
    const int m = static_cast<int>(i / cols4), n = static_cast<int>(i % cols4) * 4;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int z = 0; z < nks; ++z) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(ws + (static_cast<size_t>(z) * Mp + m) * Np + n));
        v.x += t.x;
        v.y += t.y;
        v.z += t.z;
        v.w += t.w;
    }
    if (MODE == GEMV_SWIGLU) {
        float *c = C + static_cast<size_t>(m) * (N / 2) + n / 2;
        c[0] = v.x / (1.0f + expf(-v.x)) * v.y;
        c[1] = v.z / (1.0f + expf(-v.z)) * v.w;
    } else {
        float4 *c = reinterpret_cast<float4 *>(C + static_cast<size_t>(m) * N + n);
        if (MODE == GEMV_RESID) {
            const float4 o = *c;
            v.x += o.x;
            v.y += o.y;
            v.z += o.z;
            v.w += o.w;
        }
        *c = v;
    }
}

template <int MODE>
cudaError_t launch_tc_mode(const uint8_t *Ap, const float *ainv, int M, int K, const uint8_t *Wp, int N, float *C,
                           unsigned long long *argmax_key, const DecodeIO *io, int32_t *status,
                           const GemmSplitK *sk, cudaStream_t s) {
    const float *winv = reinterpret_cast<const float *>(Wp + ut_tile_bytes(N, K)) + pad_rows(N);
    const int wt = (N + TC_BN - 1) / TC_BN, mt = (M + TC_BM - 1) / TC_BM, ksteps = K / TC_BK;
    // 128 x 256 tiles (A shared by two W tiles) where enough of them fill the
    // GPU; 128 x 128 otherwise
    const bool wide = wt % 2 == 0 && (wt / 2) * mt >= num_sms();
    const int nt = wide ? wt / 2 : wt, bne = wide ? 2 * TC_BN : TC_BN;
    // split K while the output tiles leave SMs idle (>= 4 k-steps per split,
    // partials within the workspace); the reduction is its own kernel
    int nks = 1;
    if (MODE != GEMV_ARGMAX && sk && sk->ws && nt * mt < num_sms() && N % 4 == 0) {
        nks = (num_sms() + nt * mt - 1) / (nt * mt);
        nks = std::min(nks, ksteps / 4);
        while (nks > 1 && static_cast<size_t>(nks) * mt * TC_BM * nt * bne > sk->ws_floats) --nks;
        if (nks < 1) nks = 1;
    }
    const dim3 grid(nt, mt, nks);
    if (wide)
        k_gemm_tc<MODE, 2><<<grid, TC_THREADS, tc_smem<2>(), s>>>(Ap, M, K, Wp, N, C, argmax_key, io, status,
                                                                nks > 1 ? sk->ws : nullptr, ainv, winv);
    else
        k_gemm_tc<MODE, 1><<<grid, TC_THREADS, tc_smem<1>(), s>>>(Ap, M, K, Wp, N, C, argmax_key, io, status,
                                                                nks > 1 ? sk->ws : nullptr, ainv, winv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nks == 1) return e;
    const int64_t items = static_cast<int64_t>(M) * (N / 4);
    k_splitk_reduce<MODE><<<static_cast<unsigned>((items + 255) / 256), 256, 0, s>>>(sk->ws, nks, M, N, nt * bne,
                                                                                      mt * TC_BM, C);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_tq_mode(const uint8_t *Ap, const float *ainv, int M, int K, const uint8_t *Wq, int N, float *C,
                           unsigned long long *argmax_key, const DecodeIO *io, int32_t *status,
                           const GemmSplitK *sk, cudaStream_t s) {
    const int nt = (N + TC_BN - 1) / TC_BN, mt = (M + TC_BM - 1) / TC_BM, ksteps = K / TC_BK;
    const float *wscale = reinterpret_cast<const float *>(Wq + static_cast<size_t>(nt) * ksteps * TQ_RAW);
    // two m-tiles per CTA (one conversion of W for both) where that still
    // leaves a CTA for every SM
    const bool pair = mt >= 2 && nt * ((mt + 1) / 2) >= num_sms();
    const int gy = pair ? (mt + 1) / 2 : mt;
    int nks = 1;
    if (MODE != GEMV_ARGMAX && sk && sk->ws && nt * mt < num_sms() && N % 4 == 0) {
        nks = (num_sms() + nt * mt - 1) / (nt * mt);
        nks = std::min(nks, ksteps / 4);
        while (nks > 1 && static_cast<size_t>(nks) * mt * TC_BM * nt * TC_BN > sk->ws_floats) --nks;
        if (nks < 1) nks = 1;
    }
    const dim3 grid(nt, gy, nks);
    if (pair)
        k_gemm_tc_q8<MODE, 2><<<grid, TQ_THREADS, tq_smem<2>(), s>>>(Ap, M, K, Wq, N, C, argmax_key, io, status,
                                                                   nks > 1 ? sk->ws : nullptr, ainv, wscale);
    else
        k_gemm_tc_q8<MODE, 1><<<grid, TQ_THREADS, tq_smem<1>(), s>>>(Ap, M, K, Wq, N, C, argmax_key, io, status,
                                                                   nks > 1 ? sk->ws : nullptr, ainv, wscale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nks == 1) return e;
    const int64_t items = static_cast<int64_t>(M) * (N / 4);
    k_splitk_reduce<MODE><<<static_cast<unsigned>((items + 255) / 256), 256, 0, s>>>(sk->ws, nks, M, N, nt * TC_BN,
                                                                                      mt * TC_BM, C);
    return cudaGetLastError();
}

}  // namespace

cudaError_t configure_gemm_tc() {
    cudaError_t e = cudaSuccess;
#define QW3_TC_CFG(MODE)                                                                                          \
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<MODE, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                                    static_cast<int>(tc_smem<1>()));                                \
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc<MODE, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                                    static_cast<int>(tc_smem<2>()));
    QW3_TC_CFG(GEMV_STORE)
    QW3_TC_CFG(GEMV_RESID)
    QW3_TC_CFG(GEMV_SWIGLU)
    QW3_TC_CFG(GEMV_ARGMAX)
#undef QW3_TC_CFG
#define QW3_TQ_CFG(MODE)                                                                                         \
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc_q8<MODE, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                                    static_cast<int>(tq_smem<1>()));                                \
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_gemm_tc_q8<MODE, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                                    static_cast<int>(tq_smem<2>()));
    QW3_TQ_CFG(GEMV_STORE)
    QW3_TQ_CFG(GEMV_RESID)
    QW3_TQ_CFG(GEMV_SWIGLU)
    QW3_TQ_CFG(GEMV_ARGMAX)
#undef QW3_TQ_CFG
    return e;
}

size_t ut_bytes(int rows, int K) {
    return ut_tile_bytes(rows, K) + static_cast<size_t>(pad_rows(rows)) * 8;
}

size_t apack_bytes(int rows, int K) {
    return ut_tile_bytes(rows, K) + static_cast<size_t>(pad_rows(rows)) * 4;
}

bool gemm_tc_supported(int M, int K, const QMat &W) {
    // a matrix held only as tensor-core tiles (Q4_K models) takes every M
    return (W.ut != nullptr || W.uq != nullptr) && (M >= kGemmTcMinRows || W.base == nullptr) && K % TC_BK == 0 &&
           W.cols == K;
}

size_t tq_bytes(int rows, int K) {
    return static_cast<size_t>(pad_rows(rows) / TC_BM) * (K / TC_BK) * TQ_RAW + static_cast<size_t>(pad_rows(rows)) * 8;
}

cudaError_t launch_pack_w_q8(const QMat &W, uint8_t *dst, cudaStream_t s) {
    const int rows = pad_rows(W.rows);
    float *scale = reinterpret_cast<float *>(dst + static_cast<size_t>(rows / TC_BM) * (W.cols / TC_BK) * TQ_RAW);
    k_row_exp_q8<<<static_cast<unsigned>(rows / 8), 256, 0, s>>>(W, W.rows, W.cols, scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n = static_cast<int64_t>(rows) * (W.cols / 8);
    k_pack_w_q8<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(W, W.rows, W.cols, dst);
    return cudaGetLastError();
}

cudaError_t launch_pack_w_q4k(const uint8_t *W, int N, int K, uint8_t *dst, cudaStream_t s) {
    const int rows = pad_rows(N);
    k_row_exp_q4k<<<static_cast<unsigned>(rows / 8), 256, 0, s>>>(W, N, K,
                                                                  reinterpret_cast<float *>(dst + ut_tile_bytes(N, K)));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n = static_cast<int64_t>(rows) * (K / 8);
    k_pack_w_q4k<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(W, N, K, dst);
    return cudaGetLastError();
}

size_t gemm_q8_raw_workspace_bytes(int N, int K, int M) { return tq_bytes(N, K) + apack_bytes(M, K); }

cudaError_t launch_gemm_q8_raw(const uint8_t *W, int N, int K, const float *A, int M, float *C, uint8_t *ws,
                               cudaStream_t s) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    const int rows = pad_rows(N);
    float *scale = reinterpret_cast<float *>(ws + static_cast<size_t>(rows / TC_BM) * (K / TC_BK) * TQ_RAW);
    k_row_exp_q8_raw<<<static_cast<unsigned>(rows / 8), 256, 0, s>>>(W, N, K, scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t n = static_cast<int64_t>(rows) * (K / 8);
    k_pack_w_q8_raw<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(W, N, K, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    uint8_t *apack = ws + tq_bytes(N, K);
    float *ainv = reinterpret_cast<float *>(apack + ut_tile_bytes(M, K));
    k_pack_act<<<static_cast<unsigned>(pad_rows(M)), kPackActThreads, 0, s>>>(A, M, K, apack, ainv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_tq_mode<GEMV_STORE>(apack, ainv, M, K, ws, N, C, nullptr, nullptr, nullptr, nullptr, s);
}

cudaError_t launch_gemm_tc(const float *A, int M, int K, const QMat &W, float *C, int mode,
                           unsigned long long *argmax_key, const DecodeIO *io, int32_t *status, uint8_t *apack,
                           cudaStream_t s, const GemmSplitK *sk) {
    if (M <= 0) return cudaSuccess;
    float *ainv = reinterpret_cast<float *>(apack + ut_tile_bytes(M, K));
    k_pack_act<<<static_cast<unsigned>(pad_rows(M)), kPackActThreads, 0, s>>>(A, M, K, apack, ainv);
    {
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (W.uq) {
        switch (mode) {
            case GEMV_STORE: return launch_tq_mode<GEMV_STORE>(apack, ainv, M, K, W.uq, W.rows, C, argmax_key, io, status, sk, s);
            case GEMV_RESID: return launch_tq_mode<GEMV_RESID>(apack, ainv, M, K, W.uq, W.rows, C, argmax_key, io, status, sk, s);
            case GEMV_SWIGLU: return launch_tq_mode<GEMV_SWIGLU>(apack, ainv, M, K, W.uq, W.rows, C, argmax_key, io, status, sk, s);
            case GEMV_ARGMAX: return launch_tq_mode<GEMV_ARGMAX>(apack, ainv, M, K, W.uq, W.rows, C, argmax_key, io, status, sk, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (mode) {
        case GEMV_STORE: return launch_tc_mode<GEMV_STORE>(apack, ainv, M, K, W.ut, W.rows, C, argmax_key, io, status, sk, s);
        case GEMV_RESID: return launch_tc_mode<GEMV_RESID>(apack, ainv, M, K, W.ut, W.rows, C, argmax_key, io, status, sk, s);
        case GEMV_SWIGLU: return launch_tc_mode<GEMV_SWIGLU>(apack, ainv, M, K, W.ut, W.rows, C, argmax_key, io, status, sk, s);
        case GEMV_ARGMAX: return launch_tc_mode<GEMV_ARGMAX>(apack, ainv, M, K, W.ut, W.rows, C, argmax_key, io, status, sk, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qw3
