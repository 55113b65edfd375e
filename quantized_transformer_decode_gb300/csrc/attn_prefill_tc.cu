// Causal prefill attention on the 5th-generation tensor cores ("A transformer
// from scratch", 12.3.5: scores q.k / sqrt(head_dim) over keys 0..p, softmax
// with the running maximum subtracted, weighted sum of V; GQA maps query head
// h to kv head h / (n_heads / n_kv_heads)).
//
// Flash-attention over 64-key tiles, one CTA per (128-query tile, query
// head), f32 accuracy from fp16 operands as in the GEMMs: every operand x,
// first multiplied by a power of two 2^t, is split into hi = fp16(x) and
// lo = fp16(x - hi), and each product is hi.hi + hi.lo + lo.hi (three
// tcgen05.mma, f32 accumulation in TMEM); the results are multiplied by the
// inverse powers (exact). The factors: one per query row and one per kv head
// for K (from the largest magnitude over its keys: keys after the Q/K norm
// have like magnitudes), one per (kv head, 8 dimensions) over all keys for V
// (O = P V contracts over keys, so V's factor must not vary along them); P
// lies in [0, 2^8] and needs none.
//  * Per layer, k_kv_absmax, k_pack_k and k_pack_v convert the cached K and V
//    of the sequence into per-(kv head, 64-key tile) UMMA operand tiles (K as
//    B of S = Q K^T, V transposed as B of O = P V), so attention CTAs fetch
//    each tile with one bulk copy into a two-buffer ring.
//  * The CTA packs its 128 query rows once; per key tile: S = Q K^T into 64
//    TMEM columns; each thread owns one query row (its TMEM lane) and runs
//    the online softmax on it without shuffles (in base 2); P (hi/lo) goes
//    to shared memory; then P V accumulates into a partial O in TMEM. The
//    tensor core's f32 accumulation truncates toward zero, so a long chain of
//    MMAs into one accumulator loses a relative ~1.6e-8 per MMA; the partial
//    therefore holds at most kPvChain tiles before the threads add it into
//    the master O (CUDA-core f32, round to nearest). The row's reference
//    maximum trails its true maximum by at most 8 (base 2) and moves rarely:
//    where it moves, the row's partial and master are rescaled in place, and
//    a promotion applies the tile's rescale: master = (master + partial) *
//    corr. The row's 1/l scaling is applied when O is read back.
//  * Every wait is bounded (1 s -> QW3_ERR_TIMEOUT, then the kernel drains
//    and frees its tensor memory without waiting further).
#include "qw3_internal.cuh"

namespace qw3 {

namespace {

constexpr int kQT = 128;          // queries per CTA (TMEM lanes)
constexpr int kKT = 64;           // keys per tile
constexpr int kPaThreads = 128;
constexpr int kPvChain = 4;       // key tiles per P V accumulation chain

// Bytes of the packed operand tiles.
template <int HD>
struct PaSizes {
    static constexpr uint32_t kq = (HD / 64) * 2 * (kQT * 128);   // Q: per 64-dim step hi + lo, 128 rows x 128 B
    static constexpr uint32_t kk = (HD / 64) * 2 * (kKT * 128);   // K tile: per 64-dim step hi + lo, 64 rows
    static constexpr uint32_t kv = 2 * (HD * 128);                // V^T tile: hi + lo, HD rows x 64 keys
    static constexpr uint32_t kkv = kk + kv;                      // one packed (K, V) tile
    static constexpr uint32_t kp = 2 * (kQT * 128);               // P: hi + lo, 128 rows x 64 keys
    static constexpr uint32_t smem = kq + 2 * kkv + kp + 1024 + 256;
};

// The pack buffer: nkv * ntiles (K, V^T) tiles, then V's inverse factors
// [nkv][HD], then K's [nkv] (padded to 4), then the scratch of the maxima of
// K and V [2][nkv][HD / 8].
template <int HD>
__host__ __device__ inline float *pa_vinv(uint8_t *pack, int nkv, int ntiles) {
    return reinterpret_cast<float *>(pack + static_cast<size_t>(nkv) * ntiles * PaSizes<HD>::kkv);
}
template <int HD>
__host__ __device__ inline float *pa_kinv(uint8_t *pack, int nkv, int ntiles) {
    return pa_vinv<HD>(pack, nkv, ntiles) + static_cast<size_t>(nkv) * HD;
}
template <int HD>
__host__ __device__ inline unsigned *pa_kvmax(uint8_t *pack, int nkv, int ntiles) {
    return reinterpret_cast<unsigned *>(pa_kinv<HD>(pack, nkv, ntiles) + (nkv + 3) / 4 * 4);
}

// Byte offset of element (row r, column k) in a K-major no-swizzle UMMA tile
// of 64 columns: 8x8 core matrices (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint32_t pa_core(int r, int k) {
    return static_cast<uint32_t>((r >> 3) * 1024 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint64_t pa_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(128 >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46);
}

// kind::f16 instruction descriptor: f32 accumulate (bit 4), fp16 A and B
// (format fields 0), K-major.
__host__ __device__ constexpr uint32_t pa_idesc(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// The largest magnitudes of K and of V per (kv head, 8 dimensions) over keys
// [0, ctx), as the bits of non-negative f32 (atomicMax in unsigned order;
// kvmax zeroed first; [0] K, [1] V): a CTA covers 256 keys of one head,
// thread = (key, 8 dimensions), reduced in shared memory before one atomic
// per group.
template <int HD, typename KT>
__global__ void __launch_bounds__(256) k_kv_absmax(const KT *__restrict__ kc, const KT *__restrict__ vc,
                                                   size_t head_stride, int nkv, int ctx,
                                                   unsigned *__restrict__ kvmax) {
    constexpr int G = HD / 8, KPI = 256 / G;   // dimension groups; keys per pass of the CTA
    __shared__ float red[2][256];
    const int g = blockIdx.y, tid = threadIdx.x, dg = tid % G;
    const KT *ksrc = kc + static_cast<size_t>(g) * head_stride;
    const KT *vsrc = vc + static_cast<size_t>(g) * head_stride;
    float km = 0.0f, vm = 0.0f;
    const int k_end = min(ctx, (blockIdx.x + 1) * 256);
    for (int key = blockIdx.x * 256 + tid / G; key < k_end; key += KPI) {
        const size_t off = static_cast<size_t>(key) * kv_row<KT, HD>();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            km = fmaxf(km, fabsf(kv_elem<HD>(ksrc + off, dg * 8 + j)));
            vm = fmaxf(vm, fabsf(kv_elem<HD>(vsrc + off, dg * 8 + j)));
        }
    }
    red[0][tid] = km;
    red[1][tid] = vm;
    __syncthreads();
    if (tid < G) {
        for (int k = tid + G; k < 256; k += G) {
            km = fmaxf(km, red[0][k]);
            vm = fmaxf(vm, red[1][k]);
        }
        atomicMax(&kvmax[g * G + tid], __float_as_uint(km));
        atomicMax(&kvmax[(nkv + g) * G + tid], __float_as_uint(vm));
    }
}

// K tiles: one thread per (kv head, key, 8 dimensions) of keys
// [0, ntiles * 64), every key of a head scaled by the head's factor (from
// its largest magnitude over keys and dimensions: keys after the Q/K norm
// have like magnitudes). Keys at or past ctx are zero.
template <int HD, typename KT>
__global__ void k_pack_k(const KT *__restrict__ kc, size_t head_stride, int nkv, int ctx, int ntiles,
                         const unsigned *__restrict__ kvmax, uint8_t *__restrict__ dst) {
    using Z = PaSizes<HD>;
    constexpr int G = HD / 8;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(nkv) * ntiles * kKT * G) return;
    const int d0 = static_cast<int>(i % G) * 8;
    const int64_t kid = i / G;
    const int key = static_cast<int>(kid % (static_cast<int64_t>(ntiles) * kKT));
    const int g = static_cast<int>(kid / (static_cast<int64_t>(ntiles) * kKT));
    float amax = 0.0f;
#pragma unroll
    for (int q = 0; q < G; ++q) amax = fmaxf(amax, __uint_as_float(kvmax[g * G + q]));
    const int t = f16_row_exp(amax);
    const float sr = pow2_f32(t);
    const KT *row = kc + static_cast<size_t>(g) * head_stride + static_cast<size_t>(key) * kv_row<KT, HD>();
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = key < ctx ? kv_elem<HD>(row, d0 + j) * sr : 0.0f;
    uint4 hi, lo;
    split8_f16(v, hi, lo);
    const int tile = key / kKT, r = key % kKT;
    uint8_t *base = dst + (static_cast<size_t>(g) * ntiles + tile) * Z::kkv + (d0 / 64) * 2 * (kKT * 128);
    *reinterpret_cast<uint4 *>(base + pa_core(r, d0 % 64)) = hi;
    *reinterpret_cast<uint4 *>(base + kKT * 128 + pa_core(r, d0 % 64)) = lo;
    if (key == 0 && d0 == 0) pa_kinv<HD>(dst, nkv, ntiles)[g] = pow2_f32(-t);
}

// V^T tiles: one thread per (kv head, tile, dimension, 8-key group); each
// (kv head, 8 dimensions) scaled by the factor of its maximum over all keys.
// Keys at or past ctx are zero.
template <int HD, typename KT>
__global__ void k_pack_v(const KT *__restrict__ vc, size_t head_stride, int nkv, int ctx, int ntiles,
                         const unsigned *__restrict__ kvmax, uint8_t *__restrict__ dst) {
    using Z = PaSizes<HD>;
    constexpr int kItems = HD * (kKT / 8);
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<int64_t>(nkv) * ntiles * kItems) return;
    const int item = static_cast<int>(i % kItems);
    const int tile = static_cast<int>((i / kItems) % ntiles);
    const int g = static_cast<int>(i / (static_cast<int64_t>(kItems) * ntiles));
    const int d = item / (kKT / 8), k0 = (item % (kKT / 8)) * 8;
    const int t = f16_row_exp(__uint_as_float(kvmax[(nkv + g) * (HD / 8) + d / 8]));
    const float sr = pow2_f32(t);
    const KT *src = vc + static_cast<size_t>(g) * head_stride;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int key = tile * kKT + k0 + j;
        v[j] = key < ctx ? kv_elem<HD>(src + static_cast<size_t>(key) * kv_row<KT, HD>(), d) * sr : 0.0f;
    }
    uint4 hi, lo;
    split8_f16(v, hi, lo);
    uint8_t *base = dst + (static_cast<size_t>(g) * ntiles + tile) * Z::kkv + Z::kk;
    *reinterpret_cast<uint4 *>(base + pa_core(d, k0)) = hi;
    *reinterpret_cast<uint4 *>(base + HD * 128 + pa_core(d, k0)) = lo;
    if (tile == 0 && k0 == 0) pa_vinv<HD>(dst, nkv, ntiles)[static_cast<size_t>(g) * HD + d] = pow2_f32(-t);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// 32 columns of this warp's TMEM lanes into v[o .. o + 32) (one wait).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[kKT], int o) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[o + j] = __uint_as_float(r[j]);
}

// Three MMAs (hi.hi, hi.lo, lo.hi) over one 64-deep step: A at a_hi / a_lo,
// B at b_hi / b_lo (each a K-major tile of 64 columns); accumulate unless
// first.
__device__ __forceinline__ void mma3(uint32_t tmem, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                     uint32_t idesc, bool first) {
#pragma unroll
    for (int sub = 0; sub < 4; ++sub) {
        const uint32_t off = sub * 256;
        const uint32_t acc0 = (!first || sub > 0) ? 1u : 0u;
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %3, 1;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %2, %3, 1;\n\t}"
            ::"r"(tmem), "l"(pa_desc(a_hi + off)), "l"(pa_desc(b_hi + off)), "r"(idesc), "r"(acc0),
              "l"(pa_desc(b_lo + off)), "l"(pa_desc(a_lo + off))
            : "memory");
    }
}

// This thread's row of the master O (TMEM lanes of its warp): master =
// ((has_master ? master : 0) + partial) * corr, over HD columns; the stores
// complete before it returns. Warp-collective (has_master warp-uniform).
template <int HD>
__device__ __forceinline__ void promote_o(uint32_t master, uint32_t partial, bool has_master, float corr) {
#pragma unroll 1
    for (int c0 = 0; c0 < HD; c0 += 16) {
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
        for (int j = 0; j < 16; ++j) {
            const float m = has_master ? __uint_as_float(a[j]) : 0.0f;
            a[j] = __float_as_uint((m + __uint_as_float(b[j])) * corr);
        }
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
            ::"r"(master + c0), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]),
              "r"(a[7]), "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]), "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15])
            : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// This thread's row of an O accumulator times corr, in place (warp-collective).
template <int HD>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float corr) {
#pragma unroll 1
    for (int c0 = 0; c0 < HD; c0 += 16) {
        float t16[16];
        tmem_ld16(taddr + static_cast<uint32_t>(c0), t16);
        uint32_t u[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(t16[e] * corr);
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
            ::"r"(taddr + static_cast<uint32_t>(c0)), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]),
              "r"(u[5]), "r"(u[6]), "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]),
              "r"(u[13]), "r"(u[14]), "r"(u[15])
            : "memory");
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int HD>
__global__ void __launch_bounds__(kPaThreads, 1)
    k_attn_prefill_tc(const float *__restrict__ qkv, int M, int qkv_stride, uint8_t *kvpack, int nkv,
                      int ntiles, int pos0, int group, float scale, float *__restrict__ out, int32_t *status) {
    using Z = PaSizes<HD>;
    extern __shared__ __align__(1024) uint8_t pa_smem[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(pa_smem) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *Qs = base;                    // [HD/64][hi|lo] 128 x 64 tiles
    uint8_t *KV0 = Qs + Z::kq;             // two packed (K, V^T) tiles
    uint8_t *Ps = KV0 + 2 * Z::kkv;        // [hi|lo] 128 x 64
    uint64_t *bars = reinterpret_cast<uint64_t *>(Ps + Z::kp);   // kv_full[2], s_done, o_done
    uint64_t *kv_full = bars, *s_done = bars + 2, *o_done = bars + 3;
    uint32_t *tbase = reinterpret_cast<uint32_t *>(bars + 4);
    volatile int *err = reinterpret_cast<volatile int *>(tbase + 1);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int qt = gridDim.x - 1 - blockIdx.x, h = blockIdx.y, g = h / group;   // late (heavy) query tiles first
    const int row = tid;                                   // this thread's query (TMEM lane)
    const int q = qt * kQT + row;                          // row of the chunk
    const int qpos = pos0 + q;                             // its position
    const int last_q = min(M - 1, qt * kQT + kQT - 1);
    const int ntl = min(ntiles, (pos0 + last_q) / kKT + 1);   // key tiles this CTA needs
    const uint8_t *kvg = kvpack + static_cast<size_t>(g) * ntiles * Z::kkv;
    const float kinv_g = pa_kinv<HD>(kvpack, nkv, ntiles)[g];
    const float *vinvg = pa_vinv<HD>(kvpack, nkv, ntiles) + static_cast<size_t>(g) * HD;
    // thread 0: the K/V^T pair of tile jt into buffer b
    auto fetch = [&](int jt, int b) {
        mbar_arrive_expect_tx(&kv_full[b], Z::kkv);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_u32(KV0 + b * Z::kkv)), "l"(kvg + static_cast<size_t>(jt) * Z::kkv), "r"(Z::kkv),
                       "r"(smem_u32(&kv_full[b]))
                     : "memory");
    };

    if (tid == 0) {
        mbar_init(&kv_full[0], 1);
        mbar_init(&kv_full[1], 1);
        mbar_init(s_done, 1);
        mbar_init(o_done, 1);
        *err = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tbase)),
                     "r"(512) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tbase;
    const uint32_t tS = tmem, tO = tmem + 128, tP = tmem + 256;   // S: 64 columns; master and partial O: HD
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;

    int last_issued[2] = {-1, -1};   // thread 0: the last tile fetched into each buffer
    if (tid == 0) {
        for (int j = 0; j < 2 && j < ntl; ++j) {
            last_issued[j] = j;
            fetch(j, j);
        }
    }
    // ---- this thread's query row -> Q tiles (hi / lo), scaled by its factor
    float qinv = 1.0f;
    {
        const float *src = qkv + static_cast<size_t>(q) * qkv_stride + static_cast<size_t>(h) * HD;
        float amax = 0.0f;
        if (q < M)
#pragma unroll 4
            for (int d0 = 0; d0 < HD; d0 += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(src + d0);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
            }
        const int t = f16_row_exp(amax);
        const float sr = pow2_f32(t);
        qinv = pow2_f32(-t);
#pragma unroll
        for (int d0 = 0; d0 < HD; d0 += 8) {
            float v[8];
            if (q < M) {
                const float4 a = *reinterpret_cast<const float4 *>(src + d0);
                const float4 b = *reinterpret_cast<const float4 *>(src + d0 + 4);
                v[0] = a.x * sr; v[1] = a.y * sr; v[2] = a.z * sr; v[3] = a.w * sr;
                v[4] = b.x * sr; v[5] = b.y * sr; v[6] = b.z * sr; v[7] = b.w * sr;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = 0.0f;
            }
            uint4 hi, lo;
            split8_f16(v, hi, lo);
            uint8_t *tq = Qs + (d0 / 64) * 2 * (kQT * 128);
            *reinterpret_cast<uint4 *>(tq + pa_core(row, d0 % 64)) = hi;
            *reinterpret_cast<uint4 *>(tq + kQT * 128 + pa_core(row, d0 % 64)) = lo;
        }
    }
    fence_async_smem();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();

    constexpr uint32_t kIdS = pa_idesc(kQT, kKT), kIdO = pa_idesc(kQT, HD);
    // softmax in base 2: exp(x) = 2^(x log2 e), scores pre-scaled by log2 e;
    // qs2 also undoes the row's and the head's operand factors (powers of two)
    const float scale2 = scale * 1.4426950408889634f;
    const float qs2 = (qinv * kinv_g) * scale2;
    float m_run = -INFINITY, l_run = 0.0f;
    int chain = 0;              // tiles in the partial O (CTA-uniform)
    bool has_master = false;    // the master O holds promoted tiles
    for (int j = 0; j < ntl; ++j) {
        const int buf = j & 1;
        const uint8_t *KV = KV0 + buf * Z::kkv;
        // ---- S = Q K_j^T (issued by one thread)
        if (tid == 0) {
            if (*err || !mbar_wait_bounded(&kv_full[buf], static_cast<uint32_t>((j >> 1) & 1))) {
                *err = 1;
            } else {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int s = 0; s < HD / 64; ++s) {
                    const uint32_t a = smem_u32(Qs + s * 2 * (kQT * 128));
                    const uint32_t b = smem_u32(KV + s * 2 * (kKT * 128));
                    mma3(tS, a, a + kQT * 128, b, b + kKT * 128, kIdS, s == 0);
                }
            }
            mma_commit(s_done);
        }
        __syncwarp();
        if (!mbar_wait_bounded(s_done, static_cast<uint32_t>(j & 1))) *err = 1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // ---- online softmax of this row over the tile's 64 keys
        float sv[kKT];
        tmem_ld32(tS + lane_off, sv, 0);
        tmem_ld32(tS + lane_off + 32u, sv, 32);
        float mx = -INFINITY;
        if ((j + 1) * kKT - 1 > pos0 + qt * kQT) {
            // a tile on the diagonal: keys past the row's position are masked
#pragma unroll
            for (int c = 0; c < kKT; ++c) {
                sv[c] = (j * kKT + c <= qpos) ? sv[c] * qs2 : -INFINITY;
                mx = fmaxf(mx, sv[c]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < kKT; ++c) {
                sv[c] *= qs2;
                mx = fmaxf(mx, sv[c]);
            }
        }
        // The reference maximum moves only when the tile's maximum exceeds it
        // by more than 8 (probabilities up to 2^8 are exact to represent and
        // cancel in O / l): most tiles then need no rescale of O.
        const float m_new = (mx > m_run + 8.0f) ? mx : m_run;
        const float corr = (m_new == m_run || m_new == -INFINITY) ? 1.0f : exp2f(m_run - m_new);
        float ps = 0.0f;
#pragma unroll
        for (int c = 0; c < kKT; ++c) {
            sv[c] = (sv[c] == -INFINITY) ? 0.0f : exp2f(sv[c] - m_new);
            ps += sv[c];
        }
        l_run = fmaf(l_run, corr, ps);
        m_run = m_new;
        // ---- the previous P V must be complete before P and O change
        if (j > 0) {
            if (!mbar_wait_bounded(o_done, static_cast<uint32_t>((j - 1) & 1))) *err = 1;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // its K/V buffer is free: fetch tile j + 1 into it
            if (tid == 0 && j + 1 < ntl && !*err) {
                const int nb = (j + 1) & 1;
                last_issued[nb] = j + 1;
                fetch(j + 1, nb);
            }
            if (chain == kPvChain) {
                // the partial is full: master = (master + partial) * corr
                promote_o<HD>(tO + lane_off, tP + lane_off, has_master, corr);
                has_master = true;
                chain = 0;
            } else if (__any_sync(0xffffffffu, corr != 1.0f)) {
                // a row's maximum moved: rescale its partial (and master) in place
                rescale_o<HD>(tP + lane_off, corr);
                if (has_master) rescale_o<HD>(tO + lane_off, corr);
            }
        }
        // ---- P (hi / lo) of this row
#pragma unroll
        for (int c = 0; c < kKT; c += 8) {
            const float v8[8] = {sv[c], sv[c + 1], sv[c + 2], sv[c + 3], sv[c + 4], sv[c + 5], sv[c + 6], sv[c + 7]};
            uint4 hi, lo;
            split8_f16(v8, hi, lo);
            *reinterpret_cast<uint4 *>(Ps + pa_core(row, c)) = hi;
            *reinterpret_cast<uint4 *>(Ps + kQT * 128 + pa_core(row, c)) = lo;
        }
        fence_async_smem();
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        // ---- partial O += P V_j (a new chain after a promotion)
        if (tid == 0) {
            if (!*err) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a = smem_u32(Ps);
                const uint32_t b = smem_u32(KV + Z::kk);
                mma3(tP, a, a + kQT * 128, b, b + HD * 128, kIdO, chain == 0);
            }
            mma_commit(o_done);
        }
        ++chain;
        __syncwarp();
    }
    // ---- O / l of this row to global memory
    if (ntl > 0) {
        if (!mbar_wait_bounded(o_done, static_cast<uint32_t>((ntl - 1) & 1))) *err = 1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    const float inv = l_run > 0.0f ? 1.0f / l_run : 0.0f;
    float *dst = out + static_cast<size_t>(q) * (static_cast<size_t>(gridDim.y) * HD) + static_cast<size_t>(h) * HD;
#pragma unroll
    for (int c = 0; c < HD; c += 16) {
        float t16[16];
        tmem_ld16(tP + lane_off + static_cast<uint32_t>(c), t16);
        if (has_master) {
            float m16[16];
            tmem_ld16(tO + lane_off + static_cast<uint32_t>(c), m16);
#pragma unroll
            for (int e = 0; e < 16; ++e) t16[e] += m16[e];
        }
        if (q < M && ntl > 0) {
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
                const float4 vi = *reinterpret_cast<const float4 *>(vinvg + c + e);
                *reinterpret_cast<float4 *>(dst + c + e) =
                    make_float4((t16[e] * vi.x) * inv, (t16[e + 1] * vi.y) * inv, (t16[e + 2] * vi.z) * inv,
                                (t16[e + 3] * vi.w) * inv);
            }
        }
    }
    __syncthreads();
    if (tid == 0 && *err) {
        record_status(status, QW3_ERR_TIMEOUT);
        // copies that may still be in flight (bounded)
        for (int b = 0; b < 2; ++b)
            if (last_issued[b] >= 0)
                (void)mbar_wait_bounded(&kv_full[b], static_cast<uint32_t>((last_issued[b] >> 1) & 1));
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

template <int HD, typename KT>
cudaError_t launch_pa_t(const float *qkv, int M, int qkv_stride, const KT *kc, const KT *vc,
                        size_t head_stride, int pos0, int nh, int nkv, float scale, float *out, uint8_t *kvpack,
                        int32_t *status, cudaStream_t s) {
    using Z = PaSizes<HD>;
    const int ctx = pos0 + M;
    const int ntiles = (ctx + kKT - 1) / kKT;
    unsigned *kvmax = pa_kvmax<HD>(kvpack, nkv, ntiles);
    cudaError_t e = cudaMemsetAsync(kvmax, 0, static_cast<size_t>(2 * nkv) * (HD / 8) * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    k_kv_absmax<HD, KT><<<dim3((ctx + 255) / 256, nkv), 256, 0, s>>>(kc, vc, head_stride, nkv, ctx, kvmax);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t kthreads = static_cast<int64_t>(nkv) * ntiles * kKT * (HD / 8);
    k_pack_k<HD, KT><<<static_cast<unsigned>((kthreads + 255) / 256), 256, 0, s>>>(kc, head_stride, nkv, ctx,
                                                                                    ntiles, kvmax, kvpack);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t vitems = static_cast<int64_t>(nkv) * ntiles * HD * (kKT / 8);
    k_pack_v<HD, KT><<<static_cast<unsigned>((vitems + 255) / 256), 256, 0, s>>>(vc, head_stride, nkv, ctx, ntiles,
                                                                                  kvmax, kvpack);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const dim3 grid((M + kQT - 1) / kQT, nh);
    k_attn_prefill_tc<HD><<<grid, kPaThreads, Z::smem, s>>>(qkv, M, qkv_stride, kvpack, nkv, ntiles, pos0,
                                                            nh / nkv, scale, out, status);
    return cudaGetLastError();
}

}  // namespace

size_t attn_prefill_tc_pack_bytes(int hd, int nkv, int max_seq_len) {
    const size_t ntiles = (static_cast<size_t>(max_seq_len) + kKT - 1) / kKT;
    const size_t tile = hd == 128 ? PaSizes<128>::kkv : PaSizes<64>::kkv;
    return static_cast<size_t>(nkv) * ntiles * tile + static_cast<size_t>(nkv) * hd * 4 +
           static_cast<size_t>(nkv + 3) / 4 * 16 + static_cast<size_t>(2 * nkv) * (hd / 8) * 4;
}

cudaError_t configure_attn_prefill_tc() {
    cudaError_t e = cudaFuncSetAttribute(k_attn_prefill_tc<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(PaSizes<128>::smem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_attn_prefill_tc<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PaSizes<64>::smem));
    return e;
}

template <typename KT>
static cudaError_t launch_pa_kt(const float *qkv, int M, int qkv_stride, const KT *kc, size_t kvsel_stride,
                         size_t head_stride, int pos0, int nh, int nkv, int hd, float scale, float *out,
                         uint8_t *kvpack, int32_t *status, cudaStream_t s) {
    const KT *vc = kc + kvsel_stride;
    if (hd == 128)
        return launch_pa_t<128, KT>(qkv, M, qkv_stride, kc, vc, head_stride, pos0, nh, nkv, scale, out, kvpack,
                                    status, s);
    if (hd == 64)
        return launch_pa_t<64, KT>(qkv, M, qkv_stride, kc, vc, head_stride, pos0, nh, nkv, scale, out, kvpack,
                                   status, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_prefill_tc(const float *qkv, int M, int qkv_stride, const void *kv_seq, size_t kvsel_stride,
                                   size_t head_stride, int pos0, int nh, int nkv, int hd, float scale, float *out,
                                   uint8_t *kvpack, int32_t *status, int kvtype, cudaStream_t s) {
    if (kvtype == KV_Q8)
        return launch_pa_kt(qkv, M, qkv_stride, static_cast<const kvq8 *>(kv_seq), kvsel_stride, head_stride,
                            pos0, nh, nkv, hd, scale, out, kvpack, status, s);
    if (kvtype == KV_F16)
        return launch_pa_kt(qkv, M, qkv_stride, static_cast<const __half *>(kv_seq), kvsel_stride, head_stride,
                            pos0, nh, nkv, hd, scale, out, kvpack, status, s);
    return launch_pa_kt(qkv, M, qkv_stride, static_cast<const float *>(kv_seq), kvsel_stride, head_stride, pos0, nh,
                        nkv, hd, scale, out, kvpack, status, s);
}

}  // namespace qw3
