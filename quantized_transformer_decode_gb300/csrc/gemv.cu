// Decode-time Q8_0 GEMV: y[b][r] = sum_k d[r][k/32] * q[r][k] * h[b][k] for
// B <= 4 activation rows ("A transformer from scratch", 12.5: at decode every
// projection is a matrix-vector product and the weight stream is the cost).
//
// Design (GB300):
//  * Two CTAs per SM (one where the layout needs more than half the SM's
//    shared memory): 18 warps per SM hide the dequantise-and-dot latency
//    that 9 cannot. CTA c owns a contiguous run of 8-row groups; in the
//    tiled weight layout (8 rows x kt columns per tile, codes then scales)
//    that slice is one contiguous range.
//  * The slice streams through shared memory in stages of whole tiles, one
//    1-D bulk copy (TMA, cp.async.bulk, L2 evict-first) per stage. A bulk
//    copy pays a fixed cost of a few hundred ns, so stages are large: a slice
//    that fits (up to ~100 KB) is a single copy; bigger slices use a ring of
//    up to six stages of up to 36 KB, sized to keep the most bytes in flight
//    within the CTA's share of shared memory.
//  * Warp specialisation: warp 8 is the producer; its first copies are
//    issued before griddepcontrol.wait (weights never depend on the previous
//    kernel), so under programmatic dependent launch the weight stream
//    overlaps the previous kernel. Warps 0-7 consume every stage in order
//    ("full" mbarriers, then "empty" mbarriers with 8 arrivals), so a slot is
//    never more than one phase ahead of its waiters: warp w takes row w of
//    each tile, four tiles at once for independent chains.
//  * Consumers wait for the previous kernel, then stage the input rows in
//    shared memory (optionally RMS-normalised, 12.3.2), in one of two forms.
//    Small slices (the per-layer projections at 0.6B): f32 in a padded
//    layout (36 floats per 32-value block, conflict-free 128-bit reads); per
//    16 codes a lane converts int8 -> f32 by byte-permuting q + 128 into the
//    mantissa of 2^23 and subtracting (exact) and accumulates with packed
//    fma.rn.f32x2. Large slices (lm_head; every projection at 8B): int8
//    digit planes (x = s (h + m/254 + l/254^2) per 32-block, within ~6e-8 of
//    the block maximum), so that 16 codes cost 12 exact dp4a and one f32
//    combination: about twice the f32 path's throughput, for a staging cost
//    that only a large slice amortises. f32 accumulation throughout.
//  * Row sums land in shared memory; one epilogue after the stream: store,
//    residual add (12.3.7, the residual rows are fetched early), SwiGLU over
//    interleaved gate/up rows (12.3.6), or argmax with packed (value, index)
//    u64 keys and a last-CTA finish that emits the greedy token (12.6).
#include <algorithm>

#include "qw3_internal.cuh"

namespace qw3 {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;   // + producer warp
constexpr size_t kOneShot = 100 * 1024;     // slices up to this size: one copy
constexpr size_t kStageTarget = 36 * 1024;  // ring stage size otherwise
constexpr int kMaxStages = 6;             // ring stages at most
constexpr size_t kPlanesMinSlice = 192 * 1024;   // digit-plane activations from this CTA slice size
constexpr size_t kSmemMax = 227 * 1024;     // dynamic shared memory of one CTA
constexpr size_t kSmemPair = 112 * 1024;    // per CTA when two share an SM (228 KB, 1 KB reserved each)
constexpr int kTilesPerPass = 4;            // tiles a warp reduces at once
// shared-memory header: 8 full + 8 empty mbarriers, flags, argmax keys
constexpr int kHeader = 256;

struct GemvPlan {
    int sg;           // tiles per stage
    int S;            // ring stages (1 when the slice is one copy)
    int G;            // CTAs
    int NG;           // 8-row groups
    int max_rows;     // rows of the largest CTA slice
    int resid_off;    // byte offset of the residual buffer (RESID mode)
    int planes;       // 1: activations as digit planes (large slices)
    int cs;           // 1: column-split consumer (batch 1, 2048-column tiles, several per row)
    int red8_off;     // byte offset of its per-warp row partials
    size_t stage_bytes;
    size_t smem;
};

// Activation row in shared memory, in floats: f32 padded (36 per 32 values),
// or digit planes (3 bytes per value) then block scales (f32 per 32 values).
__host__ __device__ inline int xs_floats_per_row(int K) { return (K / 32) * 36; }
__host__ __device__ inline int xs_plane_floats_per_row(int K) { return ((K * 3 + K / 8) / 4 + 3) / 4 * 4; }

__host__ __device__ inline size_t align128(size_t v) { return (v + 127) & ~static_cast<size_t>(127); }

// Plan for cps CTAs per SM: the slice of each CTA, one copy or a ring of
// stages, and the shared-memory layout within budget bytes. smem = 0 when the
// layout does not fit.
GemvPlan plan_for(const QMat &W, int N, int K, int B, int mode, int cps, size_t budget) {
    GemvPlan p{};
    p.NG = (N + 7) / 8;
    p.G = p.NG < cps * num_sms() ? p.NG : cps * num_sms();
    const int max_groups = (p.NG + p.G - 1) / p.G;
    p.max_rows = max_groups * 8;
    const size_t tb = qm_tile_bytes(W.kt);
    const int ntk = K / W.kt;
    const size_t slice = static_cast<size_t>(max_groups) * ntk * tb;
    p.planes = slice >= kPlanesMinSlice ? 1 : 0;
    const int xrow = p.planes ? xs_plane_floats_per_row(K) : xs_floats_per_row(K);
    size_t fixed = kHeader + static_cast<size_t>(B) * xrow * 4 + align128(static_cast<size_t>(p.max_rows) * B * 4) + 128;
    if (mode == GEMV_RESID) fixed += align128(static_cast<size_t>(p.max_rows) * B * 4);
    p.cs = (B == 1 && ntk > 1 && W.kt == 2048) ? 1 : 0;
    const size_t red8 = p.cs ? align128(static_cast<size_t>(max_groups) * 64 * 4) : 0;
    fixed += red8;
    if (fixed >= budget) return p;
    const size_t avail = budget - fixed;
    if (slice <= kOneShot && align128(slice) <= avail) {
        p.sg = max_groups * ntk;
        p.S = 1;
    } else {
        // ring: the largest stage (whole tiles, at most kStageTarget) of
        // which two fit, and as many of them as fit (at most kMaxStages).
        // A CTA's bulk copies complete at a roughly fixed rate, so big
        // stages beat many small ones (measured on the 8B gate/up rows:
        // two 35 KB stages 4.1 TB/s, five 17 KB stages 3.5 TB/s).
        int sg = static_cast<int>(kStageTarget / tb);
        if (sg < 1) sg = 1;
        for (; sg >= 1; --sg)
            if (avail / align128(static_cast<size_t>(sg) * tb) >= 2) break;
        if (sg < 1) return p;
        p.sg = sg;
        p.S = static_cast<int>(std::min<size_t>(kMaxStages, avail / align128(static_cast<size_t>(sg) * tb)));
    }
    p.stage_bytes = static_cast<size_t>(p.sg) * tb;
    size_t off = kHeader + align128(p.stage_bytes) * p.S + static_cast<size_t>(B) * xrow * 4;
    off += align128(static_cast<size_t>(p.max_rows) * B * 4) + 128 /*norm scratch*/;
    p.resid_off = static_cast<int>(off);
    if (mode == GEMV_RESID) off += align128(static_cast<size_t>(p.max_rows) * B * 4);
    p.red8_off = static_cast<int>(off);
    off += red8;
    if (off <= budget) p.smem = off;
    return p;
}

// Two CTAs per SM where the layout fits in half the SM's shared memory (twice
// the warps to hide the dequantise-and-dot latency, and twice the copies in
// flight), else one.
GemvPlan make_plan(const QMat &W, int N, int K, int B, int mode) {
    const GemvPlan p2 = plan_for(W, N, K, B, mode, 2, kSmemPair);
    if (p2.smem) return p2;
    return plan_for(W, N, K, B, mode, 1, kSmemMax);
}

// 16 activations of one lane, as 8 f32 pairs (read straight into 64-bit
// registers: no packing moves).
struct X16 {
    unsigned long long v[8];
};

__device__ __forceinline__ X16 load_x16(const float *xr) {
    X16 x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const ulonglong2 t = *reinterpret_cast<const ulonglong2 *>(xr + 4 * i);
        x.v[2 * i] = t.x;
        x.v[2 * i + 1] = t.y;
    }
    return x;
}

// One pair of codes (bytes SEL_LO, SEL_HI of an XOR-0x80 word) times an x
// pair, accumulated into ACC: prmt builds 2^23 + (q + 128) in each half,
// add.f32x2 removes 2^23 + 128 (exact), fma.f32x2 accumulates.
#define QW3_PAIR(WORD, SEL_LO, SEL_HI, X, ACC)              \
    "prmt.b32 l, " WORD ", 0x4B000000, " SEL_LO ";\n\t"      \
    "prmt.b32 h, " WORD ", 0x4B000000, " SEL_HI ";\n\t"      \
    "mov.b64 p, {l, h};\n\t"                                 \
    "add.rn.f32x2 p, p, bias;\n\t"                           \
    "fma.rn.f32x2 " ACC ", p, " X ", " ACC ";\n\t"

// Sum over 16 codes (w) of q * x, f32; two independent packed chains.
__device__ __forceinline__ float dot16(const uint4 w, const X16 &x) {
    float r;
    asm("{\n\t"
        ".reg .b32 t0, t1, t2, t3, l, h;\n\t"
        ".reg .b64 p, a, b, bias;\n\t"
        "mov.b64 bias, {%13, %13};\n\t"
        "mov.b64 a, 0;\n\t"
        "mov.b64 b, 0;\n\t"
        "xor.b32 t0, %1, 0x80808080;\n\t"
        "xor.b32 t1, %2, 0x80808080;\n\t"
        "xor.b32 t2, %3, 0x80808080;\n\t"
        "xor.b32 t3, %4, 0x80808080;\n\t"
        QW3_PAIR("t0", "0x7440", "0x7441", "%5", "a")
        QW3_PAIR("t0", "0x7442", "0x7443", "%6", "b")
        QW3_PAIR("t1", "0x7440", "0x7441", "%7", "a")
        QW3_PAIR("t1", "0x7442", "0x7443", "%8", "b")
        QW3_PAIR("t2", "0x7440", "0x7441", "%9", "a")
        QW3_PAIR("t2", "0x7442", "0x7443", "%10", "b")
        QW3_PAIR("t3", "0x7440", "0x7441", "%11", "a")
        QW3_PAIR("t3", "0x7442", "0x7443", "%12", "b")
        "add.rn.f32x2 a, a, b;\n\t"
        "mov.b64 {l, h}, a;\n\t"
        "add.rn.f32 %0, l, h;\n\t"
        "}"
        : "=f"(r)
        : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "l"(x.v[0]), "l"(x.v[1]), "l"(x.v[2]), "l"(x.v[3]),
          "l"(x.v[4]), "l"(x.v[5]), "l"(x.v[6]), "l"(x.v[7]), "f"(-8388736.0f));
    return r;
}
#undef QW3_PAIR

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Largest number of float4 loads of one activation row per consumer thread.
constexpr int kMaxXLoads = 12;   // K <= 12288
constexpr int kNormPre = 4;      // norm-weight float4 per thread fetched before the dependency wait (K <= 4096)

template <int B, int MODE, bool PL, bool CS>
__global__ void __launch_bounds__(kThreads, 2) k_gemv(GemvArgs a, GemvPlan p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int K = a.K;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned long long *tr = (tid == 0) ? trace_slot(a.trace) : nullptr;
    if (tr) {
        tr[0] = globaltimer_ns();
        tr[7] = smid();
    }
    const QMat &W = a.W;
    const int kt = W.kt;
    const int ntk = K / kt;                      // tiles per row group
    const size_t tb = qm_tile_bytes(kt);
    const size_t slot = align128(p.stage_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);          // [kMaxStages]
    uint64_t *empty = full + 8;                                    // [kMaxStages]
    volatile int *flags = reinterpret_cast<volatile int *>(smem + 128);                 // [8]
    unsigned long long *best = reinterpret_cast<unsigned long long *>(smem + 160);     // [4]
    uint8_t *ring = smem + kHeader;
    float *xs = reinterpret_cast<float *>(ring + slot * p.S);
    const int xrow = PL ? xs_plane_floats_per_row(K) : xs_floats_per_row(K);
    float *red = xs + B * xrow;                                    // [rows][B]
    float *nscr = red + align128(static_cast<size_t>(p.max_rows) * B * 4) / 4;  // [32]
    float *resid = reinterpret_cast<float *>(smem + p.resid_off);  // [rows][B] (RESID)

    const int g0 = static_cast<int>((static_cast<int64_t>(blockIdx.x) * p.NG) / gridDim.x);
    const int g1 = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * p.NG) / gridDim.x);
    const int row0 = g0 * 8;
    const int nrows = (g1 - g0) * 8;
    const int ntiles = (g1 - g0) * ntk;
    const int nst = (ntiles + p.sg - 1) / p.sg;
    const uint8_t *src = W.base + qm_tile_offset(W, g0, 0);

    if (tid == 0) {
        for (int i = 0; i < p.S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_mbar_init();
        flags[0] = 0;
        flags[1] = 0;
        flags[3] = 0;
    }
    if (MODE == GEMV_ARGMAX && tid < B) best[tid] = 0ull;
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int st = 0; st < nst; ++st) {
                const int si = st % p.S;
                if (st >= p.S && !mbar_wait_bounded(&empty[si], static_cast<uint32_t>(((st / p.S) - 1) & 1))) {
                    flags[0] = 1;
                    break;
                }
                if (flags[0]) break;
                const int t0 = st * p.sg;
                const int nt = min(p.sg, ntiles - t0);
                const uint32_t bytes = static_cast<uint32_t>(nt * tb);
                mbar_arrive_expect_tx(&full[si], bytes);
                bulk_g2s(ring + slot * si, src + t0 * tb, bytes, &full[si], pol);
                if (st == 0 && blockIdx.x == 0 && a.trace) a.trace[5] = globaltimer_ns();   // first copy issued
                flags[3] = st + 1;   // stages issued
            }
        }
        __syncwarp();
        pdl_trigger();
    } else {
        // ------------------------------------------------------ consumers
        // the norm weights do not depend on the previous kernel: fetch them
        // before the wait (rows up to kNormPre float4 per thread)
        const int nld = (K / 4 + kConsumers - 1) / kConsumers;   // float4 per thread
        const bool npre = a.norm_w != nullptr && nld <= kNormPre;
        float4 nw[kNormPre];
#pragma unroll
        for (int i = 0; i < kNormPre; ++i) {
            const int k = (tid + i * kConsumers) * 4;
            if (npre && i < nld && k < K) nw[i] = __ldg(reinterpret_cast<const float4 *>(a.norm_w + k));
        }
        pdl_trigger();
        pdl_wait();
        if (tr) tr[1] = globaltimer_ns();
        // residual rows of this CTA, fetched now so the epilogue does not wait
        if (MODE == GEMV_RESID) {
            for (int t = tid; t < nrows * B; t += kConsumers) {
                const int i = t / B, b = t % B;
                resid[t] = (row0 + i < a.N) ? a.y[static_cast<int64_t>(b) * a.N + row0 + i] : 0.0f;
            }
        }
        // activations: every load of a row in flight at once, then the norm
        for (int b = 0; b < B; ++b) {
            const float *xb = a.x + static_cast<int64_t>(b) * K;
            float4 v[kMaxXLoads];
#pragma unroll
            for (int i = 0; i < kMaxXLoads; ++i) {
                const int k = (tid + i * kConsumers) * 4;
                if (i < nld && k < K) v[i] = *reinterpret_cast<const float4 *>(xb + k);
            }
            float scale = 1.0f;
            if (a.norm_w) {
                float ss = 0.0f;
#pragma unroll
                for (int i = 0; i < kMaxXLoads; ++i) {
                    const int k = (tid + i * kConsumers) * 4;
                    if (i < nld && k < K) {
                        ss = fmaf(v[i].x, v[i].x, ss);
                        ss = fmaf(v[i].y, v[i].y, ss);
                        ss = fmaf(v[i].z, v[i].z, ss);
                        ss = fmaf(v[i].w, v[i].w, ss);
                    }
                }
                ss = warp_sum(ss);
                if (lane == 0) nscr[(b & 1) * 16 + warp] = ss;
                consumers_sync();
                float t = lane < kConsumerWarps ? nscr[(b & 1) * 16 + lane] : 0.0f;
                t = warp_sum(t);
                scale = 1.0f / sqrtf(t / static_cast<float>(K) + a.eps);
            }
            if constexpr (!PL) {
                float *xd = xs + b * xrow;
#pragma unroll
                for (int i = 0; i < kMaxXLoads; ++i) {
                    const int k = (tid + i * kConsumers) * 4;
                    if (i < nld) {   // uniform: every lane of the warp takes part in the round trip
                        const bool act = k < K;
                        float4 u = act ? v[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        if (a.norm_w && act) {
                            const float4 w = (i < kNormPre && npre) ? nw[i & (kNormPre - 1)]
                                                                    : *reinterpret_cast<const float4 *>(a.norm_w + k);
                            u.x = u.x * scale * w.x;
                            u.y = u.y * scale * w.y;
                            u.z = u.z * scale * w.z;
                            u.w = u.w * scale * w.w;
                        }
                        if (a.act_q8) u = q8_0_roundtrip4(u);
                        if (act) *reinterpret_cast<float4 *>(xd + (k >> 5) * 36 + (k & 31)) = u;
                    }
                }
            } else {
                // digit planes of the (normalised) row: 8 threads hold a 32-block
                uint8_t *xd = reinterpret_cast<uint8_t *>(xs + b * xrow);
                float *xsc = reinterpret_cast<float *>(xd + static_cast<size_t>(K) * 3);
#pragma unroll
                for (int i = 0; i < kMaxXLoads; ++i) {
                    if (i < nld) {
                        const int k = (tid + i * kConsumers) * 4;
                        const bool act = k < K;
                        float4 u = act ? v[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        if (a.norm_w && act) {
                            const float4 w = (i < kNormPre && npre) ? nw[i & (kNormPre - 1)]
                                                                    : *reinterpret_cast<const float4 *>(a.norm_w + k);
                            u.x = u.x * scale * w.x;
                            u.y = u.y * scale * w.y;
                            u.z = u.z * scale * w.z;
                            u.w = u.w * scale * w.w;
                        }
                        if (a.act_q8) u = q8_0_roundtrip4(u);
                        float amax = fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w)));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
                        if (act) {
                            const float sb = amax * (1.0f / 127.0f);
                            uint32_t ph = 0, pm = 0, pl = 0;
                            if (sb > 0.0f) {
                                const float vv[4] = {u.x, u.y, u.z, u.w};
                                digit_planes4(vv, __frcp_rn(sb), ph, pm, pl);
                            }
                            uint32_t *pw =
                                reinterpret_cast<uint32_t *>(xd + static_cast<size_t>(k >> 4) * 48) + ((k & 15) >> 2);
                            pw[0] = ph;
                            pw[4] = pm;
                            pw[8] = pl;
                            if ((k & 31) == 0) xsc[k >> 5] = sb;
                        }
                    }
                }
            }
        }
        consumers_sync();
        if (tr) tr[2] = globaltimer_ns();

        // Every warp consumes every stage: row `warp` of each tile.
        const int nchunk = (kt + 511) / 512;
        float carry[B];                       // running sum across k-tiles of a group
#pragma unroll
        for (int b = 0; b < B; ++b) carry[b] = 0.0f;
        // column-split consumer (batch 1, rows split into 2048-column tiles):
        // warp w takes the 256-column slice w of every tile for all 8 rows,
        // half-warp h rows h, h+2, h+4, h+6, so each lane's 16 activations
        // are read from shared memory once for four rows instead of once per
        // row; per-warp row partials of each group go to red8 and are summed
        // in a fixed order before the epilogue
        static_assert(!CS || B == 1, "the column-split consumer is for batch 1");
        float cacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float *red8 = reinterpret_cast<float *>(smem + p.red8_off);   // [groups][8 warps][8 rows]
        for (int st = 0; st < nst; ++st) {
            const int si = st % p.S;
            if (!mbar_wait_bounded(&full[si], static_cast<uint32_t>((st / p.S) & 1))) {
                flags[0] = 1;
                break;
            }
            if (tr && st == 0) tr[6] = globaltimer_ns();   // first stage landed
            const uint8_t *stage = ring + slot * si;
            const int t0 = st * p.sg;
            const int nt = min(p.sg, ntiles - t0);
            if constexpr (CS) {
                const int h = lane >> 4;
                const int cin = warp * 256 + (lane & 15) * 16;   // column within the tile
                for (int j = 0; j < nt; ++j) {
                    const int tile = t0 + j;
                    const int kti = tile % ntk;
                    const uint8_t *tp = stage + static_cast<size_t>(j) * tb;
                    const __half *sc = reinterpret_cast<const __half *>(tp + 8 * kt);
                    const int col = kti * kt + cin;               // column within the row
                    if constexpr (PL) {
                        const uint8_t *xd = reinterpret_cast<const uint8_t *>(xs);
                        const float sx = reinterpret_cast<const float *>(xd + static_cast<size_t>(K) * 3)[col >> 5];
                        uint4 P[3];
#pragma unroll
                        for (int q = 0; q < 3; ++q) P[q] = reinterpret_cast<const uint4 *>(xd)[(col >> 4) * 3 + q];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = h + 2 * i;
                            const uint4 w = *reinterpret_cast<const uint4 *>(tp + r * kt + cin);
                            const float d = __half2float(sc[r * (kt / 32) + (cin >> 5)]);
                            cacc[i] = fmaf(d * sx, pdot16(w, P), cacc[i]);
                        }
                    } else {
                        const X16 x = load_x16(xs + (col >> 5) * 36 + (col & 31));
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = h + 2 * i;
                            const uint4 w = *reinterpret_cast<const uint4 *>(tp + r * kt + cin);
                            const float d = __half2float(sc[r * (kt / 32) + (cin >> 5)]);
                            cacc[i] = fmaf(d, dot16(w, x), cacc[i]);
                        }
                    }
                    if (kti == ntk - 1) {
                        // the group's last k-tile: sum the 16 lanes of each half-warp
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                            for (int i = 0; i < 4; ++i) cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], o);
                        if ((lane & 15) == 0) {
                            float *dst = red8 + (tile / ntk) * 64 + warp * 8;
#pragma unroll
                            for (int i = 0; i < 4; ++i) dst[h + 2 * i] = cacc[i];
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) cacc[i] = 0.0f;
                    }
                }
            }
            for (int j0 = 0; j0 < (CS ? 0 : nt); j0 += kTilesPerPass) {
                const int np = min(kTilesPerPass, nt - j0);
                const uint8_t *tp0 = stage + static_cast<size_t>(j0) * tb;
                float acc[kTilesPerPass][B];
#pragma unroll
                for (int j = 0; j < kTilesPerPass; ++j)
#pragma unroll
                    for (int b = 0; b < B; ++b) acc[j][b] = 0.0f;
                // column offset of each tile of the pass within its row
                int kcol0[kTilesPerPass];
#pragma unroll
                for (int j = 0; j < kTilesPerPass; ++j) kcol0[j] = ntk == 1 ? 0 : ((t0 + j0 + j) % ntk) * kt;
                // A lone tile per pass (one row group per CTA, or one tile per
                // ring stage) has no second tile to overlap with: take its
                // chunks two at a time as independent chains instead. Lanes
                // past the tile's end read column 0 with zero codes and scale.
                const bool lone = B == 1 && np == 1;
                if (lone) {
                    const __half *dsc = reinterpret_cast<const __half *>(tp0 + 8 * kt) + warp * (kt / 32);
                    const int kc = kcol0[0];   // the tile's first column in the row
                    float s0 = 0.0f, s1 = 0.0f;
                    for (int c = 0; c < nchunk; c += 2) {
                        const int k0 = c * 512 + lane * 16, k1 = k0 + 512;
                        const bool v0 = k0 < kt, v1 = k1 < kt;
                        const int c0 = v0 ? k0 : 0, c1 = v1 ? k1 : 0;
                        const uint4 w0 = *reinterpret_cast<const uint4 *>(tp0 + warp * kt + c0);
                        const uint4 w1 = *reinterpret_cast<const uint4 *>(tp0 + warp * kt + c1);
                        const float d0 = v0 ? __half2float(dsc[c0 >> 5]) : 0.0f;
                        const float d1 = v1 ? __half2float(dsc[c1 >> 5]) : 0.0f;
                        const int x0c = kc + c0, x1c = kc + c1;
                        if constexpr (!PL) {
                            const X16 x0 = load_x16(xs + (x0c >> 5) * 36 + (x0c & 31));
                            const X16 x1 = load_x16(xs + (x1c >> 5) * 36 + (x1c & 31));
                            s0 = fmaf(d0, dot16(w0, x0), s0);
                            s1 = fmaf(d1, dot16(w1, x1), s1);
                        } else {
                            const uint8_t *xd = reinterpret_cast<const uint8_t *>(xs);
                            const float *xsc = reinterpret_cast<const float *>(xd + static_cast<size_t>(K) * 3);
                            uint4 P0[3], P1[3];
#pragma unroll
                            for (int q = 0; q < 3; ++q) {
                                P0[q] = reinterpret_cast<const uint4 *>(xd)[(x0c >> 4) * 3 + q];
                                P1[q] = reinterpret_cast<const uint4 *>(xd)[(x1c >> 4) * 3 + q];
                            }
                            s0 = fmaf(d0 * xsc[x0c >> 5], pdot16(w0, P0), s0);
                            s1 = fmaf(d1 * xsc[x1c >> 5], pdot16(w1, P1), s1);
                        }
                    }
                    acc[0][0] = s0 + s1;
                }
                for (int c = 0; c < (lone ? 0 : nchunk); ++c) {
                    const int kk = c * 512 + lane * 16;       // column within the tile
                    if (kk >= kt) continue;
                    if (ntk == 1) {
                        // every tile of the pass covers the same columns: load
                        // the pass's codes once, stream the activation rows
                        uint4 w[kTilesPerPass];
                        float d[kTilesPerPass];
#pragma unroll
                        for (int j = 0; j < kTilesPerPass; ++j) {
                            if (j < np) {
                                const uint8_t *tp = tp0 + static_cast<size_t>(j) * tb;
                                w[j] = *reinterpret_cast<const uint4 *>(tp + warp * kt + kk);
                                d[j] = __half2float(
                                    reinterpret_cast<const __half *>(tp + 8 * kt)[warp * (kt / 32) + (kk >> 5)]);
                            }
                        }
#pragma unroll
                        for (int b = 0; b < B; ++b) {
                            if constexpr (!PL) {
                                const X16 x = load_x16(xs + b * xrow + (kk >> 5) * 36 + (kk & 31));
#pragma unroll
                                for (int j = 0; j < kTilesPerPass; ++j)
                                    if (j < np) acc[j][b] = fmaf(d[j], dot16(w[j], x), acc[j][b]);
                            } else {
                                const uint8_t *xd = reinterpret_cast<const uint8_t *>(xs + b * xrow);
                                uint4 Pq[3];
#pragma unroll
                                for (int q = 0; q < 3; ++q) Pq[q] = reinterpret_cast<const uint4 *>(xd)[(kk >> 4) * 3 + q];
                                const float sx = reinterpret_cast<const float *>(xd + static_cast<size_t>(K) * 3)[kk >> 5];
#pragma unroll
                                for (int j = 0; j < kTilesPerPass; ++j)
                                    if (j < np) acc[j][b] = fmaf(d[j] * sx, pdot16(w[j], Pq), acc[j][b]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kTilesPerPass; ++j) {
                            if (j < np) {
                                const int kcol = kcol0[j] + kk;
                                const uint8_t *tp = tp0 + static_cast<size_t>(j) * tb;
                                const uint4 w = *reinterpret_cast<const uint4 *>(tp + warp * kt + kk);
                                const float d = __half2float(
                                    reinterpret_cast<const __half *>(tp + 8 * kt)[warp * (kt / 32) + (kk >> 5)]);
#pragma unroll
                                for (int b = 0; b < B; ++b) {
                                    if constexpr (!PL) {
                                        const X16 x = load_x16(xs + b * xrow + (kcol >> 5) * 36 + (kcol & 31));
                                        acc[j][b] = fmaf(d, dot16(w, x), acc[j][b]);
                                    } else {
                                        const uint8_t *xd = reinterpret_cast<const uint8_t *>(xs + b * xrow);
                                        uint4 Pq[3];
#pragma unroll
                                        for (int q = 0; q < 3; ++q)
                                            Pq[q] = reinterpret_cast<const uint4 *>(xd)[(kcol >> 4) * 3 + q];
                                        const float sx =
                                            reinterpret_cast<const float *>(xd + static_cast<size_t>(K) * 3)[kcol >> 5];
                                        acc[j][b] = fmaf(d * sx, pdot16(w, Pq), acc[j][b]);
                                    }
                                }
                            }
                        }
                    }
                }
                // one butterfly for the pass (independent chains)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int j = 0; j < kTilesPerPass; ++j)
#pragma unroll
                        for (int b = 0; b < B; ++b)
                            if (j < np) acc[j][b] += __shfl_xor_sync(0xffffffffu, acc[j][b], o);
#pragma unroll
                for (int j = 0; j < kTilesPerPass; ++j) {
                    if (j < np) {
                        const int tile = t0 + j0 + j;
#pragma unroll
                        for (int b = 0; b < B; ++b) carry[b] += acc[j][b];
                        const int kt_idx = ntk == 1 ? 0 : tile % ntk;
                        if (kt_idx == ntk - 1) {          // last k-tile of its group
                            if (lane == 0) {
                                const int rloc = (ntk == 1 ? tile : tile / ntk) * 8 + warp;
#pragma unroll
                                for (int b = 0; b < B; ++b) red[rloc * B + b] = carry[b];
                            }
#pragma unroll
                            for (int b = 0; b < B; ++b) carry[b] = 0.0f;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[si]);
        }
    }
    __syncthreads();
    if (tr) tr[3] = globaltimer_ns();

    if (flags[0]) {
        // A stage never completed: report, drain the copies that may still be
        // in flight (the last S issued stages, bounded waits), and leave.
        if (tid == 0) {
            record_status(a.status, QW3_ERR_TIMEOUT);
            const int issued = flags[3];
            for (int st = issued > p.S ? issued - p.S : 0; st < issued; ++st)
                (void)mbar_wait_bounded(&full[st % p.S], static_cast<uint32_t>((st / p.S) & 1));
        }
        return;
    }

    if constexpr (CS) {
        // row sums of the column-split consumer: the 8 warps' partials in order
        const float *red8 = reinterpret_cast<const float *>(smem + p.red8_off);
        for (int t = tid; t < nrows; t += kThreads) {
            const float *src = red8 + (t >> 3) * 64 + (t & 7);
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) v += src[w * 8];
            red[t] = v;
        }
        __syncthreads();
    }

    // ---- epilogue over the CTA's rows
    float *yout = a.y;
    if (MODE == GEMV_ARGMAX && a.io) yout = a.io->logits;
    if (MODE == GEMV_SWIGLU) {
        for (int t = tid; t < (nrows / 2) * B; t += kThreads) {
            const int i = 2 * (t / B), b = t % B;
            const float g = red[i * B + b];
            const float u = red[(i + 1) * B + b];
            const int r = row0 + i;
            if (r < a.N) a.y[static_cast<int64_t>(b) * (a.N / 2) + r / 2] = g / (1.0f + expf(-g)) * u;
        }
    } else {
        unsigned long long mykey[B];
#pragma unroll
        for (int b = 0; b < B; ++b) mykey[b] = 0ull;
        for (int t = tid; t < nrows * B; t += kThreads) {
            const int i = t / B, b = t % B;
            const float y = red[i * B + b];
            const int r = row0 + i;
            if (r < a.N) {
                if (MODE == GEMV_STORE) {
                    yout[static_cast<int64_t>(b) * a.N + r] = y;
                } else if (MODE == GEMV_RESID) {
                    yout[static_cast<int64_t>(b) * a.N + r] = resid[t] + y;
                } else {
                    if (yout) yout[static_cast<int64_t>(b) * a.N + r] = y;
                    const unsigned long long k = argmax_pack(y, r);
#pragma unroll
                    for (int bb = 0; bb < B; ++bb)
                        if (bb == b) mykey[bb] = k > mykey[bb] ? k : mykey[bb];
                }
            }
        }
        if (MODE == GEMV_ARGMAX) {
#pragma unroll
            for (int b = 0; b < B; ++b) {
                unsigned long long k = mykey[b];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
                    k = other > k ? other : k;
                }
                if (lane == 0 && k) atomicMax(&best[b], k);
            }
        }
    }

    if (MODE == GEMV_ARGMAX) {
        __syncthreads();
        if (tid < B) atomicMax(&a.argmax_key[tid], best[tid]);
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const unsigned prev = atomicAdd(a.done_counter, 1u);
            flags[1] = (prev == gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (flags[1]) {
            __threadfence();
            const int step = a.step_ctr ? *a.step_ctr : 0;
            int32_t *argmax_out = a.io ? a.io->argmax : a.argmax_out;
            int32_t *tok_hist = a.io ? a.io->hist : nullptr;
            if (tid < B) {
                const unsigned long long key = atomicAdd(&a.argmax_key[tid], 0ull);
                const int idx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(key & 0xffffffffull));
                const float v = float_from_order_key(static_cast<uint32_t>(key >> 32));
                if (isnan(v)) record_status(a.status, QW3_ERR_NONFINITE);
                if (argmax_out) argmax_out[tid] = idx;
                if (a.next_token) a.next_token[tid] = idx;
                if (tok_hist) tok_hist[static_cast<int64_t>(step) * B + tid] = idx;
                if (a.pos_inc) a.pos_inc[tid] += 1;
                a.argmax_key[tid] = 0ull;
            }
            __syncthreads();
            if (tid == 0) {
                *a.done_counter = 0u;
                if (a.step_ctr) *a.step_ctr = step + 1;
            }
        }
    }
    if (tr) tr[4] = globaltimer_ns();
}

template <int B, int MODE, bool PL, bool CS = false>
cudaError_t configure_one() {
    cudaError_t e = cudaFuncSetAttribute(k_gemv<B, MODE, PL, CS>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    // Same carveout for every decode kernel: an SM never has to drain to
    // reconfigure L1/shared memory between PDL-overlapped kernels.
    return cudaFuncSetAttribute(k_gemv<B, MODE, PL, CS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

template <int B>
cudaError_t configure_b() {
    cudaError_t e;
    if ((e = configure_one<B, GEMV_STORE, false>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_RESID, false>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_SWIGLU, false>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_ARGMAX, false>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_STORE, true>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_RESID, true>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_SWIGLU, true>()) != cudaSuccess) return e;
    if ((e = configure_one<B, GEMV_ARGMAX, true>()) != cudaSuccess) return e;
    if constexpr (B == 1) {
        if ((e = configure_one<1, GEMV_STORE, false, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_RESID, false, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_SWIGLU, false, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_ARGMAX, false, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_STORE, true, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_RESID, true, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_SWIGLU, true, true>()) != cudaSuccess) return e;
        if ((e = configure_one<1, GEMV_ARGMAX, true, true>()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int B, int MODE>
cudaError_t launch_one(const GemvArgs &a, const GemvPlan &p, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(p.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if constexpr (B == 1) {
        if (p.cs) {
            if (p.planes) return cudaLaunchKernelEx(&cfg, k_gemv<1, MODE, true, true>, a, p);
            return cudaLaunchKernelEx(&cfg, k_gemv<1, MODE, false, true>, a, p);
        }
    }
    if (p.planes) return cudaLaunchKernelEx(&cfg, k_gemv<B, MODE, true, false>, a, p);
    return cudaLaunchKernelEx(&cfg, k_gemv<B, MODE, false, false>, a, p);
}

template <int B>
cudaError_t launch_b(const GemvArgs &a, int mode, const GemvPlan &p, bool pdl, cudaStream_t s) {
    switch (mode) {
        case GEMV_STORE: return launch_one<B, GEMV_STORE>(a, p, pdl, s);
        case GEMV_RESID: return launch_one<B, GEMV_RESID>(a, p, pdl, s);
        case GEMV_SWIGLU: return launch_one<B, GEMV_SWIGLU>(a, p, pdl, s);
        case GEMV_ARGMAX: return launch_one<B, GEMV_ARGMAX>(a, p, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t configure_gemv() {
    cudaError_t e;
    if ((e = configure_b<1>()) != cudaSuccess) return e;
    if ((e = configure_b<2>()) != cudaSuccess) return e;
    if ((e = configure_b<3>()) != cudaSuccess) return e;
    return configure_b<4>();
}

cudaError_t launch_gemv(const GemvArgs &a, int mode, bool pdl, cudaStream_t s) {
    if (a.K % 32 != 0 || a.B < 1 || a.B > 4 || a.W.cols != a.K || a.W.ktile_major) return cudaErrorInvalidValue;
    // a consumer thread loads at most kMaxXLoads float4 of a row; the staged
    // rows must fit in shared memory next to the ring
    if (a.K > kMaxXLoads * 4 * kConsumers || a.B * a.K > kGemvMaxBK) return cudaErrorInvalidValue;
    const GemvPlan p = make_plan(a.W, a.N, a.K, a.B, mode);
    if (p.smem == 0) return cudaErrorInvalidValue;
    switch (a.B) {
        case 1: return launch_b<1>(a, mode, p, pdl, s);
        case 2: return launch_b<2>(a, mode, p, pdl, s);
        case 3: return launch_b<3>(a, mode, p, pdl, s);
        case 4: return launch_b<4>(a, mode, p, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qw3
