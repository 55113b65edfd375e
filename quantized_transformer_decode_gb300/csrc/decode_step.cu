// Persistent batch-1 decode step: one launch per generated token.
//
// What it computes is one greedy decode step of "A transformer from
// scratch" (sections 12.3-12.6) with the Qwen3 deltas of minfer's "Qwen3
// Support Plan (dense)" (section 2): x = dequant(E[token]); per layer
// RMSNorm -> [q; k; v] projection -> per-head Q/K RMSNorm -> NeoX RoPE ->
// KV append -> causal GQA over the f32 cache -> o_proj + residual -> RMSNorm
// -> gate/up -> SwiGLU -> down + residual; final RMSNorm, lm_head, argmax
// (lowest index on ties); the argmax is the next step's token.
//
// Why one kernel: at batch 1 a 0.6B-parameter layer moves ~22 MB, about
// 3 us of HBM time, while a dependent kernel launch costs 2 us or more on
// GB300 before it does any work. Here one CTA per SM stays resident for the
// whole step; each dependency costs one hand-off through L2.
//
// Data flow. Warp 16 of each CTA is a producer: it streams, in the order the
// consumers use them, the CTA's slices of every layer's weights (whole 8-row
// tiles of the repacked Q8_0 matrices) and its share of the cached K/V rows
// (which do not depend on this step) through a ring of shared-memory slots
// with 1-D bulk copies (TMA), then the lm_head rows. It never waits on the
// dependency chain, only for free slots. Warps 0-15 run the phases of each
// layer:
//   P1 [q; k; v] rows of the CTA (RMSNorm folded in: the dot runs on x * w
//      and the row sums are scaled by 1 / rms(x)),
//   P2 attention unit (kv head g, split j): Q/K norm + RoPE of the new
//      token, scores over the unit's cached positions and the new one,
//      online softmax; a partial (acc, max, sum) per query head,
//   P3 combine of the S partials of one kv head for a slice of its outputs,
//   P4 o_proj + residual over the CTA's rows of x,
//   P5 gate/up + SwiGLU rows (interleaved gate/up rows),
//   P6 down + residual over the same rows of x as P4.
//
// Hand-offs. A phase writes its outputs to a global f32 buffer; each writing
// thread fences, the CTA synchronises, and one thread adds 1 to an arrival
// counter with release semantics. A reader waits (one warp per CTA, with
// backoff) until the counters it needs reach the number of writers times the
// layer count, then reads the buffer through L2 (ld.global.cg). Counters are
// split eight ways (writer CTA c adds to counter c % 8) so no counter takes
// more than a few dozen atomics per phase, and the step's last CTA clears
// them all. Polling one word per counter keeps the waiting CTAs from
// flooding the L2 slices that also serve the weight stream (polling every
// data word did, and delayed the weight copies by microseconds). Each buffer
// is rewritten only after every reader of its previous contents has
// finished (each phase needs the complete output of the one before).
//
// Arithmetic. The activations of a projection are staged per CTA as three
// int8 digit planes per 32-value block, x = s (h + m / 254 + l / 254^2),
// s = max|x| / 127, within s / (2 * 254^2) ~ 6e-8 of the block maximum (an
// f32 rounding); 16 codes times 16 such values are 12 exact int8 dot
// products (dp4a), combined in f32 with the weight and activation scales.
// Sums are f32.
//
// Waits. Ring waits are bounded by 1 s; waits on other CTAs by wait_ns. A
// wait that gives up records QW3_ERR_TIMEOUT, marks the step aborted (every
// later wait on other CTAs returns at once) and the kernel runs to its end,
// draining its copies.
#include <algorithm>
#include <cmath>

#include "decode_step.cuh"

namespace qw3 {

namespace {

constexpr int kCW = kStepConsumerWarps;
constexpr int kCT = kCW * 32;          // consumer threads
constexpr int kMaxK = 12288;           // widest activation vector
constexpr int kSub = 8;                // split of each global arrival counter

__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"n"(kCT) : "memory"); }

// ------------------------------------------------------ hand-off counters

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_relaxed_add(unsigned *p, unsigned v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Tagged 64-bit words: f32 value in the low half, the step/phase tag in the
// high half. A single 64-bit access is atomic, so a reader that sees the tag
// sees the value published with it; no fence orders data and counters.
__device__ __forceinline__ unsigned long long *LLB(float *p) { return reinterpret_cast<unsigned long long *>(p); }

__device__ __forceinline__ void ll_st(float *buf, int i, float v, unsigned tag) {
    const unsigned long long w = (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(LLB(buf) + i), "l"(w) : "memory");
}

__device__ __forceinline__ void ll_ld2(const unsigned long long *p, unsigned long long &a, unsigned long long &b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ unsigned long long ll_ld1(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ bool ll_ok(unsigned long long w, unsigned tag) { return static_cast<unsigned>(w >> 32) == tag; }
__device__ __forceinline__ float ll_val(unsigned long long w) { return __uint_as_float(static_cast<unsigned>(w)); }

constexpr unsigned kTagStride = 1024;
__device__ __forceinline__ unsigned step_tag(unsigned epoch, int layer, int phase) {
    return epoch * kTagStride + static_cast<unsigned>(kStepPhases * layer + phase);
}

struct WaitCtx {
    const StepParams *P;
    unsigned epoch;
};

__device__ __forceinline__ bool step_aborted(const WaitCtx &w) { return ld_relaxed_u32(w.P->abort_word) == w.epoch; }

__device__ __noinline__ void step_abort(const WaitCtx &w) {
    atomicExch(w.P->abort_word, w.epoch);
    record_status(w.P->status, QW3_ERR_TIMEOUT);
}

// Limits of waits on other CTAs are kept in SM cycles (clock64 is cheap;
// %globaltimer and the abort word are read only every 256 polls).
// wait_ns == 0 (a test setting) gives up at the first miss.
__device__ __forceinline__ bool wait_expired(const WaitCtx &w, long long c0, int it) {
    if (w.P->wait_ns == 0) return true;
    if ((it & 255) != 255) return false;
    return clock64() - c0 > static_cast<long long>(w.P->wait_ns) * 4;   // >= 1 ns per 4 cycles up to 4 GHz
}

// Wait (one thread) until *ctr >= target (wrap-safe), with backoff.
__device__ __forceinline__ void wait_count(const unsigned *ctr, unsigned target, const WaitCtx &w) {
    if (static_cast<int>(ld_relaxed_u32(ctr) - target) >= 0) return;
    const long long c0 = clock64();
    for (int it = 1;; ++it) {
        if (it > 4) __nanosleep(32);
        if (static_cast<int>(ld_relaxed_u32(ctr) - target) >= 0) return;
        if ((it & 255) == 255 && step_aborted(w)) return;
        if (wait_expired(w, c0, it)) {
            step_abort(w);
            return;
        }
    }
}

// A wait on n writers' counter stops once all but n / 4 of them arrived;
// the readers then poll the few words still missing directly (their tags),
// which skips one L2 round trip on the critical path while keeping the
// polling to the tail of the hand-off.
__device__ __forceinline__ unsigned gate(unsigned target, unsigned n) { return target - n / 4; }

// Counter i of the step's counter array (128-byte apart).
__device__ __forceinline__ unsigned *ctr_at(const StepParams &P, int i) { return P.ctrs + 32 * i; }

// Wait for the eight split counters base..base+7 to reach mult * n[s] each
// (warp 0's lanes 0-7 poll, then every consumer thread synchronises).
__device__ __forceinline__ void wait_split(const StepParams &P, int base, const unsigned *n, unsigned mult,
                                           const WaitCtx &w, int tid) {
    if (tid < kSub) wait_count(ctr_at(P, base + tid), mult * n[tid], w);
    csync();
}

// After a phase's writes: the CTA synchronises, then one thread adds the
// CTA's arrival (relaxed: the readers check every word's tag, so the counter
// only has to say "probably published" and costs no fence). Called by all
// consumer threads. The GEMV phases and the attention units add theirs
// earlier, as soon as their dot products are done and before their
// epilogue writes the words: the readers' counter wait then overlaps that
// epilogue, and their tag polls catch the words as they land (measured
// 556 -> 536 us per 0.6B token).
__device__ __forceinline__ void arrive(unsigned *ctr, bool wrote, int tid) {
    csync();
    if (tid == 0 && wrote) red_relaxed_add(ctr, 1u);
}

// Read N (2 or 4) tagged words at word index i of buf, re-reading until all
// carry the tag (the arrival counters are relaxed: a word can trail its
// counter by a little); v receives the values. The re-reads do not sleep
// between rounds: they run only in a hand-off's tail (measured faster than
// a 32 ns back-off).
template <int N>
__device__ __forceinline__ void ll_read(const float *buf, int i, unsigned tag, float (&v)[N], const WaitCtx &w) {
    const unsigned long long *p = reinterpret_cast<const unsigned long long *>(buf) + i;
    unsigned long long u[N];
    ll_ld2(p, u[0], u[1]);
    if constexpr (N == 4) ll_ld2(p + 2, u[2], u[3]);
    bool ok = true;
#pragma unroll
    for (int k = 0; k < N; ++k) ok = ok && ll_ok(u[k], tag);
    if (!ok) {
        const long long c0 = clock64();
        for (int it = 1;; ++it) {
            ll_ld2(p, u[0], u[1]);
            if constexpr (N == 4) ll_ld2(p + 2, u[2], u[3]);
            ok = true;
#pragma unroll
            for (int k = 0; k < N; ++k) ok = ok && ll_ok(u[k], tag);
            if (ok) break;
            if ((it & 255) == 255 && step_aborted(w)) break;
            if (wait_expired(w, c0, it)) {
                step_abort(w);
                break;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = ll_val(u[k]);
}

__device__ __forceinline__ float ll_read1(const float *buf, int i, unsigned tag, const WaitCtx &w) {
    const unsigned long long *p = reinterpret_cast<const unsigned long long *>(buf) + i;
    unsigned long long u = ll_ld1(p);
    if (!ll_ok(u, tag)) {
        const long long c0 = clock64();
        for (int it = 1;; ++it) {
            __nanosleep(32);
            u = ll_ld1(p);
            if (ll_ok(u, tag)) break;
            if ((it & 255) == 255 && step_aborted(w)) break;
            if (wait_expired(w, c0, it)) {
                step_abort(w);
                break;
            }
        }
    }
    return ll_val(u);
}

// ----------------------------------------------------- ring of slots

struct Ring {
    uint64_t *full;    // [NS]
    uint64_t *empty;   // [NS] (one arrival per consumer warp)
    uint8_t *base;
    int NS;
    uint32_t SB;
    unsigned long long *ctr;   // nullable trace: when consumer thread 0 obtained chunk n < 32
};

// Bounded wait on a ring barrier phase: 1 s, or 2 ms once the step has been
// aborted (the chain is broken; the copies themselves complete in
// microseconds).
__device__ __noinline__ bool ring_bar_wait_slow(uint64_t *bar, uint32_t parity, const WaitCtx &w) {
    const long long c0 = clock64();
    long long limit = static_cast<long long>(kWaitLimitNs) * 4;
    for (int it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255) == 255) {
            if (step_aborted(w)) limit = 2000000ll * 4;
            if (clock64() - c0 > limit) {
                step_abort(w);
                return false;
            }
        }
    }
}

// The fast path inline (a landed chunk costs one try_wait), the loop out of
// line (a call would make every caller save its live registers).
__device__ __forceinline__ bool ring_bar_wait(uint64_t *bar, uint32_t parity, const WaitCtx &w) {
    if (mbar_try_wait(bar, parity)) return true;
    return ring_bar_wait_slow(bar, parity, w);
}

// Wait for chunk n; returns its slot.
__device__ __forceinline__ const uint8_t *ring_wait(const Ring &r, uint32_t n, const WaitCtx &w) {
    const uint32_t slot = n % r.NS;
    (void)ring_bar_wait(&r.full[slot], (n / r.NS) & 1u, w);
    if (r.ctr && n < 32 && threadIdx.x == 0) r.ctr[n] = clock64();
    return r.base + static_cast<size_t>(slot) * r.SB;
}

__device__ __forceinline__ void ring_release(const Ring &r, uint32_t n, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&r.empty[n % r.NS]);
}

// ------------------------------------------------- activation planes

// Byte offset of the plane word of values [k, k + 4) (k % 4 == 0) in the
// plane layout of LC-value lane chunks: plane q of values [LC c, LC c + LC)
// is the LC-byte run at (3 c + q) LC.
template <int LC>
__device__ __forceinline__ uint32_t plane_off(int k, int q) {
    return static_cast<uint32_t>(((k / LC) * 3 + q) * LC + ((k % LC) / 4) * 4);
}

// Stage K values (K % 128 == 0; from x through L2, or from the embedding
// row when x is null) as digit planes and block scales, the values
// multiplied by norm_w when given; each warp's sum of squares of the raw
// values goes to ssw[warp] (norm only). The caller synchronises after.
template <int LC>
__device__ __forceinline__ void stage_planes(const float *x, unsigned tag, const WaitCtx &w, const QMat *emb, int tok,
                                             int K, const float *norm_w, uint8_t *planes, float *scales, float *ssw,
                                             int tid) {
    const int lane = tid & 31;
    float ss = 0.0f;
#pragma unroll 1
    for (int i = tid; i < K / 4; i += kCT) {
        const int k = 4 * i;
        float v[4];
        if (x) {
            ll_read<4>(x, k, tag, v, w);
        } else {
            const int32_t c4 = *reinterpret_cast<const int32_t *>(qm_codes(*emb, tok, k));
            const float d = __half2float(*qm_scale(*emb, tok, k));
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = d * static_cast<float>(static_cast<int8_t>((c4 >> (8 * j)) & 0xff));
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) ss = fmaf(v[j], v[j], ss);
        if (norm_w) {
            const float4 nw = __ldg(reinterpret_cast<const float4 *>(norm_w + k));
            v[0] *= nw.x;
            v[1] *= nw.y;
            v[2] *= nw.z;
            v[3] *= nw.w;
        }
        float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        const float sb = amax * (1.0f / 127.0f);
        uint32_t ph = 0, pm = 0, pl = 0;
        if (sb > 0.0f) digit_planes4(v, __frcp_rn(sb), ph, pm, pl);
        *reinterpret_cast<uint32_t *>(planes + plane_off<LC>(k, 0)) = ph;
        *reinterpret_cast<uint32_t *>(planes + plane_off<LC>(k, 1)) = pm;
        *reinterpret_cast<uint32_t *>(planes + plane_off<LC>(k, 2)) = pl;
        if ((k & 31) == 0) scales[k >> 5] = sb;
    }
    if (norm_w) {
        ss = warp_sum(ss);
        if (lane == 0) ssw[tid >> 5] = ss;
    }
}

// ------------------------------------------------------- dot products

__device__ __forceinline__ float pdot8(const uint2 w, const uint2 (&P)[3]) {
    int a = __dp4a(static_cast<int>(w.x), static_cast<int>(P[0].x), 0);
    a = __dp4a(static_cast<int>(w.y), static_cast<int>(P[0].y), a);
    int b = __dp4a(static_cast<int>(w.x), static_cast<int>(P[1].x), 0);
    b = __dp4a(static_cast<int>(w.y), static_cast<int>(P[1].y), b);
    int c = __dp4a(static_cast<int>(w.x), static_cast<int>(P[2].x), 0);
    c = __dp4a(static_cast<int>(w.y), static_cast<int>(P[2].y), c);
    return fmaf(static_cast<float>(c), 1.0f / 64516.0f, fmaf(static_cast<float>(b), 1.0f / 254.0f, static_cast<float>(a)));
}

// acc[r] += sum over the lane's LC columns of row r of one 8-row tile times
// the staged activations. colt: the lane's first column within the tile;
// colx: the same column within the activation vector.
template <int LC>
__device__ __forceinline__ void dot_rows8(const uint8_t *tile, int kt, int colt, int colx, const uint8_t *planes,
                                          const float *scales, float (&acc)[8]) {
    const float sx = scales[colx >> 5];
    const __half *dsc = reinterpret_cast<const __half *>(tile + 8 * static_cast<size_t>(kt)) + (colt >> 5);
    if constexpr (LC == 16) {
        uint4 P[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) P[q] = *reinterpret_cast<const uint4 *>(planes + ((colx >> 4) * 3 + q) * 16);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint4 wv = *reinterpret_cast<const uint4 *>(tile + r * kt + colt);
            const float d = __half2float(dsc[r * (kt >> 5)]);
            acc[r] = fmaf(d * sx, pdot16(wv, P), acc[r]);
        }
    } else {
        uint2 P[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) P[q] = *reinterpret_cast<const uint2 *>(planes + ((colx >> 3) * 3 + q) * 8);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint2 wv = *reinterpret_cast<const uint2 *>(tile + r * kt + colt);
            const float d = __half2float(dsc[r * (kt >> 5)]);
            acc[r] = fmaf(d * sx, pdot8(wv, P), acc[r]);
        }
    }
}

// Sum 8 per-lane values over the warp: lane l ends with the total of row
// red8_row(l) (every row is held by four lanes: l with l % 4 == 0 is one).
__device__ __forceinline__ int red8_row(int lane) {
    return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

__device__ __forceinline__ float reduce8(float (&v)[8], int lane) {
    {
        const bool up = lane & 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float send = up ? v[i] : v[i + 4];
            const float keep = up ? v[i + 4] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    {
        const bool up = lane & 8;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float send = up ? v[i] : v[i + 2];
            const float keep = up ? v[i + 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    {
        const bool up = lane & 4;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float t = v[0];
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    return t;
}


// ------------------------------------------------------- matrix slices

// Rows [8 g0, 8 g1) of a row-group-major tiled matrix: ng groups of ntk
// tiles, contiguous from src; streamed tpc whole tiles per ring chunk.
struct Slice {
    const uint8_t *src;
    int ng, ntk, kt, tpc, row0;
    uint32_t tb;
};

__host__ __device__ inline void group_range(int NG, int c, int NCTA, int &g0, int &g1) {
    g0 = static_cast<int>((static_cast<int64_t>(c) * NG) / NCTA);
    g1 = static_cast<int>((static_cast<int64_t>(c + 1) * NG) / NCTA);
}

__device__ __forceinline__ Slice make_slice(const QMat &W, int c, int NCTA, uint32_t SB) {
    Slice s;
    int g0, g1;
    group_range((W.rows + 7) / 8, c, NCTA, g0, g1);
    s.ng = g1 - g0;
    s.kt = W.kt;
    s.ntk = W.cols / W.kt;
    s.tb = static_cast<uint32_t>(qm_tile_bytes(W.kt));
    s.tpc = static_cast<int>(SB / s.tb);
    s.row0 = g0 * 8;
    s.src = W.base + qm_tile_offset(W, g0, 0);
    return s;
}

// Layer l's copy of a layer-0 pointer (layers are laid out at a fixed stride).
template <typename T>
__device__ __forceinline__ T *at_layer(T *p0, int l, size_t lstride) {
    return reinterpret_cast<T *>(reinterpret_cast<uintptr_t>(p0) + static_cast<uintptr_t>(l) * lstride);
}

__device__ __forceinline__ Slice slice_at(const Slice &s0, int l, size_t lstride) {
    Slice s = s0;
    s.src = at_layer(s0.src, l, lstride);
    return s;
}

__device__ __forceinline__ int slice_chunks(const Slice &s) {
    return (s.ng * s.ntk + s.tpc - 1) / s.tpc;
}

// Dot tasks of one phase: task = (tile, LC*32-column segment), warp w takes
// tasks w, w + 16, ...; the 8 row partials of each task go to red[task][8].
// Every consumer warp waits for and releases every chunk of the slice, in
// order (a slot is refilled only once all of them are done with it).
template <int LC>
__device__ __forceinline__ void gemv_tasks(const Slice sl, const Ring ring, uint32_t &n, const uint8_t *planes,
                                        const float *scales, float *red, const WaitCtx w, int warp, int lane,
                                        unsigned long long *tr) {
    constexpr int kSeg = 32 * LC;
    const int nseg = sl.kt / kSeg;
    const int ntile = sl.ng * sl.ntk;
    const int ntask = ntile * nseg;
    const int nch = slice_chunks(sl);
    int task = warp;
    // (tile, segment) of `task` walked without runtime divisions
    int tile = 0, seg = task;
    while (seg >= nseg) {
        seg -= nseg;
        ++tile;
    }
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        const uint8_t *slot = ring_wait(ring, n, w);
        if (tr && c == 0) tr[1] = clock64();
        const int tile_end = min(ntile, (c + 1) * sl.tpc);
#pragma unroll 1
        for (; task < ntask && tile < tile_end; task += kCW) {
            int kti = tile;
            while (kti >= sl.ntk) kti -= sl.ntk;
            const uint8_t *tp = slot + static_cast<size_t>(tile - c * sl.tpc) * sl.tb;
            const int colt = seg * kSeg + lane * LC;
            float acc[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
            dot_rows8<LC>(tp, sl.kt, colt, kti * sl.kt + colt, planes, scales, acc);
            const float t = reduce8(acc, lane);
            if ((lane & 3) == 0) red[task * 8 + red8_row(lane)] = t;
            seg += kCW;
            while (seg >= nseg) {
                seg -= nseg;
                ++tile;
            }
        }
        ring_release(ring, n, lane);
        ++n;
    }
    if (tr) tr[2] = clock64();
}

// Sum of the task partials of local row t of the slice (fixed order).
template <int LC>
__device__ __forceinline__ float row_sum(const Slice &sl, const float *red, int t) {
    const int nseg = sl.kt / (32 * LC);
    const int gi = t >> 3, rr = t & 7;
    float y = 0.0f;
    for (int kti = 0; kti < sl.ntk; ++kti)
        for (int seg = 0; seg < nseg; ++seg) y += red[((gi * sl.ntk + kti) * nseg + seg) * 8 + rr];
    return y;
}

// 1 / rms of the staged vector from the warps' sums of squares; called by
// whole warps (the 16 partials are summed by a shuffle tree).
__device__ __forceinline__ float norm_scale(const float *ssw, int K, float eps) {
    const int lane = threadIdx.x & 31;
    float t = lane < kCW ? ssw[lane] : 0.0f;
    t = warp_sum(t);
    return 1.0f / sqrtf(t / static_cast<float>(K) + eps);
}


// ------------------------------------------------------------ attention

template <int HD>
__device__ __forceinline__ void lane_load(const float *src, float (&v)[HD / 32], int lane) {
    if constexpr (HD == 128) {
        const float4 t = *reinterpret_cast<const float4 *>(src + lane * 4);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2 *>(src + lane * 2);
        v[0] = t.x; v[1] = t.y;
    }
}

// The same, through L2 (buffers written by other CTAs).
template <int HD>
__device__ __forceinline__ void lane_load_cg(const float *src, float (&v)[HD / 32], int lane) {
    if constexpr (HD == 128) {
        const float4 t = __ldcg(reinterpret_cast<const float4 *>(src + lane * 4));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        const float2 t = __ldcg(reinterpret_cast<const float2 *>(src + lane * 2));
        v[0] = t.x; v[1] = t.y;
    }
}

template <int HD>
__device__ __forceinline__ void lane_store(float *dst, const float (&v)[HD / 32], int lane) {
    if constexpr (HD == 128) {
        *reinterpret_cast<float4 *>(dst + lane * 4) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        *reinterpret_cast<float2 *>(dst + lane * 2) = make_float2(v[0], v[1]);
    }
}

// Per-head RMSNorm over head_dim (minfer 2.2) then the NeoX rotation of the
// pairs (i, i + hd/2) by p * theta^(-2i/hd) (course 12.3.4): lane l holds
// dims [l E, l E + E); its partner half sits in lane l ^ 16.
template <int HD>
__device__ __forceinline__ void norm_rope(float (&v)[HD / 32], const float (&nw)[HD / 32], const float2 (&cs)[HD / 32],
                                          float eps, int lane) {
    constexpr int E = HD / 32;
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
    ss = warp_sum(ss);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(HD) + eps);
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = v[e] * r * nw[e];
    const bool lo = lane < 16;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[e], 16);
        v[e] = lo ? (v[e] * cs[e].x - o * cs[e].y) : (o * cs[e].y + v[e] * cs[e].x);
    }
}

// Position range of attention unit (g, j): [a, b) of the context 0..p.
struct UnitRange {
    int g, j, a, b, ncached;
    bool has_new;
};

__device__ __forceinline__ UnitRange unit_range(int unit, int S, int p) {
    UnitRange u;
    u.g = unit / S;
    u.j = unit - u.g * S;
    const int ctx = p + 1, cpu = (ctx + S - 1) / S;
    u.a = u.j * cpu;
    u.b = min(ctx, u.a + cpu);
    u.ncached = max(0, min(u.b, p) - u.a);
    u.has_new = u.a <= p && p < u.b;
    return u;
}

// P2: attention unit (kv head g, split j); the cached rows [a, min(b, p))
// arrive through the ring, the new token's k, v come from the projection
// (read after the group's projection counter is complete). scr: G*HD q,
// HD k, HD v, then [warps][G][HD + 4] warp partials. Publishes acc[HD],
// max, sum per query head to partb.
template <int HD, int G>
__device__ __forceinline__ void attention_phase(const StepParams &P, int l, int unit, int seq, int p, const Ring &ring,
                                                uint32_t &n, float *scr, unsigned nq, const WaitCtx &w, int tid,
                                                unsigned long long *tr) {
    constexpr int E = HD / 32;
    constexpr int PS = HD + 2;   // a published partial: acc[HD], max, sum
    constexpr int PW = HD + 4;   // a warp partial in shared memory (16-byte rows)
    const int warp = tid >> 5, lane = tid & 31;
    const UnitRange u = unit_range(unit, P.S, p);
    const int nch = (u.ncached + P.CP - 1) / P.CP;
    float *qs = scr, *kn = qs + G * HD, *vn = kn + HD, *wp = vn + HD;
    float *kbase = P.kv + static_cast<size_t>(l) * P.layer_stride + static_cast<size_t>(seq) * P.seq_stride +
                   static_cast<size_t>(u.g) * P.head_stride;
    float *vbase = kbase + P.kvsel_stride;
    const bool role = warp < G || (u.has_new && warp < G + 2);

    // operands that do not depend on this layer's projection, then the wait
    float nw[E];
    float2 cs[E];
    if (role && warp <= G) {
        lane_load<HD>(at_layer(warp < G ? P.L0.q_norm : P.L0.k_norm, l, P.lstride), nw, lane);
        const float2 *rrow = P.rope + static_cast<size_t>(p) * (HD / 2);
#pragma unroll
        for (int e = 0; e < E; ++e) cs[e] = __ldg(rrow + (lane & 15) * E + e);
    }
    if (tid == 0) wait_count(ctr_at(P, 24 + u.g), gate(static_cast<unsigned>(l + 1) * nq, nq), w);
    csync();
    if (tr) tr[1] = globaltimer_ns();
    if (role) {
        const int row = warp < G ? (u.g * G + warp) * HD
                                 : (warp == G ? (P.nh + u.g) * HD : (P.nh + P.nkv + u.g) * HD);
        float v[E];
        ll_read<E>(P.qkvb, row + lane * E, step_tag(w.epoch, l, 1), v, w);
        if (warp <= G) norm_rope<HD>(v, nw, cs, P.eps, lane);
        if (warp < G) {
            lane_store<HD>(qs + warp * HD, v, lane);
        } else if (warp == G) {
            lane_store<HD>(kn, v, lane);
            lane_store<HD>(kbase + static_cast<size_t>(p) * HD, v, lane);
        } else {
            lane_store<HD>(vn, v, lane);
            lane_store<HD>(vbase + static_cast<size_t>(p) * HD, v, lane);
        }
    }
    csync();
    if (tr) tr[2] = globaltimer_ns();

    float qv[G][E], acc[G][E], m[G], ls[G];
#pragma unroll
    for (int t = 0; t < G; ++t) {
        lane_load<HD>(qs + t * HD, qv[t], lane);
        m[t] = -INFINITY;
        ls[t] = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[t][e] = 0.0f;
    }
    auto consume = [&](const float *krow, const float *vrow) {
        float k[E], vv[E];
        lane_load<HD>(krow, k, lane);
        lane_load<HD>(vrow, vv, lane);
        float sc[G];
#pragma unroll
        for (int t = 0; t < G; ++t) {
            float d = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) d = fmaf(qv[t][e], k[e], d);
            sc[t] = d;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int t = 0; t < G; ++t) sc[t] += __shfl_xor_sync(0xffffffffu, sc[t], o);
#pragma unroll
        for (int t = 0; t < G; ++t) {
            const float s = sc[t] * P.scale;
            const float mn = fmaxf(m[t], s);
            const float corr = expf(m[t] - mn);
            const float pr = expf(s - mn);
            ls[t] = fmaf(ls[t], corr, pr);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[t][e] = fmaf(pr, vv[e], acc[t][e] * corr);
            m[t] = mn;
        }
    };
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        const float *slot = reinterpret_cast<const float *>(ring_wait(ring, n, w));
        const int np = min(P.CP, u.ncached - c * P.CP);
#pragma unroll 1
        for (int i = warp; i < np; i += kCW) consume(slot + i * HD, slot + (P.CP + i) * HD);
        ring_release(ring, n, lane);
        ++n;
    }
    if (u.has_new && warp == kCW - 1) consume(kn, vn);
    if (tr) tr[3] = globaltimer_ns();

    // merge the warps' partials, publish (acc, max, sum) per query head
#pragma unroll
    for (int t = 0; t < G; ++t) {
        float *dst = wp + (warp * G + t) * PW;
        lane_store<HD>(dst, acc[t], lane);
        if (lane == 0) {
            dst[HD] = m[t];
            dst[HD + 1] = ls[t];
        }
    }
    csync();
    if (tid == 0) red_relaxed_add(ctr_at(P, 24 + P.nkv + u.g), 1u);
    {
        // one (head, dim) output per consumer thread: max and weights over
        // the 16 warps' partials, independent loads and exps in flight
        const unsigned tag = step_tag(w.epoch, l, 2);
        const int base = (u.g * P.S + u.j) * G;
        for (int o = tid; o < G * HD; o += kCT) {
            const int t = o / HD, d = o - (o / HD) * HD;
            float mw[kCW];
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kCW; ++ww) {
                mw[ww] = wp[(ww * G + t) * PW + HD];
                M = fmaxf(M, mw[ww]);
            }
            float L = 0.0f, A = 0.0f;
            if (M != -INFINITY) {
#pragma unroll
                for (int ww = 0; ww < kCW; ++ww) {
                    const float f = expf(mw[ww] - M);
                    L = fmaf(wp[(ww * G + t) * PW + HD + 1], f, L);
                    A = fmaf(wp[(ww * G + t) * PW + d], f, A);
                }
            }
            ll_st(P.partb, (base + t) * PS + d, A, tag);
            if (d == 0) {
                ll_st(P.partb, (base + t) * PS + HD, M, tag);
                ll_st(P.partb, (base + t) * PS + HD + 1, L, tag);
            }
        }
    }
    // the scratch is the next phase's plane buffer
    csync();
}

// P3: outputs [j GD / S, (j + 1) GD / S) of kv head g's G*HD attention
// outputs from the S unit partials (flash-decoding combine); one output per
// warp at a time, split jj of the partials in lane jj % 32 (S <= 96).
template <int HD, int G>
__device__ __forceinline__ void combine_phase(const StepParams &P, int l, int unit, const WaitCtx &w, int tid) {
    constexpr int PS = HD + 2;
    constexpr int GD = G * HD;
    const int warp = tid >> 5, lane = tid & 31;
    const int S = P.S, g = unit / S, j = unit - (unit / S) * S;
    const int e0 = j * GD / S, e1 = (j + 1) * GD / S;
    const unsigned tag2 = step_tag(w.epoch, l, 2);
    if (tid == 0) wait_count(ctr_at(P, 24 + P.nkv + g), gate(static_cast<unsigned>((l + 1) * S), S), w);
    csync();
    bool wrote = false;
#pragma unroll 1
    for (int e = e0 + warp; e < e1; e += kCW) {
        const int t = e / HD, d = e - (e / HD) * HD;
        float mv[3], lv[3], av[3];
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int jj = lane + 32 * k;
            mv[k] = -INFINITY;
            lv[k] = 0.0f;
            av[k] = 0.0f;
            if (jj < S) {
                const int src = ((g * S + jj) * G + t) * PS;
                const unsigned long long *pw = reinterpret_cast<const unsigned long long *>(P.partb);
                unsigned long long um, ul, ua;
                ll_ld2(pw + src + HD, um, ul);
                ua = ll_ld1(pw + src + d);
                if (ll_ok(um, tag2) && ll_ok(ul, tag2) && ll_ok(ua, tag2)) {
                    mv[k] = ll_val(um);
                    lv[k] = ll_val(ul);
                    av[k] = ll_val(ua);
                } else {
                    float ml[2];
                    ll_read<2>(P.partb, src + HD, tag2, ml, w);
                    mv[k] = ml[0];
                    lv[k] = ml[1];
                    av[k] = ll_read1(P.partb, src + d, tag2, w);
                }
                M = fmaxf(M, mv[k]);
            }
        }
        M = warp_max(M);
        float num = 0.0f, den = 0.0f;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            if (mv[k] != -INFINITY) {
                const float f = expf(mv[k] - M);
                num = fmaf(f, av[k], num);
                den = fmaf(f, lv[k], den);
            }
        }
        num = warp_sum(num);
        den = warp_sum(den);
        if (lane == 0) {
            ll_st(P.ob, g * GD + e, den > 0.0f ? num / den : 0.0f, step_tag(w.epoch, l, 3));
            wrote = true;
        }
    }
    (void)wrote;
    arrive(ctr_at(P, 8 + blockIdx.x % kSub), e1 > e0, tid);
}

// ---------------------------------------------------------------- kernel

// Rows [r0, r1) of the fused [q; k; v] matrix hold rows of kv head g's group.
__device__ __forceinline__ bool rows_touch_group(int r0, int r1, int g, int G, int HD, int nh, int nkv) {
    auto hit = [&](int a, int b) { return r0 < b && a < r1; };
    return hit(g * G * HD, (g + 1) * G * HD) || hit((nh + g) * HD, (nh + g + 1) * HD) ||
           hit((nh + nkv + g) * HD, (nh + nkv + g + 1) * HD);
}

template <int LC, int HD, int G>
__global__ void __launch_bounds__(kStepThreads, 1) k_step(const __grid_constant__ StepParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, NCTA = P.NCTA;
    const int nph = kStepPhases * P.L + 2;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + P.NS;
    // trace: per traced CTA (the first and the last), 4 words per phase
    // (inputs staged, first ring chunk in, dot tasks done, outputs
    // published), 32 producer issue times, 32 consumer times of the first 32
    // chunks; then 16 words per CTA for layer 1
    const bool traced = P.trace && (c == 0 || c == NCTA - 1);
    unsigned long long *tbase = traced ? P.trace + static_cast<size_t>(c == 0 ? 0 : 1) * (nph * 4 + 64) : nullptr;
    const Ring ring{full, empty, smem + P.o_ring, P.NS, P.SB, traced ? tbase + nph * 4 + 32 : nullptr};
    float *ssw = reinterpret_cast<float *>(smem + P.o_misc);                        // [16]
    unsigned long long *best = reinterpret_cast<unsigned long long *>(smem + P.o_misc + 64);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + P.o_misc + 80);
    float *xown = reinterpret_cast<float *>(smem + P.o_xown);
    uint8_t *planes = smem + P.o_planes;
    float *scr = reinterpret_cast<float *>(smem + P.o_planes);
    float *scales = reinterpret_cast<float *>(smem + P.o_scales);
    float *red = reinterpret_cast<float *>(smem + P.o_red);

    const unsigned epoch = *P.epoch;
    const int tok = *P.tok, seq = P.seq_ids[0], p = P.pos[0];
    const WaitCtx wc{&P, epoch};
    const int unit = c < P.nkv * P.S ? c : -1;
    unsigned long long *trace = tid == 0 ? tbase : nullptr;
    auto rec = [&](int ph, int k) {
        if (trace) trace[ph * 4 + (k ? 3 : 0)] = clock64();
    };
    unsigned long long *ctr1 = (P.trace && tid == 0) ? P.trace + 2 * (nph * 4 + 64) + static_cast<size_t>(c) * 16
                                                      : nullptr;
    auto rec1 = [&](int l, int k) {
        if (ctr1 && l == 1) ctr1[k] = globaltimer_ns();
    };
    rec(0, 0);

    if (tid == 0) {
        for (int i = 0; i < P.NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCW);
        }
        fence_mbar_init();
        *best = 0ull;
        flags[0] = 0;
        flags[1] = 0;
    }
    // this CTA's slices of the five streamed matrices (layer 0; layer l adds
    // l * lstride), computed once
    Slice *sls = reinterpret_cast<Slice *>(smem + P.o_misc + 256);   // qkv, o, gu, down, lm_head
    float *rsc = reinterpret_cast<float *>(smem + P.o_misc + 96);    // norm scale of the staged vector
    if (tid < 5) {
        const QMat *mats[5] = {&P.L0.qkv, &P.L0.o, &P.L0.gu, &P.L0.down, &P.out};
        sls[tid] = make_slice(*mats[tid], c, NCTA, P.SB);
    }
    __syncthreads();
    const unsigned *nX = P.cnt_x, *nO = P.cnt_o, *nA = P.cnt_act;
    const unsigned nq = unit >= 0 ? P.cnt_qkv[unit / P.S] : 0u;

    if (warp == kCW) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t n = 0;
            auto emit = [&](const void *src, uint32_t bytes, const void *src2, uint32_t bytes2, uint32_t off2) {
                const uint32_t slot = n % P.NS;
                if (n >= static_cast<uint32_t>(P.NS)) (void)ring_bar_wait(&empty[slot], ((n / P.NS) - 1) & 1u, wc);
                if (tbase && n < 32) tbase[nph * 4 + n] = clock64();
                uint8_t *dst = smem + P.o_ring + static_cast<size_t>(slot) * P.SB;
                mbar_arrive_expect_tx(&full[slot], bytes + bytes2);
                bulk_g2s(dst, src, bytes, &full[slot], pol);
                if (bytes2) bulk_g2s(dst + off2, src2, bytes2, &full[slot], pol);
                ++n;
            };
            auto tiles = [&](const Slice &sl) {
                const int nt = sl.ng * sl.ntk;
                for (int t0 = 0; t0 < nt; t0 += sl.tpc) {
                    const int cnt_t = min(sl.tpc, nt - t0);
                    emit(sl.src + static_cast<size_t>(t0) * sl.tb, static_cast<uint32_t>(cnt_t) * sl.tb, nullptr, 0, 0);
                }
            };
            for (int l = 0; l < P.L; ++l) {
                if (l == 1 && P.trace) P.trace[2 * (nph * 4 + 64) + static_cast<size_t>(c) * 16 + 13] = globaltimer_ns();
                tiles(slice_at(sls[0], l, P.lstride));
                if (unit >= 0) {
                    const UnitRange u = unit_range(unit, P.S, p);
                    const float *kb = P.kv + static_cast<size_t>(l) * P.layer_stride +
                                      static_cast<size_t>(seq) * P.seq_stride + static_cast<size_t>(u.g) * P.head_stride;
                    const float *vb = kb + P.kvsel_stride;
                    for (int i0 = 0; i0 < u.ncached; i0 += P.CP) {
                        const int cnt_p = min(P.CP, u.ncached - i0);
                        const uint32_t bytes = static_cast<uint32_t>(cnt_p * HD * 4);
                        emit(kb + static_cast<size_t>(u.a + i0) * HD, bytes, vb + static_cast<size_t>(u.a + i0) * HD,
                             bytes, static_cast<uint32_t>(P.CP * HD * 4));
                    }
                }
                tiles(slice_at(sls[1], l, P.lstride));
                tiles(slice_at(sls[2], l, P.lstride));
                tiles(slice_at(sls[3], l, P.lstride));
            }
            tiles(sls[4]);
            // drain: every copy has landed before the CTA can exit
            const uint32_t first = n > static_cast<uint32_t>(P.NS) ? n - P.NS : 0;
            for (uint32_t k = first; k < n; ++k) (void)ring_bar_wait(&full[k % P.NS], (k / P.NS) & 1u, wc);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    uint32_t n = 0;
    {
        // this CTA's rows of the residual stream: the embedding row
        const Slice so = sls[1];
        for (int t = tid; t < so.ng * 8; t += kCT) {
            const int r = so.row0 + t;
            xown[t] = __half2float(*qm_scale(P.embd, tok, r)) * static_cast<float>(*qm_codes(P.embd, tok, r));
        }
    }
    rec(0, 1);
    const int xsub = c % kSub;
    for (int l = 0; l < P.L; ++l) {
        const int ph = kStepPhases * l;

        // ---- P1: [q; k; v] = W_qkv RMSNorm(x)
        {
            const Slice sl = slice_at(sls[0], l, P.lstride);
            if (l > 0 && sl.ng > 0 && tid < kSub) wait_count(ctr_at(P, tid), gate(2u * l * nX[tid], nX[tid]), wc);
            csync();
            if (sl.ng > 0)
                stage_planes<LC>(l == 0 ? nullptr : P.xb, step_tag(epoch, l - 1, 6), wc, &P.embd, tok, P.H, at_layer(P.L0.attn_norm, l, P.lstride),
                                 planes, scales, ssw, tid);
            csync();
            rec(ph + 1, 0);
            if (warp == kCW - 1 && sl.ng > 0) {
                const float r = norm_scale(ssw, P.H, P.eps);
                if (lane == 0) *rsc = r;
            }
            rec1(l, 0);
            gemv_tasks<LC>(sl, ring, n, planes, scales, red, wc, warp, lane, trace ? trace + (ph + 1) * 4 : nullptr);
            csync();
            const int r0 = sl.row0, r1 = min(sl.row0 + 8 * sl.ng, P.qkv_w);
            if (tid == 0 && sl.ng > 0)
                for (int g = 0; g < P.nkv; ++g)
                    if (rows_touch_group(r0, r1, g, G, HD, P.nh, P.nkv)) red_relaxed_add(ctr_at(P, 24 + g), 1u);
            if (sl.ng > 0) {
                const float r = *rsc;
                bool wrote = false;
                for (int t = tid; t < r1 - r0; t += kCT) {
                    ll_st(P.qkvb, r0 + t, row_sum<LC>(sl, red, t) * r, step_tag(epoch, l, 1));
                    wrote = true;
                }
                (void)wrote;
            }
            csync();
            rec(ph + 1, 1);
            rec1(l, 1);
        }
        // ---- P2: attention partials; P3: their combine
        if (unit >= 0) {
            attention_phase<HD, G>(P, l, unit, seq, p, ring, n, scr, nq, wc, tid, (ctr1 && l == 1) ? ctr1 + 1 : nullptr);
            rec(ph + 2, 1);
            rec1(l, 5);
            combine_phase<HD, G>(P, l, unit, wc, tid);
            rec(ph + 3, 1);
            rec1(l, 6);
        }
        // ---- P4: x += W_o o
        {
            const Slice sl = slice_at(sls[1], l, P.lstride);
            if (sl.ng > 0 && tid < kSub) wait_count(ctr_at(P, 8 + tid), gate(static_cast<unsigned>(l + 1) * nO[tid], nO[tid]), wc);
            csync();
            if (sl.ng > 0)
                stage_planes<LC>(P.ob, step_tag(epoch, l, 3), wc, nullptr, 0, P.nh * HD, nullptr, planes, scales, ssw, tid);
            csync();
            rec(ph + 4, 0);
            rec1(l, 7);
            gemv_tasks<LC>(sl, ring, n, planes, scales, red, wc, warp, lane, trace ? trace + (ph + 4) * 4 : nullptr);
            csync();
            if (tid == 0 && sl.ng > 0) red_relaxed_add(ctr_at(P, xsub), 1u);
            bool wrote = false;
            for (int t = tid; t < sl.ng * 8; t += kCT) {
                const float y = xown[t] + row_sum<LC>(sl, red, t);
                xown[t] = y;
                ll_st(P.xb, sl.row0 + t, y, step_tag(epoch, l, 4));
                wrote = true;
            }
            (void)wrote;
            csync();
            rec(ph + 4, 1);
            rec1(l, 8);
        }
        // ---- P5: act = silu(W_gate h) * (W_up h), h = RMSNorm(x)
        {
            const Slice sl = slice_at(sls[2], l, P.lstride);
            if (sl.ng > 0 && tid < kSub) wait_count(ctr_at(P, tid), gate((2u * l + 1u) * nX[tid], nX[tid]), wc);
            csync();
            if (sl.ng > 0)
                stage_planes<LC>(P.xb, step_tag(epoch, l, 4), wc, nullptr, 0, P.H, at_layer(P.L0.ffn_norm, l, P.lstride), planes, scales, ssw, tid);
            csync();
            rec(ph + 5, 0);
            if (warp == kCW - 1 && sl.ng > 0) {
                const float r = norm_scale(ssw, P.H, P.eps);
                if (lane == 0) *rsc = r;
            }
            rec1(l, 9);
            gemv_tasks<LC>(sl, ring, n, planes, scales, red, wc, warp, lane, trace ? trace + (ph + 5) * 4 : nullptr);
            csync();
            if (tid == 0 && sl.ng > 0) red_relaxed_add(ctr_at(P, 16 + xsub), 1u);
            if (sl.ng > 0) {
                const float r = *rsc;
                for (int t = 2 * tid; t < sl.ng * 8; t += 2 * kCT) {
                    const int row = sl.row0 + t;
                    if (row < 2 * P.I) {
                        const float gt = row_sum<LC>(sl, red, t) * r;
                        const float up = row_sum<LC>(sl, red, t + 1) * r;
                        ll_st(P.actb, row / 2, __fdividef(gt, 1.0f + __expf(-gt)) * up, step_tag(epoch, l, 5));
                    }
                }
            }
            csync();
            rec(ph + 5, 1);
            rec1(l, 10);
        }
        // ---- P6: x += W_down act
        {
            const Slice sl = slice_at(sls[3], l, P.lstride);
            if (sl.ng > 0 && tid < kSub) wait_count(ctr_at(P, 16 + tid), gate(static_cast<unsigned>(l + 1) * nA[tid], nA[tid]), wc);
            csync();
            if (sl.ng > 0)
                stage_planes<LC>(P.actb, step_tag(epoch, l, 5), wc, nullptr, 0, P.I, nullptr, planes, scales, ssw, tid);
            csync();
            rec(ph + 6, 0);
            rec1(l, 11);
            gemv_tasks<LC>(sl, ring, n, planes, scales, red, wc, warp, lane, trace ? trace + (ph + 6) * 4 : nullptr);
            csync();
            if (tid == 0 && sl.ng > 0) red_relaxed_add(ctr_at(P, xsub), 1u);
            bool wrote = false;
            for (int t = tid; t < sl.ng * 8; t += kCT) {
                const float y = xown[t] + row_sum<LC>(sl, red, t);
                xown[t] = y;
                ll_st(P.xb, sl.row0 + t, y, step_tag(epoch, l, 6));
                wrote = true;
            }
            (void)wrote;
            csync();
            rec(ph + 6, 1);
            rec1(l, 12);
        }
    }

    // ---- final RMSNorm, lm_head, argmax (lowest index on ties)
    {
        const int phl = kStepPhases * P.L + 1;
        const Slice sl = sls[4];
        if (sl.ng > 0 && tid < kSub) wait_count(ctr_at(P, tid), gate(2u * P.L * nX[tid], nX[tid]), wc);
        csync();
        if (sl.ng > 0)
            stage_planes<LC>(P.xb, step_tag(epoch, P.L - 1, 6), wc, nullptr, 0, P.H, P.out_norm, planes, scales, ssw,
                             tid);
        csync();
        rec(phl, 0);
        if (warp == kCW - 1 && sl.ng > 0) {
            const float r = norm_scale(ssw, P.H, P.eps);
            if (lane == 0) *rsc = r;
        }
        gemv_tasks<LC>(sl, ring, n, planes, scales, red, wc, warp, lane, trace ? trace + phl * 4 : nullptr);
        csync();
        float *logits = P.io->logits;
        unsigned long long key = 0ull;
        if (sl.ng > 0) {
            const float r = *rsc;
            for (int t = tid; t < sl.ng * 8; t += kCT) {
                const int row = sl.row0 + t;
                if (row < P.V) {
                    const float y = row_sum<LC>(sl, red, t) * r;
                    if (logits) logits[row] = y;
                    const unsigned long long k = argmax_pack(y, row);
                    key = k > key ? k : key;
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
            key = other > key ? other : key;
        }
        if (lane == 0 && key) atomicMax(best, key);
        csync();
        if (tid == 0) {
            atomicMax(P.argmax_key, *best);
            __threadfence();
            const unsigned prev = atomicAdd(P.done_counter, 1u);
            if (prev == static_cast<unsigned>(NCTA - 1)) {
                // last CTA: every other CTA is done with this step
                __threadfence();
                const unsigned long long k = atomicAdd(P.argmax_key, 0ull);
                const int idx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
                const float v = float_from_order_key(static_cast<uint32_t>(k >> 32));
                if (isnan(v)) record_status(P.status, QW3_ERR_NONFINITE);
                const int step = *P.step_ctr;
                if (P.io->argmax) P.io->argmax[0] = idx;
                if (P.io->hist) P.io->hist[step] = idx;
                *P.tok = idx;
                *P.pos = p + 1;
                *P.step_ctr = step + 1;
                *P.argmax_key = 0ull;
                *P.done_counter = 0u;
                for (int i = 0; i < 24 + 2 * P.nkv; ++i) *ctr_at(P, i) = 0u;
                *P.epoch = epoch + 1;
            }
        }
        rec(phl, 1);
    }
}

}  // namespace

}  // namespace qw3

// ------------------------------------------------------------------ host

namespace qw3 {

namespace {

template <int LC, int HD, int G>
constexpr bool kStepInst = (LC == 16 && HD == 128 && (G == 2 || G == 4)) || (LC == 8 && HD == 64 && G == 2) ||
                           (LC == 8 && HD == 128 && G == 2);

// The tile width the model's repack gives a row of `cols` columns.
int model_tile_width(int cols) {
    if (cols <= 3072) return cols;
    for (int kt = 2048; kt >= 256; kt -= 256)
        if (cols % kt == 0) return kt;
    return cols;
}

int step_lc(const qw3_config &c) {
    const int cols[3] = {c.hidden, c.n_heads * c.head_dim, c.intermediate};
    bool k512 = true, k256 = true;
    for (int k : cols) {
        const int kt = model_tile_width(k);
        if (kt % 512) k512 = false;
        if (kt % 256) k256 = false;
    }
    return k512 ? 16 : (k256 ? 8 : 0);
}

template <int LC, int HD, int G>
const void *step_fn() {
    return reinterpret_cast<const void *>(k_step<LC, HD, G>);
}

const void *step_kernel(int LC, int HD, int G) {
    if (LC == 16 && HD == 128 && G == 2) return step_fn<16, 128, 2>();
    if (LC == 16 && HD == 128 && G == 4) return step_fn<16, 128, 4>();
    if (LC == 8 && HD == 64 && G == 2) return step_fn<8, 64, 2>();
    if (LC == 8 && HD == 128 && G == 2) return step_fn<8, 128, 2>();
    return nullptr;
}

uint32_t al128(size_t v) { return static_cast<uint32_t>((v + 127) / 128 * 128); }

}  // namespace

bool step_supported(const qw3_config &c) {
    if (c.n_kv_heads < 1 || c.n_kv_heads > 64 || c.n_heads % c.n_kv_heads) return false;
    const int LC = step_lc(c);
    if (!LC || !step_kernel(LC, c.head_dim, c.n_heads / c.n_kv_heads)) return false;
    const int kmax = std::max(c.hidden, std::max(c.intermediate, c.n_heads * c.head_dim));
    if (kmax > kMaxK) return false;
    return true;
}

bool step_plan(StepParams &P, const LayerDev &L0) {
    const int NCTA = num_sms();
    P.NCTA = NCTA;
    P.S = std::min(NCTA / P.nkv, 96);
    if (P.S < 1) return false;
    P.kmax = std::max(P.H, std::max(P.I, P.nh * P.hd));
    const QMat *mats[5] = {&L0.qkv, &L0.o, &L0.gu, &L0.down, &P.out};
    bool k512 = true, k256 = true;
    for (const QMat *W : mats) {
        if (W->ktile_major) return false;
        if (W->kt % 512) k512 = false;
        if (W->kt % 256) k256 = false;
    }
    P.LC = k512 ? 16 : (k256 ? 8 : 0);
    const void *fn = P.LC ? step_kernel(P.LC, P.hd, P.G) : nullptr;
    if (!fn) return false;
    // a ring slot holds the widest tile; red holds the most dot tasks of one
    // CTA in one phase (8 row partials each)
    size_t sb = 0;
    int tasks_max = 1;
    for (const QMat *W : mats) {
        sb = std::max(sb, qm_tile_bytes(W->kt));
        const int NG = (W->rows + 7) / 8;
        const int gmax = (NG + NCTA - 1) / NCTA;
        tasks_max = std::max(tasks_max, gmax * (W->cols / (32 * P.LC)));
    }
    // writers behind each arrival counter
    for (int sidx = 0; sidx < kSub; ++sidx) P.cnt_x[sidx] = P.cnt_o[sidx] = P.cnt_act[sidx] = 0;
    for (int g = 0; g < 64; ++g) P.cnt_qkv[g] = 0;
    const int GD = P.G * P.hd;
    for (int c2 = 0; c2 < NCTA; ++c2) {
        int g0, g1;
        group_range(P.H / 8, c2, NCTA, g0, g1);
        P.cnt_x[c2 % kSub] += g1 > g0;
        if (c2 < P.nkv * P.S) {
            const int j = c2 % P.S;
            P.cnt_o[c2 % kSub] += (j + 1) * GD / P.S > j * GD / P.S;
        }
        group_range((2 * P.I + 7) / 8, c2, NCTA, g0, g1);
        P.cnt_act[c2 % kSub] += g1 > g0;
        group_range((P.qkv_w + 7) / 8, c2, NCTA, g0, g1);
        if (g1 > g0)
            for (int g = 0; g < P.nkv; ++g) {
                const int r0 = 8 * g0, r1 = std::min(8 * g1, P.qkv_w);
                auto hit = [&](int a, int b) { return r0 < b && a < r1; };
                if (hit(g * GD, (g + 1) * GD) || hit((P.nh + g) * P.hd, (P.nh + g + 1) * P.hd) ||
                    hit((P.nh + P.nkv + g) * P.hd, (P.nh + P.nkv + g + 1) * P.hd))
                    ++P.cnt_qkv[g];
            }
    }
    P.SB = al128(sb);
    P.CP = std::min(64, static_cast<int>(P.SB / (8u * P.hd)));
    if (P.CP < 1) return false;
    const size_t planes = 3 * static_cast<size_t>(P.kmax) + 16 + static_cast<size_t>(P.kmax / 32) * 4;
    const size_t attn = (static_cast<size_t>(P.G) * P.hd + 2 * P.hd +
                         static_cast<size_t>(kCW) * P.G * (P.hd + 4)) * 4;
    P.o_misc = 512;   // ring barriers below (2 x up to 32 slots)
    P.o_xown = P.o_misc + 512;
    const int gown = (P.H / 8 + NCTA - 1) / NCTA;
    P.o_planes = P.o_xown + al128(static_cast<size_t>(gown) * 8 * 4);
    P.o_scales = P.o_planes + static_cast<uint32_t>((3 * static_cast<size_t>(P.kmax) + 15) / 16 * 16);
    P.o_red = P.o_planes + al128(std::max(planes, attn));
    P.o_ring = P.o_red + al128(static_cast<size_t>(tasks_max) * 8 * 4);
    const size_t budget = 227 * 1024;
    if (P.o_ring + 2 * static_cast<size_t>(P.SB) > budget) return false;
    P.NS = static_cast<int>(std::min<size_t>(32, (budget - P.o_ring) / P.SB));
    P.smem = P.o_ring + static_cast<uint32_t>(P.NS) * P.SB;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kStepThreads, P.smem) != cudaSuccess || nb < 1)
        return false;
    return true;
}

cudaError_t configure_step() {
    const void *fns[4] = {step_fn<16, 128, 2>(), step_fn<16, 128, 4>(), step_fn<8, 64, 2>(), step_fn<8, 128, 2>()};
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_step(const StepParams &P, cudaStream_t s) {
    const void *fn = step_kernel(P.LC, P.hd, P.G);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(P.NCTA);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = P.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<StepParams *>(&P)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace qw3
