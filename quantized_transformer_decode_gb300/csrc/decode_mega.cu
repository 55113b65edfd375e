// Persistent batch-1 decode: every layer of every greedy step in one kernel.
//
// What it computes is the decode step of "A transformer from scratch"
// (sections 12.3-12.6) with the Qwen3 deltas of minfer's "Qwen3 Support Plan
// (dense)" (section 2): for each step, embed the token, run L layers
// (RMSNorm, QKV, per-head Q/K RMSNorm, NeoX RoPE, KV append, causal GQA over
// the f32 cache, o_proj + residual, RMSNorm, gate/up, SwiGLU, down +
// residual), final RMSNorm, lm_head, argmax (lowest index on ties); the
// argmax is the next step's token.
//
// Why one kernel (GB300): at batch 1 a 0.6B-parameter layer moves ~22 MB,
// about 3 us of HBM time, so per-launch ramp-up and tail cost as much as the
// data. Here the weight and KV stream never stops: weights do not depend on
// activations and KV rows before the current position are already final, so
// a producer warp per CTA streams its slices of the coming layers through a
// shared-memory ring with 1-D bulk copies (TMA) while the consumer warps are
// still waiting on the dependency chain of the current one.
//
// Work split. Clusters of CS = 8 CTAs. Cluster g < NA (NA = n_kv_heads) owns
// KV head g: it computes the group's QKV rows (the G query heads, k and v;
// QKV rows are stored group by group), exchanges them through distributed
// shared memory, normalises and rotates, appends k and v to the cache,
// splits the positions of the causal attention over its CTAs, combines the
// partial softmax states through distributed shared memory, and multiplies
// by its head group's columns of W_o (split-K over head groups): a partial
// o_proj vector per group. All NC clusters then run the FFN: cluster c owns a
// range of intermediate channels (gate/up rows split over its CTAs, SwiGLU,
// exchange of the channel values, then a split-K slice of W_down). The
// lm_head rows are split over all CTAs.
//
// Synchronisation. Inside a cluster: mbarriers that every CTA arrives on
// remotely (two, alternating, so arrivals of consecutive rounds never mix).
// Across the grid: one monotonically increasing arrival counter in global
// memory, two rounds per layer and one per step; every CTA keeps its own
// copy of the residual stream x and adds the partial vectors in a fixed
// order, so all copies are bit-identical. Every wait is bounded (1 s); a
// timeout records QW3_ERR_TIMEOUT and the kernel runs to its end without
// further waiting, draining its in-flight copies.
//
// Arithmetic: f32 throughout; Q8_0 codes are converted exactly (int8 -> f32
// by byte-permuting into the mantissa of 2^23) and accumulated with packed
// fma.rn.f32x2, d applied per 32-block.
#include <algorithm>
#include <cmath>

#include "qw3_internal.cuh"
#include "decode_mega.cuh"

namespace qw3 {

namespace {

constexpr int kMegaConsumers = 256;   // 8 consumer warps
constexpr int kMegaThreads = 288;     // + 1 producer warp

__device__ __forceinline__ void mcons_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

// Relaxed remote arrive: the caller publishes its writes with one
// fence.acq_rel.cluster before a series of these (a release per arrive would
// pay a cluster-scope fence each time).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Activation vectors enter the GEMVs as three int8 digit planes per 32-value
// block: x = s * (h + m / 254 + l / 254^2), s = max|x| / 127, |h|, |m|, |l|
// <= 127, which represents x to within s / (2 * 254^2) ~ 6e-8 of the block
// maximum (about f32 rounding). Plane q of values [16c, 16c + 16) is the
// uint4 at planes[3c + q]; the block scale s is at scales[k / 32]. A dot of
// 16 codes with the planes is then 12 exact int8 dot-products (dp4a).
struct Planes {
    const uint4 *pl;
    const float *sc;
};

// Split the 32 values a warp holds (lane i: value v of block element i) into
// digit planes; writes the block's 3 x 32 plane bytes and its scale.
__device__ __forceinline__ void to_planes(float v, int block, uint8_t *planes, float *scales, int lane) {
    const float amax = warp_max(fabsf(v));
    const float sb = amax / 127.0f;
    int h = 0, m = 0, l = 0;
    if (sb > 0.0f) digit_planes(v, 1.0f / sb, h, m, l);
    uint8_t *dst = planes + static_cast<size_t>(block * 2 + (lane >> 4)) * 48 + (lane & 15);
    dst[0] = static_cast<uint8_t>(static_cast<int8_t>(h));
    dst[16] = static_cast<uint8_t>(static_cast<int8_t>(m));
    dst[32] = static_cast<uint8_t>(static_cast<int8_t>(l));
    if (lane == 0) scales[block] = sb;
}

// ------------------------------------------------------------ item plan

enum MegaItem : int { MI_QKV = 0, MI_K, MI_V, MI_O, MI_GU, MI_DOWN, MI_LM };

// A contiguous run of equal units (tiles or KV rows) in global memory.
struct Run {
    const uint8_t *src;
    uint32_t unit;    // bytes per unit
    uint32_t n;       // units
    uint32_t upc;     // units per chunk (ring slot)
};

struct Role {
    int c, j, cta;    // cluster, rank in cluster, CTA index
    bool att;         // owns a KV head group (c < NA)
    int a0, kt_c;     // FFN: first channel of the cluster, channels of the cluster
    int apc;          // FFN channels of this CTA
};

__device__ __forceinline__ uint32_t tile_bytes(int kt) { return static_cast<uint32_t>(kt) * 17u / 2u; }

__device__ __forceinline__ int ffn_a(const MegaParams &P, int c) { return (c * P.act_units / P.NC) * 32; }

template <typename T>
__device__ __forceinline__ const T *at_layer(const T *base, int l, size_t stride) {
    return reinterpret_cast<const T *>(reinterpret_cast<const uint8_t *>(base) + static_cast<size_t>(l) * stride);
}

__device__ Run make_run(const MegaParams &P, const Role &R, int kind, int l, int p) {
    Run r{};
    switch (kind) {
        case MI_QKV: {
            const int row0 = R.c * P.RG + R.j * P.RPC;
            r.unit = tile_bytes(P.H);
            r.src = at_layer(P.qkv0, l, P.mstride) + static_cast<size_t>(row0 / 8) * r.unit;
            r.n = P.RPC / 8;
            break;
        }
        case MI_K:
        case MI_V: {
            const int a = static_cast<int>((static_cast<long long>(R.j) * p) / P.CS);
            const int b = static_cast<int>((static_cast<long long>(R.j + 1) * p) / P.CS);
            const float *base = P.kv + static_cast<size_t>(l) * P.layer_stride + static_cast<size_t>(P.seq) * P.seq_stride +
                                (kind == MI_V ? P.kvsel_stride : 0) + static_cast<size_t>(R.c) * P.head_stride +
                                static_cast<size_t>(a) * P.hd;
            r.src = reinterpret_cast<const uint8_t *>(base);
            r.unit = static_cast<uint32_t>(P.hd) * 4u;
            r.n = static_cast<uint32_t>(b - a);
            break;
        }
        case MI_O: {
            r.unit = tile_bytes(P.G * P.hd);
            r.src = at_layer(P.o0, l, P.mstride) + (static_cast<size_t>(R.c) * P.o_groups + R.j * (P.ORPC / 8)) * r.unit;
            r.n = P.ORPC / 8;
            break;
        }
        case MI_GU: {
            const int row0 = 2 * (R.a0 + R.j * R.apc);
            r.unit = tile_bytes(P.H);
            r.src = at_layer(P.gu0, l, P.wstride) + static_cast<size_t>(row0 / 8) * r.unit;
            r.n = 2 * R.apc / 8;
            break;
        }
        case MI_DOWN: {
            r.unit = tile_bytes(R.kt_c);
            const size_t cl_base = static_cast<size_t>(P.o_groups) * 17u * static_cast<size_t>(R.a0) / 2u;
            r.src = at_layer(P.down0, l, P.mstride) + cl_base + static_cast<size_t>(R.j * (P.ORPC / 8)) * r.unit;
            r.n = P.ORPC / 8;
            break;
        }
        default: {  // MI_LM
            const int ng = (P.V + 7) / 8;
            const int g0 = static_cast<int>((static_cast<long long>(R.cta) * ng) / P.NCTA);
            const int g1 = static_cast<int>((static_cast<long long>(R.cta + 1) * ng) / P.NCTA);
            r.unit = tile_bytes(P.H);
            r.src = P.out.base + static_cast<size_t>(g0) * r.unit;
            r.n = static_cast<uint32_t>(g1 - g0);
            break;
        }
    }
    r.upc = P.SB / r.unit;
    if (r.upc < 1) r.upc = 1;
    return r;
}

__device__ __forceinline__ uint32_t run_chunks(const Run &r) { return (r.n + r.upc - 1) / r.upc; }

// ---------------------------------------------------------------- state

struct Smem {
    uint64_t *full, *empty, *clbar;   // clbar[2]
    float *x, *wbuf, *qkvpub, *qkv, *scores, *apub, *vred, *guout, *actpub, *red;
    uint8_t *xpl, *opl, *apl;   // digit planes of the GEMV inputs (normed x, attention output, channels)
    float *xsc, *osc, *asc;     // their block scales
    unsigned long long *keys;
    volatile int *err;
    int *tok;
    uint8_t *ring;
};

__device__ Smem carve(const MegaParams &P, uint8_t *s) {
    Smem m;
    m.full = reinterpret_cast<uint64_t *>(s + P.o_bar);
    m.empty = m.full + P.NS;
    m.clbar = m.empty + P.NS;
    m.x = reinterpret_cast<float *>(s + P.o_x);
    m.xpl = s + P.o_xn;
    m.xsc = reinterpret_cast<float *>(s + P.o_xn + static_cast<size_t>(P.H) * 3);
    m.wbuf = reinterpret_cast<float *>(s + P.o_wbuf);
    m.qkvpub = reinterpret_cast<float *>(s + P.o_qkvpub);
    m.qkv = reinterpret_cast<float *>(s + P.o_qkv);
    m.scores = reinterpret_cast<float *>(s + P.o_scores);
    m.apub = reinterpret_cast<float *>(s + P.o_apub);
    m.vred = reinterpret_cast<float *>(s + P.o_vred);
    m.opl = s + P.o_oall;
    m.osc = reinterpret_cast<float *>(s + P.o_oall + static_cast<size_t>(P.G) * P.hd * 3);
    m.guout = reinterpret_cast<float *>(s + P.o_guout);
    m.actpub = reinterpret_cast<float *>(s + P.o_actpub);
    m.apl = s + P.o_act;
    m.asc = reinterpret_cast<float *>(s + P.o_act + static_cast<size_t>(P.o_act_cap) * 3);
    m.red = reinterpret_cast<float *>(s + P.o_red);
    m.keys = reinterpret_cast<unsigned long long *>(s + P.o_red + 256);
    m.err = reinterpret_cast<volatile int *>(s + P.o_red + 512);
    m.tok = reinterpret_cast<int *>(s + P.o_red + 516);
    m.ring = s + P.o_ring;
    return m;
}

// Bounded wait on an mbarrier phase (CTA scope); false in error mode.
__device__ bool wait_full(const Smem &S, uint64_t *bar, uint32_t parity, int32_t *status) {
    if (*S.err) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*S.err) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *S.err = 1;
            record_status(status, QW3_ERR_TIMEOUT);
            return false;
        }
    }
}

// Producer-side bounded wait for a free ring slot. It backs off between
// polls: the producer shares a scheduler with two consumer warps, and a
// tight poll loop would take their issue slots for the whole step.
__device__ bool wait_free_slot(const Smem &S, uint64_t *bar, uint32_t parity, int32_t *status) {
    if (*S.err) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(128);
        if (mbar_try_wait(bar, parity)) return true;
        if (*S.err) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *S.err = 1;
            record_status(status, QW3_ERR_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------ consumers

struct Cons {
    const MegaParams &P;
    const Smem &S;
    const Role &R;
    int tid, warp, lane;
    uint32_t q;        // ring chunk counter
    uint32_t clround;  // cluster sync rounds
    uint32_t gsync;    // global sync rounds passed
    unsigned long long *trec;   // this CTA's timeline records (traced CTAs only)
    bool last_step;
    unsigned long long w_full, w_grid, w_cl;   // wait totals (thread 0, traced runs)

    __device__ void mark(int rec, int word) {
        if (trec && last_step && tid == 0) trec[rec * 8 + word] = globaltimer_ns();
    }

    __device__ uint8_t *stage_wait() {
        const int s = static_cast<int>(q % static_cast<uint32_t>(P.NS));
        const bool timed = P.trace && tid == 0;
        const uint64_t t0 = timed ? globaltimer_ns() : 0;
        wait_full(S, S.full + s, (q / static_cast<uint32_t>(P.NS)) & 1u, P.status);
        if (timed) w_full += globaltimer_ns() - t0;
        return S.ring + static_cast<size_t>(s) * P.SB;
    }
    __device__ void stage_release() {
        const int s = static_cast<int>(q % static_cast<uint32_t>(P.NS));
        __syncwarp();
        if (lane == 0) mbar_arrive(S.empty + s);
        ++q;
    }

    // Every CTA of the cluster has published: arrive on every peer's round
    // barrier, then wait for the CS arrivals on ours.
    __device__ void cluster_sync() {
        mcons_sync();
        uint64_t *bar = S.clbar + (clround & 1u);
        if (tid == 0) {
            asm volatile("fence.acq_rel.cluster;" ::: "memory");   // publishes the CTA's writes (ordered by the bar.sync)
            for (int r = 0; r < P.CS; ++r) mbar_arrive_remote_relaxed(dsmem_map(bar, static_cast<uint32_t>(r)));
        }
        const uint32_t parity = (clround >> 1) & 1u;
        const uint64_t tw0 = (P.trace && tid == 0) ? globaltimer_ns() : 0;
        if (!*S.err && !mbar_try_wait_cluster(bar, parity)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_cluster(bar, parity)) {
                if (*S.err) break;
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    *S.err = 1;
                    record_status(P.status, QW3_ERR_TIMEOUT);
                    break;
                }
            }
        }
        if (P.trace && tid == 0) w_cl += globaltimer_ns() - tw0;
        ++clround;
        mcons_sync();
    }

    __device__ void grid_arrive() {
        mcons_sync();
        if (tid == 0) {
            __threadfence();
            atomicAdd(P.gctr, 1u);
        }
    }

    __device__ void grid_wait() {
        const unsigned target = (gsync + 1u) * static_cast<unsigned>(P.NCTA);
        const uint64_t tw0 = (P.trace && tid == 0) ? globaltimer_ns() : 0;
        if (tid == 0 && !*S.err && ld_acquire_gpu(P.gctr) < target) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(P.gctr) < target) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    *S.err = 1;
                    record_status(P.status, QW3_ERR_TIMEOUT);
                    break;
                }
            }
        }
        if (P.trace && tid == 0) w_grid += globaltimer_ns() - tw0;
        ++gsync;
        mcons_sync();
    }

    // x += sum over n partial vectors (fixed order), read from L2: the loads
    // of up to four elements per thread are issued before their stores.
    __device__ void add_partials(const float *part, int n) {
        for (int i0 = tid; i0 < P.H; i0 += 4 * kMegaConsumers) {
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int g = 0; g < n; ++g) {
                const float *pg = part + static_cast<size_t>(g) * P.H;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = i0 + k * kMegaConsumers;
                    if (i < P.H) v[k] += __ldcg(pg + i);
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = i0 + k * kMegaConsumers;
                if (i < P.H) S.x[i] += v[k];
            }
        }
        mcons_sync();
    }

    // Norm weights for the next rmsnorm: cp.async into shared memory, issued
    // ahead of the wait before the norm.
    __device__ void prefetch_w(const float *w) {
        for (int i = tid * 4; i < P.H; i += 4 * kMegaConsumers)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(S.wbuf + i)), "l"(w + i)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    __device__ float block_sum(float v) {
        v = warp_sum(v);
        if (lane == 0) S.red[warp] = v;
        mcons_sync();
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) t += S.red[w];
        mcons_sync();
        return t;
    }

    // xn = x / sqrt(mean(x^2) + eps) * w (course 12.3.2), w from prefetch_w,
    // written as digit planes: warp w handles blocks w, w + 8, ...
    __device__ void rmsnorm() {
        float ss = 0.0f;
        for (int i = tid; i < P.H; i += kMegaConsumers) ss = fmaf(S.x[i], S.x[i], ss);
        asm volatile("cp.async.wait_all;" ::: "memory");   // this thread's weights; block_sum syncs all
        const float r = 1.0f / sqrtf(block_sum(ss) / static_cast<float>(P.H) + P.eps);
        for (int i0 = tid; i0 < P.H; i0 += 4 * kMegaConsumers) to_planes4(i0, r);
        mcons_sync();
    }

    // Digit planes of up to four normalised values per thread (elements i0,
    // i0 + 256, ...): the four warp reductions run as independent chains.
    __device__ void to_planes4(int i0, float r) {
        float v[4], am[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kMegaConsumers;
            v[u] = (i < P.H) ? S.x[i] * r * S.wbuf[i] : 0.0f;
            am[u] = fabsf(v[u]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < 4; ++u) am[u] = fmaxf(am[u], __shfl_xor_sync(0xffffffffu, am[u], o));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kMegaConsumers;
            if (i < P.H) {
                const float sb = am[u] / 127.0f;
                int h = 0, m = 0, l = 0;
                if (sb > 0.0f) digit_planes(v[u], 1.0f / sb, h, m, l);
                uint8_t *dst = S.xpl + static_cast<size_t>((i >> 5) * 2 + (lane >> 4)) * 48 + (lane & 15);
                dst[0] = static_cast<uint8_t>(static_cast<int8_t>(h));
                dst[16] = static_cast<uint8_t>(static_cast<int8_t>(m));
                dst[32] = static_cast<uint8_t>(static_cast<int8_t>(l));
                if (lane == 0) S.xsc[i >> 5] = sb;
            }
        }
    }

    // One chunk of tiles (8 rows x kt): warp w takes row w of each tile, four
    // tiles (eight on the half-warp path, kt <= 256) per pass sharing each
    // load of the activation planes.
    template <typename Sink>
    __device__ void gemv_chunk(const uint8_t *stage, int ntiles, int kt, const Planes xin, int tile0, Sink sink) {
        const uint32_t tb = tile_bytes(kt);
        if (kt > 256) {
            for (int t0 = 0; t0 < ntiles; t0 += 4) {
                const int T = min(4, ntiles - t0);
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int k = lane * 16; k < kt; k += 512) {
                    uint4 Pq[3];
#pragma unroll
                    for (int q = 0; q < 3; ++q) Pq[q] = xin.pl[(k >> 4) * 3 + q];
                    const float sx = xin.sc[k >> 5];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        if (t < T) {
                            const uint8_t *tile = stage + static_cast<size_t>(t0 + t) * tb;
                            const uint4 w = *reinterpret_cast<const uint4 *>(tile + warp * kt + k);
                            const float d = __half2float(
                                reinterpret_cast<const __half *>(tile + 8 * kt)[warp * (kt >> 5) + (k >> 5)]);
                            acc[t] = fmaf(d * sx, pdot16(w, Pq), acc[t]);
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) acc[t] = warp_sum(acc[t]);
                if (lane == 0) {
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        if (t < T) sink(tile0 + t0 + t, warp, acc[t]);
                }
            }
        } else {
            const int half = lane >> 4, hl = lane & 15;
            for (int t0 = 0; t0 < ntiles; t0 += 8) {
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int k = hl * 16; k < kt; k += 256) {
                    uint4 Pq[3];
#pragma unroll
                    for (int q = 0; q < 3; ++q) Pq[q] = xin.pl[(k >> 4) * 3 + q];
                    const float sx = xin.sc[k >> 5];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = t0 + 2 * u + half;
                        if (t < ntiles) {
                            const uint8_t *tile = stage + static_cast<size_t>(t) * tb;
                            const uint4 w = *reinterpret_cast<const uint4 *>(tile + warp * kt + k);
                            const float d = __half2float(
                                reinterpret_cast<const __half *>(tile + 8 * kt)[warp * (kt >> 5) + (k >> 5)]);
                            acc[u] = fmaf(d * sx, pdot16(w, Pq), acc[u]);
                        }
                    }
                }
#pragma unroll
                for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], o);
                if (hl == 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int t = t0 + 2 * u + half;
                        if (t < ntiles) sink(tile0 + t, warp, acc[u]);
                    }
                }
            }
        }
    }

    template <typename Sink>
    __device__ void gemv_item(const Run &r, int kt, const Planes xin, Sink sink) {
        const uint32_t nch = run_chunks(r);
        for (uint32_t ch = 0; ch < nch; ++ch) {
            const uint8_t *st = stage_wait();
            const int u0 = static_cast<int>(ch * r.upc);
            const int nt = min(static_cast<int>(r.upc), static_cast<int>(r.n) - u0);
            gemv_chunk(st, nt, kt, xin, u0, sink);
            stage_release();
        }
    }
};

template <int HD, int G>
__device__ void phase_attention(Cons &C, int l, int p) {
    const MegaParams &P = C.P;
    const Smem &S = C.S;
    const Role &R = C.R;
    constexpr int E = HD / 32;

    // RoPE row of position p and the Q/K norm weights, ahead of their use
    float2 rp[E];
    {
        const float2 *rope_p = P.rope + static_cast<size_t>(p) * (HD / 2);
#pragma unroll
        for (int e = 0; e < E; ++e) rp[e] = __ldg(rope_p + (C.lane & 15) * E + e);
    }
    const float *qn = at_layer(P.q_norm0, l, P.wstride), *kn = at_layer(P.k_norm0, l, P.wstride);
    const float *nw = C.warp < G ? qn : kn;
    float nwr[E];
#pragma unroll
    for (int e = 0; e < E; ++e) nwr[e] = __ldg(nw + C.lane * E + e);

    // QKV rows of this CTA -> qkvpub
    C.mark(2 * l, 0);
    C.rmsnorm();
    {
        const Run r = make_run(P, R, MI_QKV, l, p);
        float *pub = S.qkvpub;
        C.gemv_item(r, P.H, Planes{reinterpret_cast<const uint4 *>(S.xpl), S.xsc},
                    [pub](int tile, int w, float v) { pub[tile * 8 + w] = v; });
    }
    C.mark(2 * l, 1);
    C.cluster_sync();
    // gather the group's q, k, v from the cluster: issue every remote load first
    {
        float g[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = C.tid + u * kMegaConsumers;
            g[u] = 0.0f;
            if (i < P.RG) {
                const int src = i / P.RPC, off = i - src * P.RPC;
                g[u] = dsmem_ld(dsmem_map(S.qkvpub + off, static_cast<uint32_t>(src)));
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = C.tid + u * kMegaConsumers;
            if (i < P.RG) S.qkv[i] = g[u];
        }
    }
    mcons_sync();
    // Q/K RMSNorm over head_dim then RoPE (warp h < G: query head h; warp G: k)
    if (C.warp <= G) {
        float *v = S.qkv + C.warp * HD;
        float a[E];
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            a[e] = v[C.lane * E + e];
            ss = fmaf(a[e], a[e], ss);
        }
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss / static_cast<float>(HD) + P.eps);
#pragma unroll
        for (int e = 0; e < E; ++e) a[e] = a[e] * r * nwr[e];
        const bool first = C.lane < 16;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, a[e], 16);
            a[e] = first ? (a[e] * rp[e].x - o * rp[e].y) : (o * rp[e].y + a[e] * rp[e].x);
        }
        __syncwarp();
#pragma unroll
        for (int e = 0; e < E; ++e) v[C.lane * E + e] = a[e];
    }
    mcons_sync();
    const float *knew = S.qkv + G * HD, *vnew = S.qkv + (G + 1) * HD;
    if (R.j == 0 && C.tid < 2 * HD) {
        float *dst = P.kv + static_cast<size_t>(l) * P.layer_stride + static_cast<size_t>(P.seq) * P.seq_stride +
                     static_cast<size_t>(R.c) * P.head_stride + static_cast<size_t>(p) * HD;
        if (C.tid < HD) dst[C.tid] = knew[C.tid];
        else dst[P.kvsel_stride + (C.tid - HD)] = vnew[C.tid - HD];
        fence_proxy_async_global();
    }
    C.mark(2 * l, 2);

    // scores over this CTA's cached positions (+ the new one on the last rank)
    const Run rk = make_run(P, R, MI_K, l, p);
    const int nk = static_cast<int>(rk.n);
    const bool has_new = (R.j == P.CS - 1);
    const int ntot = nk + (has_new ? 1 : 0);
    float qreg[G][E];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < E; ++e) qreg[h][e] = S.qkv[h * HD + C.lane * E + e];
    {
        const uint32_t nch = run_chunks(rk);
        for (uint32_t ch = 0; ch < nch; ++ch) {
            const uint8_t *st = C.stage_wait();
            const int u0 = static_cast<int>(ch * rk.upc);
            const int nr = min(static_cast<int>(rk.upc), nk - u0);
            // four rows per warp per pass: 4 x G independent reductions
            for (int i0 = C.warp; i0 < nr; i0 += 32) {
                float sc[4][G];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = i0 + 8 * u;
                    float kv[E];
                    if (i < nr) {
                        const float *krow = reinterpret_cast<const float *>(st) + static_cast<size_t>(i) * HD + C.lane * E;
                        if constexpr (E == 4) {
                            const float4 t = *reinterpret_cast<const float4 *>(krow);
                            kv[0] = t.x; kv[1] = t.y; kv[2] = t.z; kv[3] = t.w;
                        } else {
#pragma unroll
                            for (int e = 0; e < E; ++e) kv[e] = krow[e];
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < E; ++e) kv[e] = 0.0f;
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float a = 0.0f;
#pragma unroll
                        for (int e = 0; e < E; ++e) a = fmaf(qreg[h][e], kv[e], a);
                        sc[u][h] = a;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int h = 0; h < G; ++h) sc[u][h] += __shfl_xor_sync(0xffffffffu, sc[u][h], o);
                if (C.lane == 0) {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int h = 0; h < G; ++h)
                            if (i0 + 8 * u < nr) S.scores[h * P.maxpos + u0 + i0 + 8 * u] = sc[u][h] * P.scale;
                }
            }
            C.stage_release();
        }
    }
    if (has_new && C.warp == 0) {
        float sc[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float a = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) a = fmaf(qreg[h][e], knew[C.lane * E + e], a);
            sc[h] = a;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
        if (C.lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) S.scores[h * P.maxpos + nk] = sc[h] * P.scale;
        }
    }
    mcons_sync();
    C.mark(2 * l, 3);
    // per-head partial softmax: warp h
    if (C.warp < G) {
        float *sc = S.scores + C.warp * P.maxpos;
        float m = -INFINITY;
        for (int i = C.lane; i < ntot; i += 32) m = fmaxf(m, sc[i]);
        m = warp_max(m);
        float lsum = 0.0f;
        for (int i = C.lane; i < ntot; i += 32) {
            const float e = expf(sc[i] - m);
            sc[i] = e;
            lsum += e;
        }
        lsum = warp_sum(lsum);
        if (C.lane == 0) {
            S.apub[C.warp * (HD + 4) + HD] = m;
            S.apub[C.warp * (HD + 4) + HD + 1] = lsum;
        }
    }
    mcons_sync();
    // acc = sum_i e_i v_i : warp w takes rows i = w mod 8
    float acc[G][E];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[h][e] = 0.0f;
    {
        const Run rv = make_run(P, R, MI_V, l, p);
        const uint32_t nch = run_chunks(rv);
        for (uint32_t ch = 0; ch < nch; ++ch) {
            const uint8_t *st = C.stage_wait();
            const int u0 = static_cast<int>(ch * rv.upc);
            const int nr = min(static_cast<int>(rv.upc), nk - u0);
            for (int i = C.warp; i < nr; i += 8) {
                const float *vrow = reinterpret_cast<const float *>(st) + static_cast<size_t>(i) * HD;
                float vv[E];
                if constexpr (E == 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(vrow + C.lane * E);
                    vv[0] = t.x; vv[1] = t.y; vv[2] = t.z; vv[3] = t.w;
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) vv[e] = vrow[C.lane * E + e];
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float wgt = S.scores[h * P.maxpos + u0 + i];
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[h][e] = fmaf(wgt, vv[e], acc[h][e]);
                }
            }
            C.stage_release();
        }
    }
    if (has_new && C.warp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float wgt = S.scores[h * P.maxpos + nk];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[h][e] = fmaf(wgt, vnew[C.lane * E + e], acc[h][e]);
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < E; ++e) S.vred[(C.warp * G + h) * HD + C.lane * E + e] = acc[h][e];
    mcons_sync();
    for (int i = C.tid; i < G * HD; i += kMegaConsumers) {
        const int h = i / HD, d = i - h * HD;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += S.vred[(w * G + h) * HD + d];
        S.apub[h * (HD + 4) + d] = s;
    }
    C.mark(2 * l, 4);
    C.cluster_sync();
    // combine the CS partial states of each head (every CTA, same order)
    for (int i = C.tid; i < G * HD; i += kMegaConsumers) {
        const int h = i / HD, d = i - h * HD;
        // issue all 3 x CS remote loads before using any of them
        float mr[kMegaCS], lr[kMegaCS], ar[kMegaCS];
#pragma unroll
        for (int r = 0; r < kMegaCS; ++r) {
            const uint32_t base = dsmem_map(S.apub + h * (HD + 4), static_cast<uint32_t>(r));
            mr[r] = dsmem_ld(base + 4u * HD);
            lr[r] = dsmem_ld(base + 4u * (HD + 1));
            ar[r] = dsmem_ld(base + 4u * d);
        }
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMegaCS; ++r) M = fmaxf(M, mr[r]);
        float L = 0.0f, O = 0.0f;
#pragma unroll
        for (int r = 0; r < kMegaCS; ++r) {
            const float f = (lr[r] > 0.0f) ? expf(mr[r] - M) : 0.0f;
            L = fmaf(lr[r], f, L);
            O = fmaf(ar[r], f, O);
        }
        to_planes(O / L, i >> 5, S.opl, S.osc, C.lane);
    }
    mcons_sync();
    C.mark(2 * l, 5);
    // o_proj rows of this CTA over the group's columns -> opart[group]
    {
        const Run r = make_run(P, R, MI_O, l, p);
        float *dst = P.opart + static_cast<size_t>(R.c) * P.H + R.j * P.ORPC;
        C.gemv_item(r, G * HD, Planes{reinterpret_cast<const uint4 *>(S.opl), S.osc},
                    [dst](int tile, int w, float v) { dst[tile * 8 + w] = v; });
    }
    C.mark(2 * l, 6);
}

__device__ void phase_ffn(Cons &C, int l, int p) {
    const MegaParams &P = C.P;
    const Smem &S = C.S;
    const Role &R = C.R;
    C.mark(2 * l + 1, 0);
    C.rmsnorm();
    C.mark(2 * l + 1, 1);
    {
        const Run r = make_run(P, R, MI_GU, l, p);
        float *gu = S.guout;
        C.gemv_item(r, P.H, Planes{reinterpret_cast<const uint4 *>(S.xpl), S.xsc},
                    [gu](int tile, int w, float v) { gu[tile * 8 + w] = v; });
    }
    mcons_sync();
    C.mark(2 * l + 1, 2);
    for (int a = C.tid; a < R.apc; a += kMegaConsumers) {
        const float g = S.guout[2 * a], u = S.guout[2 * a + 1];
        S.actpub[a] = g / (1.0f + expf(-g)) * u;   // SwiGLU (course 12.3.6)
    }
    C.cluster_sync();
    {
        float g[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = C.tid + u * kMegaConsumers;
            g[u] = 0.0f;
            if (i < R.kt_c) {
                const int src = i / R.apc, off = i - src * R.apc;
                g[u] = dsmem_ld(dsmem_map(S.actpub + off, static_cast<uint32_t>(src)));
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i0 = u * kMegaConsumers + C.warp * 32;   // warp-uniform block start
            if (i0 < R.kt_c) to_planes(g[u], (C.tid + u * kMegaConsumers) >> 5, S.apl, S.asc, C.lane);
        }
    }
    mcons_sync();
    C.mark(2 * l + 1, 3);
    {
        const Run r = make_run(P, R, MI_DOWN, l, p);
        float *dst = P.dpart + static_cast<size_t>(R.c) * P.H + R.j * P.ORPC;
        C.gemv_item(r, R.kt_c, Planes{reinterpret_cast<const uint4 *>(S.apl), S.asc},
                    [dst](int tile, int w, float v) { dst[tile * 8 + w] = v; });
    }
    C.mark(2 * l + 1, 4);
}

__device__ void embed(Cons &C, int tok) {
    const MegaParams &P = C.P;
    for (int i = C.tid; i < P.H; i += kMegaConsumers)
        C.S.x[i] = __half2float(*qm_scale(P.embd, tok, i)) * static_cast<float>(*qm_codes(P.embd, tok, i));
    mcons_sync();
}

// lm_head rows of this CTA with the argmax fold (before the arrive).
__device__ void phase_lm(Cons &C, int s) {
    const MegaParams &P = C.P;
    const Smem &S = C.S;
    const Role &R = C.R;
    C.mark(2 * P.L, 0);
    C.rmsnorm();
    C.mark(2 * P.L, 1);
    const Run r = make_run(P, R, MI_LM, 0, 0);
    const int ng = (P.V + 7) / 8;
    const int g0 = static_cast<int>((static_cast<long long>(R.cta) * ng) / P.NCTA);
    unsigned long long best = 0ull;
    float *logits = P.logits;
    const int V = P.V;
    C.gemv_item(r, P.H, Planes{reinterpret_cast<const uint4 *>(S.xpl), S.xsc}, [&best, logits, V, g0](int tile, int w, float v) {
        const int row = (g0 + tile) * 8 + w;
        if (row < V) {
            if (logits) logits[row] = v;
            const unsigned long long k = argmax_pack(v, row);
            best = k > best ? k : best;
        }
    });
    // rows land in lane 0 (and lane 16 on the half-warp path): fold the warp
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
    }
    if (C.lane == 0) S.keys[C.warp] = best;
    mcons_sync();
    if (C.tid == 0) {
        unsigned long long b = 0ull;
        for (int w = 0; w < 8; ++w) b = S.keys[w] > b ? S.keys[w] : b;
        if (b) atomicMax(P.key + (s & 1), b);
    }
    C.mark(2 * P.L, 2);
}

template <int HD, int G>
__global__ void __launch_bounds__(kMegaThreads, 1) k_decode_mega(const MegaParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    const Smem S = carve(P, smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Role R;
    R.c = static_cast<int>(cluster_id_x());
    R.j = static_cast<int>(cluster_rank());
    R.cta = R.c * P.CS + R.j;
    R.att = R.c < P.NA;
    R.a0 = ffn_a(P, R.c);
    R.kt_c = ffn_a(P, R.c + 1) - R.a0;
    R.apc = R.kt_c / P.CS;

    const unsigned long long t_entry = globaltimer_ns();
    if (tid == 0) {
        for (int i = 0; i < P.NS; ++i) {
            mbar_init(S.full + i, 1);
            mbar_init(S.empty + i, 8);
        }
        mbar_init(S.clbar, static_cast<uint32_t>(P.CS));
        mbar_init(S.clbar + 1, static_cast<uint32_t>(P.CS));
        *S.err = 0;
        fence_mbar_init();
    }
    __syncthreads();
    hw_cluster_sync();   // peers' barriers exist before any remote arrive

    if (warp == 8) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t q = 0;
            bool stop = false;
            unsigned long long w_empty = 0;
            auto issue_run = [&](const Run &r) {
                const uint32_t nch = run_chunks(r);
                for (uint32_t ch = 0; ch < nch && !stop; ++ch) {
                    const int s = static_cast<int>(q % static_cast<uint32_t>(P.NS));
                    const uint32_t n = q / static_cast<uint32_t>(P.NS);
                    const uint64_t tw0 = P.trace ? globaltimer_ns() : 0;
                    if (n >= 1 && !wait_free_slot(S, S.empty + s, (n - 1) & 1u, P.status)) {
                        stop = true;
                        break;
                    }
                    if (P.trace) w_empty += globaltimer_ns() - tw0;
                    const uint32_t u0 = ch * r.upc;
                    const uint32_t nu = min(r.upc, r.n - u0);
                    const uint32_t bytes = nu * r.unit;
                    mbar_arrive_expect_tx(S.full + s, bytes);
                    bulk_g2s(S.ring + static_cast<size_t>(s) * P.SB, r.src + static_cast<size_t>(u0) * r.unit, bytes,
                             S.full + s, pol);
                    ++q;
                }
            };
            for (int st = 0; st < P.n_steps && !stop; ++st) {
                const int p = P.pos0 + st;
                fence_proxy_async_global();
                for (int l = 0; l < P.L && !stop; ++l) {
                    if (R.att) {
                        issue_run(make_run(P, R, MI_QKV, l, p));
                        issue_run(make_run(P, R, MI_K, l, p));
                        issue_run(make_run(P, R, MI_V, l, p));
                        issue_run(make_run(P, R, MI_O, l, p));
                    }
                    issue_run(make_run(P, R, MI_GU, l, p));
                    issue_run(make_run(P, R, MI_DOWN, l, p));
                }
                if (!stop) issue_run(make_run(P, R, MI_LM, 0, p));
            }
            // drain: the last fill of every slot must land before exit
            const uint32_t first = q > static_cast<uint32_t>(P.NS) ? q - static_cast<uint32_t>(P.NS) : 0u;
            for (uint32_t r = first; r < q; ++r) {
                const int s = static_cast<int>(r % static_cast<uint32_t>(P.NS));
                const uint32_t par = (r / static_cast<uint32_t>(P.NS)) & 1u;
                if (!mbar_try_wait(S.full + s, par)) {
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(S.full + s, par) && globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
            if (P.trace) P.trace[(2 * (2 * P.L + 1) + R.cta) * 8 + 3] = w_empty;
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- consumers
        Cons C{P, S, R, tid, warp, lane, 0u, 0u, 0u, nullptr, false, 0ull, 0ull, 0ull};
        if (P.trace && (R.cta == 0 || R.cta == P.NCTA - 1))
            C.trec = P.trace + static_cast<size_t>(R.cta == 0 ? 0 : 1) * (2 * P.L + 1) * 8;
        int tok = P.first_token[0];
        for (int st = 0; st < P.n_steps; ++st) {
            const int p = P.pos0 + st;
            C.last_step = (st == P.n_steps - 1);
            tok = tok < 0 ? 0 : (tok >= P.V ? P.V - 1 : tok);
            if (R.att) C.prefetch_w(P.attn_norm0);
            embed(C, tok);
            for (int l = 0; l < P.L; ++l) {
                if (l > 0) {
                    if (R.att) C.prefetch_w(at_layer(P.attn_norm0, l, P.wstride));
                    C.grid_wait();
                    C.add_partials(P.dpart, P.NC);
                }
                if (R.att) phase_attention<HD, G>(C, l, p);
                C.grid_arrive();
                C.prefetch_w(at_layer(P.ffn_norm0, l, P.wstride));
                C.grid_wait();
                C.add_partials(P.opart, P.NA);
                phase_ffn(C, l, p);
                C.grid_arrive();
            }
            C.prefetch_w(P.out_norm);
            C.grid_wait();
            C.add_partials(P.dpart, P.NC);
            phase_lm(C, st);
            C.grid_arrive();
            C.grid_wait();
            if (tid == 0) {
                const unsigned long long k = __ldcg(P.key + (st & 1));
                const int idx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
                *S.tok = idx;
                if (R.cta == 0) {
                    const float v = float_from_order_key(static_cast<uint32_t>(k >> 32));
                    if (isnan(v) || k == 0ull) record_status(P.status, QW3_ERR_NONFINITE);
                    if (P.hist) P.hist[st] = idx;
                    if (P.argmax_out && st == P.n_steps - 1) P.argmax_out[0] = idx;
                    P.key[(st + 1) & 1] = 0ull;
                }
            }
            mcons_sync();
            C.mark(2 * P.L, 3);
            tok = *S.tok;
        }
        if (P.trace && tid == 0) {
            unsigned long long *rec = P.trace + (2 * (2 * P.L + 1) + R.cta) * 8;
            rec[0] = C.w_full;
            rec[1] = C.w_grid;
            rec[2] = C.w_cl;
            rec[4] = t_entry;
            rec[5] = globaltimer_ns();
            rec[6] = static_cast<unsigned long long>(R.c);
            rec[7] = smid();
        }
    }
    hw_cluster_sync();   // no CTA leaves while a peer may still read its shared memory
}

}  // namespace

// ------------------------------------------------------------------ host

size_t mega_smem_bytes(const MegaParams &P) { return P.o_ring + static_cast<size_t>(P.NS) * P.SB; }

// Instantiations: head_dim 64 or 128, query heads per KV head 1, 2 or 4.
template <typename F>
static cudaError_t mega_dispatch(int hd, int G, F f) {
    if (hd == 128 && G == 1) return f(k_decode_mega<128, 1>);
    if (hd == 128 && G == 2) return f(k_decode_mega<128, 2>);
    if (hd == 128 && G == 4) return f(k_decode_mega<128, 4>);
    if (hd == 64 && G == 1) return f(k_decode_mega<64, 1>);
    if (hd == 64 && G == 2) return f(k_decode_mega<64, 2>);
    if (hd == 64 && G == 4) return f(k_decode_mega<64, 4>);
    return cudaErrorInvalidValue;
}

bool mega_supported_heads(int hd, int G) { return (hd == 64 || hd == 128) && (G == 1 || G == 2 || G == 4); }

cudaError_t configure_mega() {
    cudaError_t e = cudaSuccess;
    for (int hd : {64, 128})
        for (int G : {1, 2, 4}) {
            if (e == cudaSuccess)
                e = mega_dispatch(hd, G, [](auto k) {
                    cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                    if (r == cudaSuccess) r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMegaMaxSmem);
                    return r;
                });
        }
    return e;
}

static void mega_launch_config(const MegaParams &P, cudaLaunchConfig_t &cfg, cudaLaunchAttribute *attr,
                               cudaStream_t s) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(static_cast<unsigned>(P.NCTA));
    cfg.blockDim = dim3(kMegaThreads);
    cfg.dynamicSmemBytes = mega_smem_bytes(P);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(P.CS);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

cudaError_t mega_max_clusters(const MegaParams &P, int *n) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    mega_launch_config(P, cfg, attr, nullptr);
    return mega_dispatch(P.hd, P.G, [&](auto k) { return cudaOccupancyMaxActiveClusters(n, k, &cfg); });
}

cudaError_t launch_mega(const MegaParams &P, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    mega_launch_config(P, cfg, attr, s);
    return mega_dispatch(P.hd, P.G, [&](auto k) { return cudaLaunchKernelEx(&cfg, k, P); });
}

// Column-partitioned down matrix: cluster c owns channels [a_c, a_{c+1}),
// a_c = floor(c * U / NC) * 32 with U = cols / 32; its block holds tiles of
// 8 rows x (a_{c+1} - a_c) columns for every 8-row group, in row order.
__global__ void k_repack_colpart(const uint8_t *__restrict__ raw, int rows, int nbpr, int NC, uint8_t *__restrict__ dst) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= static_cast<int64_t>(rows) * nbpr) return;
    const int r = static_cast<int>(t / nbpr);
    const int jb = static_cast<int>(t % nbpr);
    int c = 0;
    while (c + 1 < NC && ((c + 1) * nbpr / NC) <= jb) ++c;
    const int a = (c * nbpr / NC) * 32, b = ((c + 1) * nbpr / NC) * 32;
    const int kt = b - a;
    const size_t base = static_cast<size_t>(rows / 8) * 17u * static_cast<size_t>(a) / 2u +
                        static_cast<size_t>(r / 8) * (static_cast<size_t>(kt) * 17u / 2u);
    const int kk = 32 * jb - a;
    const uint16_t *bsrc = reinterpret_cast<const uint16_t *>(raw + t * 34);
    reinterpret_cast<uint16_t *>(dst + base + 8 * static_cast<size_t>(kt))[(r & 7) * (kt / 32) + kk / 32] = bsrc[0];
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = static_cast<uint32_t>(bsrc[1 + 2 * k]) | (static_cast<uint32_t>(bsrc[2 + 2 * k]) << 16);
    uint4 *o = reinterpret_cast<uint4 *>(dst + base + static_cast<size_t>(r & 7) * kt + kk);
    o[0] = make_uint4(w[0], w[1], w[2], w[3]);
    o[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

cudaError_t launch_repack_colpart(const uint8_t *raw, int rows, int cols, int NC, uint8_t *dst, cudaStream_t s) {
    const int nbpr = cols / 32;
    const int64_t n = static_cast<int64_t>(rows) * nbpr;
    if (n == 0) return cudaSuccess;
    k_repack_colpart<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(raw, rows, nbpr, NC, dst);
    return cudaGetLastError();
}

}  // namespace qw3
