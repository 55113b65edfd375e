// Grouped-query causal attention ("A transformer from scratch", 12.3.5):
// query head h reads KV head h / (n_heads / n_kv_heads); scores q.k * scale,
// scale = 1/sqrt(head_dim) (minfer 2.1); softmax with the running maximum
// subtracted; output = softmax-weighted sum of V. The cache holds K after the
// per-head norm and RoPE and V as projected (12.4).
//
// KV cache layout (device, f32): [layer][seq][K|V][kv_head][capacity][head_dim]
// so one head's positions are contiguous and stream as single bulk copies.
//
// Decode kernel (one new token per sequence): split-K over the context.
// CTA (g, s, b) covers positions [s*chunk, min((s+1)*chunk, ctx)) of kv head g
// for sequence b, for all n_heads/n_kv query heads of the group at once, so
// each K/V byte is read once. Cached rows are staged by 1-D bulk copies
// (TMA) issued before griddepcontrol.wait: they were written by earlier
// steps. After the wait the CTA applies the per-head Q/K RMSNorm and RoPE to
// the new q/k (minfer 2.2, course 12.3.4); the CTA whose range holds the new
// position also appends k, v to the cache. The nsplit CTAs of one (g, b)
// form a thread-block cluster: each keeps its partial (max, sum, acc) per
// head in shared memory, and after one cluster barrier every CTA merges a
// 1/nsplit share of the outputs from its peers' partials (flash-decoding
// combine through distributed shared memory; no global round trip).
#include "qw3_internal.cuh"

namespace qw3 {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kTileP = 32;   // positions per staged tile
constexpr int kAttnMaxClusters = 8;   // clusters per (sequence, kv head): their partials merge in global memory
constexpr int kStages = 3;

// Splits of one (sequence, kv head) form one cluster; its leader holds a
// partial row per split and head, which caps the cluster at 8 for G = 8.
__host__ __device__ constexpr int attn_max_cluster(int G) { return G <= 4 ? 16 : 8; }

// A partial row holds acc[HD], then m and l; padded to HD + 4 floats so every
// row starts on a 16-byte boundary for the vector stores.
template <int HD>
__host__ __device__ constexpr int part_stride() { return HD + 4; }

template <int HD>
__device__ __forceinline__ void load_lane(const float *src, float (&v)[HD / 32], int lane) {
    constexpr int E = HD / 32;
    if constexpr (E == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(src + lane * 4);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
        const float2 t = *reinterpret_cast<const float2 *>(src + lane * 2);
        v[0] = t.x; v[1] = t.y;
    }
}

template <int HD>
__device__ __forceinline__ void store_lane(float *dst, const float (&v)[HD / 32], int lane) {
    constexpr int E = HD / 32;
    if constexpr (E == 4) {
        *reinterpret_cast<float4 *>(dst + lane * 4) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
        *reinterpret_cast<float2 *>(dst + lane * 2) = make_float2(v[0], v[1]);
    }
}

// load_lane / store_lane for cache elements of type KT (f32 or IEEE half).
template <int HD>
__device__ __forceinline__ void load_lane_kv(const float *src, float (&v)[HD / 32], int lane) {
    load_lane<HD>(src, v, lane);
}

template <int HD>
__device__ __forceinline__ void load_lane_kv(const __half *src, float (&v)[HD / 32], int lane) {
    constexpr int E = HD / 32;
    if constexpr (E == 4) {
        const uint2 t = *reinterpret_cast<const uint2 *>(src + lane * 4);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&t.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&t.y));
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(src + lane * 2));
        v[0] = a.x; v[1] = a.y;
    }
}

// A q8_0 row: the lane's E values from their block's codes and f16 scale.
template <int HD>
__device__ __forceinline__ void load_lane_kv(const kvq8 *src, float (&v)[HD / 32], int lane) {
    constexpr int E = HD / 32, L = 32 / E;
    const uint8_t *blk = &src->b + (lane / L) * 34;
    const float sc = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(blk)));
    const uint16_t *cp = reinterpret_cast<const uint16_t *>(blk + 2 + (lane % L) * E);   // 2-byte aligned
#pragma unroll
    for (int h = 0; h < E / 2; ++h) {
        const uint16_t w = cp[h];
        v[2 * h] = sc * static_cast<float>(static_cast<int8_t>(w & 0xff));
        v[2 * h + 1] = sc * static_cast<float>(static_cast<int8_t>(w >> 8));
    }
}

template <int HD, typename KT>
__device__ __forceinline__ void store_lane_kv(KT *dst, const float (&v)[HD / 32], int lane) {
    constexpr int E = HD / 32;
    if constexpr (kv_is_q8<KT>::value) {
        q8_store_lanes<HD>(dst, v, lane);   // every lane of the warp takes part
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[lane * E + e] = kv_cvt<KT>(v[e]);
    }
}

// Round a lane's values to the cache type and back (identity for f32): the
// value a reader of the cache sees. For q8_0 every lane of the warp calls it.
template <int HD, typename KT>
__device__ __forceinline__ void round_lane_kv(float (&v)[HD / 32]) {
    if constexpr (kv_is_q8<KT>::value) {
        int q[HD / 32];
        __half dh;
        q8_encode_lanes<HD>(v, q, dh);
        const float sc = __half2float(dh);
#pragma unroll
        for (int e = 0; e < HD / 32; ++e) v[e] = sc * static_cast<float>(q[e]);
    } else {
#pragma unroll
        for (int e = 0; e < HD / 32; ++e) v[e] = kv_f32(kv_cvt<KT>(v[e]));
    }
}

// Row j of a run of cached rows (rows are kv_row<KT, HD>() elements apart).
template <int HD, typename T>
__device__ __forceinline__ const T *kv_rowp(const T *rows, int j) {
    return rows + static_cast<size_t>(j) * kv_row<T, HD>();
}

// Positions per staged K/V tile: the tile buffers hold kTileP f32 rows;
// half and q8_0 rows take at most half the bytes, so a tile holds twice the
// positions (kept at kTileP for groups of 8, whose warps score 4 positions at
// a time).
template <typename KT, int G>
__host__ __device__ constexpr int tile_positions() { return (sizeof(KT) <= 2 && G <= 4) ? 2 * kTileP : kTileP; }

// Bytes of one bulk copy of `rows` cached rows, rounded up to the 16 bytes a
// bulk copy moves (a q8_0 row is 34 * HD / 32 bytes; the cache allocation
// carries the padding the last rows may need).
template <typename KT, int HD>
__device__ __forceinline__ uint32_t kv_copy_bytes(int rows) {
    return static_cast<uint32_t>((static_cast<size_t>(rows) * kv_row<KT, HD>() * sizeof(KT) + 15) / 16 * 16);
}

// Preloaded operands of one per-head norm + RoPE: the lane's norm weights
// and (cos, sin) pairs (neither depends on the previous kernel).
template <int HD>
struct NormRope {
    float w[HD / 32];
    float2 cs[HD / 32];
};

template <int HD>
__device__ __forceinline__ void load_norm_rope(NormRope<HD> &nr, const float *w, const float2 *rope_row, int lane) {
    constexpr int E = HD / 32;
    load_lane<HD>(w, nr.w, lane);
#pragma unroll
    for (int e = 0; e < E; ++e) nr.cs[e] = rope_row[(lane & 15) * E + e];
}

// Per-head RMSNorm over head_dim then NeoX rotation, from preloaded operands.
template <int HD>
__device__ __forceinline__ void norm_rope_pre(float (&v)[HD / 32], const NormRope<HD> &nr, float eps, int lane) {
    constexpr int E = HD / 32;
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
    ss = warp_sum(ss);
    const float r = 1.0f / sqrtf(ss / static_cast<float>(HD) + eps);
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = v[e] * r * nr.w[e];
    const bool first_half = lane < 16;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, v[e], 16);
        v[e] = first_half ? (v[e] * nr.cs[e].x - other * nr.cs[e].y) : (other * nr.cs[e].y + v[e] * nr.cs[e].x);
    }
}

template <int HD, int G, typename KT>
__global__ void __launch_bounds__(kAttnThreads) k_attn_decode(AttnDecodeArgs a, int nsplit, int csize) {
    constexpr int E = HD / 32;
    constexpr int TP = tile_positions<KT, G>();
    constexpr int RW = kv_row<KT, HD>();   // cache elements per row
    static_assert((TP * RW * sizeof(KT) + 15) / 16 * 16 <= kTileP * HD * 4, "a K/V tile fits its slot");
    constexpr int PS = part_stride<HD>();
    constexpr int CM = attn_max_cluster(G);
    static_assert(kAttnWarps * G * PS <= kStages * kTileP * HD, "warp-merge rows must fit in the K tiles");
    static_assert(CM * G * PS <= kStages * kTileP * HD, "the leader's partial rows must fit in the V tiles");
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                 // [kStages] K/V tiles
    uint64_t *rbar = bars + kStages;                                      // partials received (leader)
    int *flags = reinterpret_cast<int *>(smem + 64);
    float *ktile_f = reinterpret_cast<float *>(smem + 128);             // [kStages][kTileP][HD] f32 slots
    float *vtile_f = ktile_f + kStages * kTileP * HD;                     // [kStages][kTileP][HD]
    KT *ktile = reinterpret_cast<KT *>(ktile_f);                          // [kStages][TP][HD] cache rows
    KT *vtile = reinterpret_cast<KT *>(vtile_f);
    float *qn = vtile_f + kStages * kTileP * HD;                          // [G][HD]
    float *knew = qn + G * HD;                                            // [HD]
    float *vnew = knew + HD;                                              // [HD]
    // once the tiles are consumed: the warp-merge rows in the K tiles, the
    // split partials pushed to the leader in the V tiles
    float *mrg = ktile_f;                                                 // [kAttnWarps][G][PS]
    float *recv = vtile_f;                                                // [CM][G][PS] (leader)
    float *wts = vnew + HD;                                               // [G][CM] merge weights (leader)
    float *pbuf = wts + G * CM;                                           // [kAttnWarps][32] probabilities
    float *cbuf = pbuf + kAttnWarps * 32;                                 // [kAttnWarps][8] rescale factors

    const int g = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // nsplit splits of the context per (b, g), in nsplit / csize clusters of
    // csize CTAs: cluster kc = s / C, rank r = s % C (rank 0 leads)
    const int C = csize, r = s % csize, kc = s / csize, K2 = nsplit / csize;
    unsigned long long *tr = (tid == 0) ? trace_slot(a.trace) : nullptr;
    if (tr) {
        tr[0] = globaltimer_ns();
        tr[5] = clock64();
        tr[7] = smid();
    }
    // seq_ids and pos are step inputs: the embedding kernel at the head of the
    // step waits for the previous step before it lets later kernels start.
    const int seq = a.seq_ids[b];
    const int p = a.pos[b];
    const int ctx = p + 1;
    // a bulk copy starts 16-byte aligned: f32 and half rows always do; a
    // q8_0 row is 68 or 136 bytes, so a split starts at a multiple of 4
    // positions (4 * 68 = 17 * 16)
    constexpr int kStartAlign = kv_is_q8<KT>::value ? 4 : 1;
    const int chunk = ((ctx + nsplit - 1) / nsplit + kStartAlign - 1) / kStartAlign * kStartAlign;
    const int start = s * chunk;
    const int end = min(ctx, start + chunk);
    const bool has_new = (start <= p) && (p < end);
    const int n_cached = max(0, min(end, p) - start);
    const int ntiles = (n_cached + TP - 1) / TP;

    KT *kbase = static_cast<KT *>(a.kv) + static_cast<size_t>(seq) * a.seq_stride +
                static_cast<size_t>(g) * a.head_stride;
    KT *vbase = kbase + a.kvsel_stride;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
        mbar_init(rbar, 1);
        fence_mbar_init();
        flags[0] = 0;
        flags[1] = 0;
        flags[2] = 0;
        flags[3] = 0;
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    if (tid == 0) {
        for (int t = 0; t < ntiles && t < kStages; ++t) {
            const int rows = min(TP, n_cached - t * TP);
            const uint32_t bytes = kv_copy_bytes<KT, HD>(rows);
            const size_t off = static_cast<size_t>(start + t * TP) * RW;
            mbar_arrive_expect_tx(&bars[t], 2 * bytes);
            bulk_g2s(ktile + t * TP * RW, kbase + off, bytes, &bars[t], pol);
            bulk_g2s(vtile + t * TP * RW, vbase + off, bytes, &bars[t], pol);
        }
        // the leader expects every peer's partial rows (acc, m, l per head)
        if (r == 0) mbar_arrive_expect_tx(rbar, static_cast<uint32_t>((C - 1) * G * (HD * 4 + 8)));
    }
    // norm weights and rotation of this warp's first head task, before the wait
    const float2 *rope_row = a.rope + static_cast<size_t>(p) * (HD / 2);
    NormRope<HD> nr;
    if (warp <= G) load_norm_rope<HD>(nr, warp < G ? a.q_norm : a.k_norm, rope_row, lane);
    pdl_wait();
    if (tr) tr[1] = globaltimer_ns();

    // ---- new token: per-head norm + RoPE of q (and k), append k and v
    const float *qkv_b = a.qkv + static_cast<size_t>(b) * a.qkv_stride;
    for (int t = warp; t < G + 2; t += kAttnWarps) {
        if (t != warp && t <= G) load_norm_rope<HD>(nr, t < G ? a.q_norm : a.k_norm, rope_row, lane);
        float v[E];
        if (t < G) {
            load_lane<HD>(qkv_b + (g * G + t) * HD, v, lane);
            norm_rope_pre<HD>(v, nr, a.eps, lane);
            // q8_0 cache: the query row goes through Q8_0 once per head, so
            // each f32 score below is (k.d * q.d) * the integer dot of the
            // codes, to f32 rounding ("The LLM stack", 13.4)
            if constexpr (kv_is_q8<KT>::value) round_lane_kv<HD, KT>(v);
            store_lane<HD>(qn + t * HD, v, lane);
        } else if (has_new && t == G) {
            load_lane<HD>(qkv_b + a.nh * HD + g * HD, v, lane);
            norm_rope_pre<HD>(v, nr, a.eps, lane);
            round_lane_kv<HD, KT>(v);   // the new position is scored from its cached value
            store_lane<HD>(knew, v, lane);
            store_lane_kv<HD>(kbase + static_cast<size_t>(p) * RW, v, lane);
        } else if (has_new && t == G + 1) {
            load_lane<HD>(qkv_b + (a.nh + a.nkv) * HD + g * HD, v, lane);
            round_lane_kv<HD, KT>(v);
            store_lane<HD>(vnew, v, lane);
            store_lane_kv<HD>(vbase + static_cast<size_t>(p) * RW, v, lane);
        }
    }
    __syncthreads();
    pdl_trigger();
    if (tr) tr[2] = globaltimer_ns();

    float qv[G][E];
#pragma unroll
    for (int t = 0; t < G; ++t) load_lane<HD>(qn + t * HD, qv[t], lane);
    float acc[G][E];
#pragma unroll
    for (int t = 0; t < G; ++t)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[t][e] = 0.0f;

    // A warp scores NP positions at once: the G*NP dot products (each spread
    // over the lanes' dims) are summed by one reduce-scatter butterfly, after
    // which lane k (k < V = G*NP, repeated above V) holds the score of head
    // k / NP at position k % NP. Each lane keeps the running max and sum of
    // its own head (online softmax, one exp per lane per batch); the
    // probabilities and rescale factors reach every lane through the warp's
    // shared-memory slots for the P.V accumulation over the lanes' dims.
    constexpr int NP = G <= 4 ? 8 : 4;
    constexpr int V = G * NP;
    static_assert(V <= 32, "one score per lane");
    float *pb = pbuf + warp * 32;
    float *cb = cbuf + warp * 8;
    const int k_own = lane & (V - 1);
    const int t_own = k_own / NP, j_own = k_own % NP;
    float m_own = -INFINITY, l_own = 0.0f;
    auto consume = [&](const auto *krows, const auto *vrows, int n) {
        float sc[V];
        {
            float kv_[NP][E];
#pragma unroll
            for (int j = 0; j < NP; ++j) {
                if (j < n) {
                    load_lane_kv<HD>(kv_rowp<HD>(krows, j), kv_[j], lane);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) kv_[j][e] = 0.0f;
                }
            }
#pragma unroll
            for (int t = 0; t < G; ++t)
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    float d = 0.0f;
#pragma unroll
                    for (int e = 0; e < E; ++e) d = fmaf(qv[t][e], kv_[j][e], d);
                    sc[t * NP + j] = d;
                }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            if (o >= V) {
#pragma unroll
                for (int i = 0; i < V; ++i) sc[i] += __shfl_xor_sync(0xffffffffu, sc[i], o);
            } else {
                // keep the upper half of the 2o values when lane bit o is set
                const bool up = (lane & o) != 0;
#pragma unroll
                for (int i = 0; i < o; ++i) {
                    const float send = up ? sc[i] : sc[i + o];
                    const float keep = up ? sc[i + o] : sc[i];
                    sc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
        }
        const bool valid = j_own < n;
        const float sv = valid ? sc[0] * a.scale : -INFINITY;
        float mx = sv;
#pragma unroll
        for (int o = 1; o < NP; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m_own, mx);
        const float pr = valid ? expf(sv - m_new) : 0.0f;
        const float corr = expf(m_own - m_new);
        float ps = pr;
#pragma unroll
        for (int o = 1; o < NP; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l_own = fmaf(l_own, corr, ps);
        m_own = m_new;
        if (lane < V) {
            pb[lane] = pr;
            if (j_own == 0) cb[t_own] = corr;
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < G; ++t) {
            const float c = cb[t];
#pragma unroll
            for (int e = 0; e < E; ++e) acc[t][e] *= c;
        }
#pragma unroll
        for (int j = 0; j < NP; ++j) {
            if (j < n) {
                float vv[E];
                load_lane_kv<HD>(kv_rowp<HD>(vrows, j), vv, lane);
#pragma unroll
                for (int t = 0; t < G; ++t) {
                    const float pj = pb[t * NP + j];
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[t][e] = fmaf(pj, vv[e], acc[t][e]);
                }
            }
        }
        __syncwarp();
    };

    // WPT warps share a tile (NP positions each); TPI tiles are consumed per
    // round, the next ones already in flight in the remaining stages.
    constexpr int WPT = TP / NP;
    constexpr int TPI = kAttnWarps / WPT;
    static_assert(TPI >= 1 && TPI < kStages, "a stage stays in flight while a round is consumed");
    for (int t0 = 0; t0 < ntiles; t0 += TPI) {
        const int t = t0 + warp / WPT;
        if (t < ntiles) {
            const int si = t % kStages;
            if (!mbar_wait_bounded(&bars[si], static_cast<uint32_t>((t / kStages) & 1))) {
                flags[0] = 1;
                flags[1] = t0;
            } else {
                const int rows = min(TP, n_cached - t * TP);
                const int j0 = (warp % WPT) * NP;
                if (j0 < rows)
                    consume(ktile + (si * TP + j0) * RW, vtile + (si * TP + j0) * RW, min(NP, rows - j0));
            }
        }
        __syncthreads();
        if (flags[0]) break;
        if (tid == 0) {
            for (int tt = t0 + kStages; tt < t0 + kStages + TPI && tt < ntiles; ++tt) {
                const int si = tt % kStages;
                const int rows = min(TP, n_cached - tt * TP);
                const uint32_t bytes = kv_copy_bytes<KT, HD>(rows);
                const size_t off = static_cast<size_t>(start + tt * TP) * RW;
                mbar_arrive_expect_tx(&bars[si], 2 * bytes);
                bulk_g2s(ktile + si * TP * RW, kbase + off, bytes, &bars[si], pol);
                bulk_g2s(vtile + si * TP * RW, vbase + off, bytes, &bars[si], pol);
            }
        }
        __syncthreads();
    }
    if (flags[0]) {
        // A stage never completed: report, drain the copies that may still
        // be in flight (bounded), and contribute an empty partial so that
        // the leader's combine still completes.
        if (tid == 0) {
            record_status(a.status, QW3_ERR_TIMEOUT);
            const int first = flags[1];
            for (int t = first; t < ntiles && t < first + kStages; ++t)
                (void)mbar_wait_bounded(&bars[t % kStages], static_cast<uint32_t>((t / kStages) & 1));
        }
        m_own = -INFINITY;
        l_own = 0.0f;
#pragma unroll
        for (int t = 0; t < G; ++t)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[t][e] = 0.0f;
    } else if (has_new && warp == kAttnWarps - 1) {
        consume(knew, vnew, 1);
    }
    __syncthreads();   // no copy in flight and no warp reading the K/V tiles: they hold mrg and recv next
    // the leader's V tiles take partials only once it is done with them (and
    // its barrier is armed): arrive now, wait just before the push
    cluster_arrive_release();
    if (tr) tr[3] = globaltimer_ns();

    // ---- merge the warps into this split's partial and push it to the
    // leader (split 0): acc, then (m, l), into its slot s of recv
#pragma unroll
    for (int t = 0; t < G; ++t) {
        float *mw = mrg + (warp * G + t) * PS;
        store_lane<HD>(mw, acc[t], lane);
        if (lane == t * NP) {   // a lane of head t's group holds its (m, l)
            mw[HD] = m_own;
            mw[HD + 1] = l_own;
        }
    }
    __syncthreads();
    cluster_wait_acquire();
    const uint32_t rbar_leader = dsmem_map(rbar, 0u);
    for (int t = warp; t < G; t += kAttnWarps) {
        float M = -INFINITY;
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mrg[(w * G + t) * PS + HD]);
        float L = 0.0f, o[E];
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = 0.0f;
        if (M != -INFINITY) {
            for (int w = 0; w < kAttnWarps; ++w) {
                const float *mw = mrg + (w * G + t) * PS;
                const float f = expf(mw[HD] - M);
                L = fmaf(mw[HD + 1], f, L);
                float aw[E];
                load_lane<HD>(mw, aw, lane);
#pragma unroll
                for (int e = 0; e < E; ++e) o[e] = fmaf(aw[e], f, o[e]);
            }
        }
        float *slot = recv + (r * G + t) * PS;
        if (r == 0) {
            store_lane<HD>(slot, o, lane);
            if (lane == 0) {
                slot[HD] = M;
                slot[HD + 1] = L;
            }
        } else {
            const uint32_t dst = dsmem_map(slot, 0u);
            if constexpr (E == 4) {
                st_async_f32x4(dst + 16u * lane, o[0], o[1], o[2], o[3], rbar_leader);
            } else {
                st_async_f32x2(dst + 8u * lane, o[0], o[1], rbar_leader);
            }
            if (lane == 0) st_async_f32x2(dst + 4u * HD, M, L, rbar_leader);
        }
    }
    if (r == 0) {
        // ---- leader: flash-decoding combine of the C split partials (with
        // several clusters per (b, g): the cluster's unnormalised partial to
        // global memory, the last leader to arrive merges them)
        if (tid == 0 && !mbar_wait_bounded_cluster(rbar, 0u)) flags[2] = 1;
        __syncthreads();
        // On a timeout the peers' partials are not trusted: every split
        // counts as empty, but the merge (and, with several clusters, the
        // arrival on the counter the last leader resets) still runs.
        const bool tmo = flags[2] != 0;
        if (tmo && tid == 0) record_status(a.status, QW3_ERR_TIMEOUT);
        {
            if (warp < G) {
                // warp t: lane j holds split j's (m, l) of head t
                const int t = warp;
                const float mj = (lane < C && !tmo) ? recv[(lane * G + t) * PS + HD] : -INFINITY;
                const float lj = (lane < C && !tmo) ? recv[(lane * G + t) * PS + HD + 1] : 0.0f;
                const float M = warp_max(mj);
                const float f = (mj == -INFINITY) ? 0.0f : expf(mj - M);
                const float L = warp_sum(lj * f);
                if (lane < C) wts[t * CM + lane] = K2 > 1 ? f : (L > 0.0f ? f * (1.0f / L) : 0.0f);
                if (K2 > 1 && lane == 0) {
                    float *cp = a.cpart + ((static_cast<size_t>(b) * a.nkv + g) * K2 + kc) * G * PS + t * PS;
                    cp[HD] = M;
                    cp[HD + 1] = L;
                }
            }
            __syncthreads();
            float *ob = K2 > 1 ? a.cpart + ((static_cast<size_t>(b) * a.nkv + g) * K2 + kc) * G * PS
                               : a.out + static_cast<size_t>(b) * a.nh * HD + static_cast<size_t>(g) * G * HD;
            for (int o = tid; o < G * HD; o += kAttnThreads) {
                const int t = o / HD, d = o - (o / HD) * HD;
                float v[CM];
#pragma unroll
                for (int j = 0; j < CM; ++j) v[j] = (j < C && !tmo) ? recv[(j * G + t) * PS + d] : 0.0f;
                float sum = 0.0f;
#pragma unroll
                for (int j = 0; j < CM; ++j)
                    if (j < C) sum = fmaf(wts[t * CM + j], v[j], sum);
                if (K2 > 1) {
                    ob[t * PS + d] = sum;
                } else {
                    ob[o] = sum;
                }
            }
            if (K2 > 1) {
                // second level: the last of the K2 leaders merges the clusters
                __threadfence();
                __syncthreads();
                if (tid == 0) {
                    const unsigned prev = atomicAdd(&a.ccnt[b * a.nkv + g], 1u);
                    flags[3] = (prev == static_cast<unsigned>(K2 - 1)) ? 1 : 0;
                }
                __syncthreads();
                if (flags[3]) {
                    __threadfence();
                    const float *cp = a.cpart + (static_cast<size_t>(b) * a.nkv + g) * K2 * G * PS;
                    if (warp < G) {
                        const int t = warp;
                        const float mc = lane < K2 ? __ldcg(cp + (lane * G + t) * PS + HD) : -INFINITY;
                        const float lc = lane < K2 ? __ldcg(cp + (lane * G + t) * PS + HD + 1) : 0.0f;
                        const float M = warp_max(mc);
                        const float f = (mc == -INFINITY) ? 0.0f : expf(mc - M);
                        const float L = warp_sum(lc * f);
                        if (lane < K2) wts[t * CM + lane] = L > 0.0f ? f * (1.0f / L) : 0.0f;
                    }
                    __syncthreads();
                    float *out = a.out + static_cast<size_t>(b) * a.nh * HD + static_cast<size_t>(g) * G * HD;
                    for (int o = tid; o < G * HD; o += kAttnThreads) {
                        const int t = o / HD, d = o - (o / HD) * HD;
                        float sum = 0.0f;
                        for (int c = 0; c < K2; ++c) sum = fmaf(wts[t * CM + c], __ldcg(cp + (c * G + t) * PS + d), sum);
                        out[o] = sum;
                    }
                    if (tid == 0) a.ccnt[b * a.nkv + g] = 0u;
                }
            }
        }
    }
    if (tr) {
        tr[4] = globaltimer_ns();
        tr[6] = clock64();
    }
}

size_t attn_decode_smem(int HD, int G) {
    // K/V tiles (the warp-merge rows and the leader's partials reuse them),
    // q rows, new k and v, merge weights, per-warp probabilities and factors
    const size_t floats = static_cast<size_t>(2) * kStages * kTileP * HD + static_cast<size_t>(G) * HD + 2 * HD +
                          static_cast<size_t>(G) * attn_max_cluster(G) + kAttnWarps * 32 + kAttnWarps * 8;
    return 128 + floats * 4;
}

template <int HD, int G, typename KT>
cudaError_t configure_attn_kt() {
    cudaError_t e = cudaFuncSetAttribute(k_attn_decode<HD, G, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(attn_decode_smem(HD, G)));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_attn_decode<HD, G, KT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_attn_decode<HD, G, KT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

template <int HD, int G>
cudaError_t configure_attn_t() {
    cudaError_t e = configure_attn_kt<HD, G, float>();
    if (e == cudaSuccess) e = configure_attn_kt<HD, G, __half>();
    if (e == cudaSuccess) e = configure_attn_kt<HD, G, kvq8>();
    return e;
}

// Largest cluster (splits per kv head) of at most attn_max_cluster(G) CTAs
// such that `units` clusters run at once on this device (one wave for batch
// 1); else the largest that fits at all.
template <int HD, int G>
int max_cluster_t(int units) {
    int fallback = 1;
    for (int c = attn_max_cluster(G); c > 1; c /= 2) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(1, c, 1);
        cfg.blockDim = dim3(kAttnThreads);
        cfg.dynamicSmemBytes = attn_decode_smem(HD, G);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = static_cast<unsigned>(c);
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_attn_decode<HD, G, float>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        if (n >= units) return c;
        if (n >= 1 && fallback == 1) fallback = c;
    }
    return fallback;
}

template <int HD, int G>
cudaError_t launch_attn_t(const AttnDecodeArgs &a, int B, int nsplit, int csize, bool pdl, cudaStream_t s) {
    const size_t smem = attn_decode_smem(HD, G);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.nkv, nsplit, B);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    if (a.kvtype == KV_F16) return cudaLaunchKernelEx(&cfg, k_attn_decode<HD, G, __half>, a, nsplit, csize);
    if (a.kvtype == KV_Q8) return cudaLaunchKernelEx(&cfg, k_attn_decode<HD, G, kvq8>, a, nsplit, csize);
    return cudaLaunchKernelEx(&cfg, k_attn_decode<HD, G, float>, a, nsplit, csize);
}

// ------------------------------------------------------------- prefill
// Causal flash attention over a chunk of M query rows at positions
// pos0..pos0+M-1, keys 0..pos0+M-1 from the cache (this chunk's rows were
// appended just before). CTA = (64-query tile, query head); warp w owns 8
// query rows; for each 32-key tile lane j scores key j, then lanes own
// head_dim slices for the P.V product. f32 throughout.
// Values c..c+3 (c % 4 == 0) of a cached row.
template <int HD>
__device__ __forceinline__ float4 ld4_row(const float *row, int c) { return *reinterpret_cast<const float4 *>(row + c); }
__device__ __forceinline__ float4 ld4_kv(const __half *p);
template <int HD>
__device__ __forceinline__ float4 ld4_row(const __half *row, int c) { return ld4_kv(row + c); }
template <int HD>
__device__ __forceinline__ float4 ld4_row(const kvq8 *row, int c) {
    const uint8_t *blk = &row->b + (c >> 5) * 34;
    const float sc = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(blk)));
    const uint16_t *cp = reinterpret_cast<const uint16_t *>(blk + 2 + (c & 31));   // 2-byte aligned
    const uint16_t a = cp[0], b = cp[1];
    return make_float4(sc * static_cast<float>(static_cast<int8_t>(a & 0xff)),
                       sc * static_cast<float>(static_cast<int8_t>(a >> 8)),
                       sc * static_cast<float>(static_cast<int8_t>(b & 0xff)),
                       sc * static_cast<float>(static_cast<int8_t>(b >> 8)));
}
__device__ __forceinline__ float4 ld4_kv(const __half *p) {
    const uint2 t = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&t.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&t.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int HD, typename KT>
__global__ void __launch_bounds__(256) k_attn_prefill(const float *__restrict__ qkv, int M, int qkv_stride,
                                                      const KT *__restrict__ kv_k, const KT *__restrict__ kv_v,
                                                      size_t head_stride, int pos0, int nh, int group, float scale,
                                                      float *__restrict__ out) {
    constexpr int E = HD / 32;
    constexpr int KP = HD + 4;   // padded K row
    extern __shared__ __align__(16) float sm[];
    float *Qs = sm;                       // [64][HD]
    float *Ks = Qs + 64 * HD;             // [32][KP]
    float *Vs = Ks + 32 * KP;             // [32][HD]
    float *Ps = Vs + 32 * HD;             // [8 warps][8][32]
    const int tile = gridDim.x - 1 - blockIdx.x;   // heavy (late) tiles first
    const int h = blockIdx.y;
    const int g = h / group;
    const int q0 = tile * 64;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const KT *kb = kv_k + static_cast<size_t>(g) * head_stride;
    const KT *vb = kv_v + static_cast<size_t>(g) * head_stride;

    for (int i = tid; i < 64 * HD / 4; i += 256) {
        const int r = (i * 4) / HD, c = (i * 4) % HD;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q0 + r < M) v = *reinterpret_cast<const float4 *>(qkv + static_cast<size_t>(q0 + r) * qkv_stride + h * HD + c);
        *reinterpret_cast<float4 *>(Qs + r * HD + c) = v;
    }
    float m[8], l[8], acc[8][E];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[r][e] = 0.0f;
    }
    const int last_q = min(M, q0 + 64) - 1;
    const int nkeys = pos0 + last_q + 1;
    for (int t0 = 0; t0 < nkeys; t0 += 32) {
        __syncthreads();
        for (int i = tid; i < 32 * HD / 4; i += 256) {
            const int r = (i * 4) / HD, c = (i * 4) % HD;
            float4 kv4 = make_float4(0.f, 0.f, 0.f, 0.f), vv4 = kv4;
            if (t0 + r < nkeys) {
                kv4 = ld4_row<HD>(kv_rowp<HD>(kb, t0 + r), c);
                vv4 = ld4_row<HD>(kv_rowp<HD>(vb, t0 + r), c);
            }
            *reinterpret_cast<float4 *>(Ks + r * KP + c) = kv4;
            *reinterpret_cast<float4 *>(Vs + r * HD + c) = vv4;
        }
        __syncthreads();
        float s[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) s[r] = 0.0f;
        for (int d = 0; d < HD; d += 4) {
            const float4 k4 = *reinterpret_cast<const float4 *>(Ks + lane * KP + d);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float4 q4 = *reinterpret_cast<const float4 *>(Qs + (warp * 8 + r) * HD + d);
                s[r] = fmaf(q4.x, k4.x, s[r]);
                s[r] = fmaf(q4.y, k4.y, s[r]);
                s[r] = fmaf(q4.z, k4.z, s[r]);
                s[r] = fmaf(q4.w, k4.w, s[r]);
            }
        }
        const int kpos = t0 + lane;
        float corr[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int qpos = pos0 + q0 + warp * 8 + r;
            const float sc = (kpos <= qpos && kpos < nkeys) ? s[r] * scale : -INFINITY;
            const float mx = warp_max(sc);
            const float mn = fmaxf(m[r], mx);
            // rows beyond M, or with nothing visible yet, keep m = -inf
            const float pr = (mn == -INFINITY) ? 0.0f : expf(sc - mn);
            corr[r] = (mn == -INFINITY) ? 1.0f : expf(m[r] - mn);
            l[r] = l[r] * corr[r] + warp_sum(pr);
            m[r] = mn;
            Ps[(warp * 8 + r) * 32 + lane] = pr;
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] *= corr[r];
        for (int j = 0; j < 32; ++j) {
            float vv[E];
            load_lane<HD>(Vs + j * HD, vv, lane);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float pj = Ps[(warp * 8 + r) * 32 + j];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[r][e] = fmaf(pj, vv[e], acc[r][e]);
            }
        }
        __syncwarp();
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int row = q0 + warp * 8 + r;
        if (row < M) {
            const float inv = 1.0f / l[r];
            float o[E];
#pragma unroll
            for (int e = 0; e < E; ++e) o[e] = acc[r][e] * inv;
            store_lane<HD>(out + static_cast<size_t>(row) * nh * HD + h * HD, o, lane);
        }
    }
}

template <int HD>
size_t prefill_smem() {
    return static_cast<size_t>(64 * HD + 32 * (HD + 4) + 32 * HD + 8 * 8 * 32) * 4;
}

template <int HD, typename KT>
cudaError_t launch_prefill_t(const float *qkv, int M, int qkv_stride, const KT *kv_k, const KT *kv_v,
                             size_t head_stride, int pos0, int nh, int group, float scale, float *out,
                             cudaStream_t s) {
    const size_t smem = prefill_smem<HD>();
    dim3 grid((M + 63) / 64, nh);
    k_attn_prefill<HD, KT><<<grid, 256, smem, s>>>(qkv, M, qkv_stride, kv_k, kv_v, head_stride, pos0, nh, group,
                                                   scale, out);
    return cudaGetLastError();
}

template <typename KT>
cudaError_t launch_prefill_kt(const float *qkv, int M, int qkv_stride, const KT *kk, size_t kvsel_stride,
                              size_t head_stride, int pos0, int nh, int nkv, int hd, float scale, float *out,
                              cudaStream_t s) {
    const KT *vv = kk + kvsel_stride;
    const int group = nh / nkv;
    if (hd == 128) return launch_prefill_t<128, KT>(qkv, M, qkv_stride, kk, vv, head_stride, pos0, nh, group, scale, out, s);
    if (hd == 64) return launch_prefill_t<64, KT>(qkv, M, qkv_stride, kk, vv, head_stride, pos0, nh, group, scale, out, s);
    return cudaErrorInvalidValue;
}

}  // namespace

int attn_decode_max_nsplit(int hd, int G, int units) {
    if (hd == 128) {
        switch (G) {
            case 1: return max_cluster_t<128, 1>(units);
            case 2: return max_cluster_t<128, 2>(units);
            case 4: return max_cluster_t<128, 4>(units);
            case 8: return max_cluster_t<128, 8>(units);
            default: break;
        }
    } else if (hd == 64) {
        switch (G) {
            case 1: return max_cluster_t<64, 1>(units);
            case 2: return max_cluster_t<64, 2>(units);
            case 4: return max_cluster_t<64, 4>(units);
            case 8: return max_cluster_t<64, 8>(units);
            default: break;
        }
    }
    return 8;
}

cudaError_t configure_attention() {
    cudaError_t e;
#define QW3_CFG(x) if ((e = (x)) != cudaSuccess) return e
    QW3_CFG((configure_attn_t<128, 1>()));
    QW3_CFG((configure_attn_t<128, 2>()));
    QW3_CFG((configure_attn_t<128, 4>()));
    QW3_CFG((configure_attn_t<128, 8>()));
    QW3_CFG((configure_attn_t<64, 1>()));
    QW3_CFG((configure_attn_t<64, 2>()));
    QW3_CFG((configure_attn_t<64, 4>()));
    QW3_CFG((configure_attn_t<64, 8>()));
    QW3_CFG(cudaFuncSetAttribute(k_attn_prefill<128, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem<128>())));
    QW3_CFG(cudaFuncSetAttribute(k_attn_prefill<64, float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem<64>())));
    QW3_CFG(cudaFuncSetAttribute(k_attn_prefill<128, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem<128>())));
    QW3_CFG(cudaFuncSetAttribute(k_attn_prefill<64, __half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem<64>())));
    QW3_CFG(cudaFuncSetAttribute(k_attn_prefill<128, kvq8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem<128>())));
    QW3_CFG(cudaFuncSetAttribute(k_attn_prefill<64, kvq8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(prefill_smem<64>())));
#undef QW3_CFG
    return cudaSuccess;
}

cudaError_t launch_attn_decode(const AttnDecodeArgs &a, int B, int nsplit, int csize, bool pdl, cudaStream_t s) {
    const int G = a.nh / a.nkv;
    if (csize < 1 || csize > attn_max_cluster(G) || nsplit % csize != 0 || nsplit / csize > kAttnMaxClusters ||
        (nsplit > csize && (!a.cpart || !a.ccnt)))
        return cudaErrorInvalidValue;
    if (a.hd == 128) {
        switch (G) {
            case 1: return launch_attn_t<128, 1>(a, B, nsplit, csize, pdl, s);
            case 2: return launch_attn_t<128, 2>(a, B, nsplit, csize, pdl, s);
            case 4: return launch_attn_t<128, 4>(a, B, nsplit, csize, pdl, s);
            case 8: return launch_attn_t<128, 8>(a, B, nsplit, csize, pdl, s);
            default: break;
        }
    } else if (a.hd == 64) {
        switch (G) {
            case 1: return launch_attn_t<64, 1>(a, B, nsplit, csize, pdl, s);
            case 2: return launch_attn_t<64, 2>(a, B, nsplit, csize, pdl, s);
            case 4: return launch_attn_t<64, 4>(a, B, nsplit, csize, pdl, s);
            case 8: return launch_attn_t<64, 8>(a, B, nsplit, csize, pdl, s);
            default: break;
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_prefill(const float *qkv, int M, int qkv_stride, const void *kv_seq, size_t kvsel_stride,
                                size_t head_stride, int pos0, int nh, int nkv, int hd, float scale, float *out,
                                int kvtype, cudaStream_t s) {
    if (kvtype == KV_F16)
        return launch_prefill_kt(qkv, M, qkv_stride, static_cast<const __half *>(kv_seq), kvsel_stride, head_stride,
                                 pos0, nh, nkv, hd, scale, out, s);
    if (kvtype == KV_Q8)
        return launch_prefill_kt(qkv, M, qkv_stride, static_cast<const kvq8 *>(kv_seq), kvsel_stride, head_stride,
                                 pos0, nh, nkv, hd, scale, out, s);
    return launch_prefill_kt(qkv, M, qkv_stride, static_cast<const float *>(kv_seq), kvsel_stride, head_stride, pos0,
                             nh, nkv, hd, scale, out, s);
}

}  // namespace qw3
