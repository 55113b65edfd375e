// Small glue kernels: embedding gather (course 12.3.1), row RMSNorm (12.3.2),
// per-head Q/K norm + RoPE + KV append over many rows (minfer 2.2, course
// 12.3.4, 12.4), the argmax finish of the batched path (12.6) and a KV
// read-back for diagnostics.
#include <algorithm>
#include <climits>

#include "qw3_internal.cuh"

namespace qw3 {

namespace {

// x[i][:] = d * q of embedding row tokens[i] (dequantised on the fly).
__global__ void __launch_bounds__(256) k_embed(const int32_t *__restrict__ tokens, const QMat E, int H, int vocab,
                                               float *__restrict__ x, unsigned long long *trace) {
    unsigned long long *tr = (threadIdx.x == 0) ? trace_slot(trace) : nullptr;
    if (tr) {
        tr[0] = globaltimer_ns();
        tr[5] = clock64();
        tr[7] = smid();
    }
    pdl_wait();
    pdl_trigger();
    if (tr) tr[1] = tr[2] = tr[3] = globaltimer_ns();
    const int i = blockIdx.x;
    int t = tokens[i];
    t = t < 0 ? 0 : (t >= vocab ? vocab - 1 : t);   // ids are validated on the host
    for (int k = threadIdx.x; k < H; k += blockDim.x)
        x[static_cast<size_t>(i) * H + k] = __half2float(*qm_scale(E, t, k)) * static_cast<float>(*qm_codes(E, t, k));
    if (tr) {
        tr[4] = globaltimer_ns();
        tr[6] = clock64();
    }
}

__global__ void __launch_bounds__(256) k_rmsnorm_rows(const float *__restrict__ x, int K,
                                                      const float *__restrict__ w, float eps,
                                                      float *__restrict__ y) {
    __shared__ float red[9];
    const int m = blockIdx.x;
    const float *xr = x + static_cast<size_t>(m) * K;
    float ss = 0.0f;
    for (int k = threadIdx.x; k < K; k += 256) ss = fmaf(xr[k], xr[k], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float t = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
        t = warp_sum(t);
        if (threadIdx.x == 0) red[8] = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
    }
    __syncthreads();
    const float r = red[8];
    for (int k = threadIdx.x; k < K; k += 256) y[static_cast<size_t>(m) * K + k] = xr[k] * r * w[k];
}

// One warp per (row, head task): q heads normalised and rotated in place,
// k heads normalised, rotated and written to the cache, v heads copied.
template <int HD, typename KT>
__global__ void __launch_bounds__(128) k_qk_rope_append(float *__restrict__ qkv, int M, int qkv_stride,
                                                        const float *__restrict__ q_norm,
                                                        const float *__restrict__ k_norm, float eps,
                                                        const float2 *__restrict__ rope,
                                                        const int32_t *__restrict__ row_seq, int seq0,
                                                        const int32_t *__restrict__ row_pos, int pos0,
                                                        KT *__restrict__ kv_layer, size_t seq_stride,
                                                        size_t kvsel_stride, size_t head_stride, int nh,
                                                        int nkv) {
    constexpr int E = HD / 32;
    const int lane = threadIdx.x & 31;
    const int task = blockIdx.y * 4 + (threadIdx.x >> 5);
    const int row = blockIdx.x;
    if (task >= nh + 2 * nkv || row >= M) return;
    const int seq = row_seq ? row_seq[row] : seq0;
    const int pos = row_pos ? row_pos[row] : pos0 + row;
    float *src = qkv + static_cast<size_t>(row) * qkv_stride + task * HD;
    constexpr int RW = kv_row<KT, HD>();
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = src[lane * E + e];
    if (task < nh + nkv) {
        const float *w = task < nh ? q_norm : k_norm;
        float ss = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) ss = fmaf(v[e], v[e], ss);
        ss = warp_sum(ss);
        const float r = 1.0f / sqrtf(ss / static_cast<float>(HD) + eps);
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = v[e] * r * w[lane * E + e];
        const float2 *rr = rope + static_cast<size_t>(pos) * (HD / 2);
        const bool first = lane < 16;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float o = __shfl_xor_sync(0xffffffffu, v[e], 16);
            const float2 cs = rr[(lane & 15) * E + e];
            v[e] = first ? (v[e] * cs.x - o * cs.y) : (o * cs.y + v[e] * cs.x);
        }
    }
    if (task < nh) {
#pragma unroll
        for (int e = 0; e < E; ++e) src[lane * E + e] = v[e];
    } else {
        const int kvsel = task < nh + nkv ? 0 : 1;
        const int g = task - nh - kvsel * nkv;
        KT *dst = kv_layer + static_cast<size_t>(seq) * seq_stride + kvsel * kvsel_stride +
                  static_cast<size_t>(g) * head_stride + static_cast<size_t>(pos) * RW;
        if constexpr (kv_is_q8<KT>::value) {
            q8_store_lanes<HD>(dst, v, lane);   // the whole warp runs this task
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) dst[lane * E + e] = kv_cvt<KT>(v[e]);
        }
    }
}

// One CTA per row: each thread keeps the first maximum of its strided
// columns, then (value, index) pairs reduce to the largest value, lowest
// index on ties.
__global__ void __launch_bounds__(512) k_argmax_rows(const float *__restrict__ logits, int V,
                                                     int32_t *__restrict__ out, int32_t *status) {
    __shared__ float sv[16];
    __shared__ int si[16];
    const float *row = logits + static_cast<size_t>(blockIdx.x) * V;
    float best = -INFINITY;
    int bi = INT_MAX;
    bool nan = false;
    for (int i = threadIdx.x; i < V; i += blockDim.x) {
        const float v = row[i];
        if (v != v) nan = true;
        else if (v > best || bi == INT_MAX) {
            best = v;
            bi = i;
        }
    }
    if (nan) record_status(status, QW3_ERR_NONFINITE);
    auto better = [](float v, int i, float bv, int bj) { return v > bv || (v == bv && i < bj); };
    for (int o = 16; o > 0; o >>= 1) {
        const float v = __shfl_xor_sync(0xffffffffu, best, o);
        const int i = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(v, i, best, bi)) {
            best = v;
            bi = i;
        }
    }
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) {
        sv[warp] = best;
        si[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x / 32;
        best = lane < nw ? sv[lane] : -INFINITY;
        bi = lane < nw ? si[lane] : INT_MAX;
        for (int o = 16; o > 0; o >>= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, best, o);
            const int i = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(v, i, best, bi)) {
                best = v;
                bi = i;
            }
        }
        if (lane == 0) out[blockIdx.x] = bi;
    }
}

__global__ void k_argmax_finalize(unsigned long long *__restrict__ key, int B, const DecodeIO *io,
                                  int32_t *next_token, int32_t *step_ctr, int32_t *pos_inc, int32_t *status) {
    const int step = step_ctr ? *step_ctr : 0;
    int32_t *argmax_out = io ? io->argmax : nullptr;
    int32_t *hist = io ? io->hist : nullptr;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        const unsigned long long k = key[b];
        const int idx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
        const float v = float_from_order_key(static_cast<uint32_t>(k >> 32));
        if (isnan(v)) record_status(status, QW3_ERR_NONFINITE);
        if (argmax_out) argmax_out[b] = idx;
        if (next_token) next_token[b] = idx;
        if (hist) hist[static_cast<size_t>(step) * B + b] = idx;
        if (pos_inc) pos_inc[b] += 1;
        key[b] = 0ull;
    }
    __syncthreads();
    if (threadIdx.x == 0 && step_ctr) *step_ctr = step + 1;
}

template <typename KT>
__global__ void k_copy_kv_rows(const KT *__restrict__ base, size_t kvsel_stride, size_t head_stride, int pos0,
                               int n, int nkv, int hd, float *__restrict__ k_out, float *__restrict__ v_out) {
    const size_t total = static_cast<size_t>(n) * nkv * hd;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int d = static_cast<int>(i % hd);
        const int g = static_cast<int>((i / hd) % nkv);
        const int r = static_cast<int>(i / (static_cast<size_t>(hd) * nkv));
        const size_t row = static_cast<size_t>(g) * head_stride +
                           static_cast<size_t>(pos0 + r) * (kv_is_q8<KT>::value ? hd / 32 * 34 : hd);
        k_out[i] = kv_elem<0>(base + row, d);
        v_out[i] = kv_elem<0>(base + kvsel_stride + row, d);
    }
}

}  // namespace

cudaError_t configure_misc() {
    return cudaFuncSetAttribute(k_embed, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_embed(const int32_t *tokens, int n, const QMat &E, float *x, bool pdl, cudaStream_t s,
                         unsigned long long *trace) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_embed, tokens, E, E.cols, E.rows, x, trace);
}

cudaError_t launch_rmsnorm_rows(const float *x, int M, int K, const float *w, float eps, float *y, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    k_rmsnorm_rows<<<M, 256, 0, s>>>(x, K, w, eps, y);
    return cudaGetLastError();
}

template <typename KT>
cudaError_t qk_rope_append_t(float *qkv, int M, int qkv_stride, const float *q_norm, const float *k_norm, float eps,
                             const float2 *rope, const int32_t *row_seq, int seq0, const int32_t *row_pos, int pos0,
                             KT *kv_layer, size_t seq_stride, size_t kvsel_stride, size_t head_stride, int nh, int nkv,
                             int hd, cudaStream_t s) {
    const dim3 grid(M, (nh + 2 * nkv + 3) / 4);
    if (hd == 128)
        k_qk_rope_append<128, KT><<<grid, 128, 0, s>>>(qkv, M, qkv_stride, q_norm, k_norm, eps, rope, row_seq, seq0,
                                                       row_pos, pos0, kv_layer, seq_stride, kvsel_stride, head_stride,
                                                       nh, nkv);
    else if (hd == 64)
        k_qk_rope_append<64, KT><<<grid, 128, 0, s>>>(qkv, M, qkv_stride, q_norm, k_norm, eps, rope, row_seq, seq0,
                                                      row_pos, pos0, kv_layer, seq_stride, kvsel_stride, head_stride,
                                                      nh, nkv);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_qk_rope_append(float *qkv, int M, int qkv_stride, const float *q_norm, const float *k_norm,
                                  float eps, const float2 *rope, const int32_t *row_seq, int seq0,
                                  const int32_t *row_pos, int pos0, void *kv_layer, size_t seq_stride,
                                  size_t kvsel_stride, size_t head_stride, int nh, int nkv, int hd, int kvtype,
                                  cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    if (kvtype == KV_Q8)
        return qk_rope_append_t(qkv, M, qkv_stride, q_norm, k_norm, eps, rope, row_seq, seq0, row_pos, pos0,
                                static_cast<kvq8 *>(kv_layer), seq_stride, kvsel_stride, head_stride, nh, nkv, hd, s);
    if (kvtype == KV_F16)
        return qk_rope_append_t(qkv, M, qkv_stride, q_norm, k_norm, eps, rope, row_seq, seq0, row_pos, pos0,
                                static_cast<__half *>(kv_layer), seq_stride, kvsel_stride, head_stride, nh, nkv, hd, s);
    return qk_rope_append_t(qkv, M, qkv_stride, q_norm, k_norm, eps, rope, row_seq, seq0, row_pos, pos0,
                            static_cast<float *>(kv_layer), seq_stride, kvsel_stride, head_stride, nh, nkv, hd, s);
}

namespace {
__global__ void __launch_bounds__(256) k_q8act_rows(float4 *__restrict__ x, int64_t n4) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool act = i < n4;
    const float4 u = act ? x[i] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4 r = q8_0_roundtrip4(u);   // every lane of the warp takes part
    if (act) x[i] = r;
}
}  // namespace

cudaError_t launch_q8act_rows(float *x, int M, int K, cudaStream_t s) {
    if (M < 1 || K % 32) return cudaErrorInvalidValue;
    const int64_t n4 = static_cast<int64_t>(M) * K / 4;
    k_q8act_rows<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, s>>>(reinterpret_cast<float4 *>(x), n4);
    return cudaGetLastError();
}

cudaError_t launch_argmax_rows(const float *logits, int M, int V, int32_t *out, int32_t *status, cudaStream_t s) {
    if (M < 1 || V < 1) return cudaErrorInvalidValue;
    k_argmax_rows<<<M, 512, 0, s>>>(logits, V, out, status);
    return cudaGetLastError();
}

cudaError_t launch_argmax_finalize(unsigned long long *key, int B, const DecodeIO *io, int32_t *next_token,
                                   int32_t *step_ctr, int32_t *pos_inc, int32_t *status, cudaStream_t s) {
    k_argmax_finalize<<<1, 256, 0, s>>>(key, B, io, next_token, step_ctr, pos_inc, status);
    return cudaGetLastError();
}

cudaError_t launch_copy_kv_rows(const void *kv_layer_seq, size_t kvsel_stride, size_t head_stride, int pos0, int n,
                                int nkv, int hd, float *k_out, float *v_out, int kvtype, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const size_t total = static_cast<size_t>(n) * nkv * hd;
    const unsigned grid = static_cast<unsigned>(std::min<size_t>((total + 255) / 256, 4096));
    if (kvtype == KV_Q8)
        k_copy_kv_rows<<<grid, 256, 0, s>>>(static_cast<const kvq8 *>(kv_layer_seq), kvsel_stride, head_stride, pos0,
                                            n, nkv, hd, k_out, v_out);
    else if (kvtype == KV_F16)
        k_copy_kv_rows<<<grid, 256, 0, s>>>(static_cast<const __half *>(kv_layer_seq), kvsel_stride, head_stride, pos0,
                                            n, nkv, hd, k_out, v_out);
    else
        k_copy_kv_rows<<<grid, 256, 0, s>>>(static_cast<const float *>(kv_layer_seq), kvsel_stride, head_stride, pos0,
                                            n, nkv, hd, k_out, v_out);
    return cudaGetLastError();
}

}  // namespace qw3
