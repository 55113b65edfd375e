// Internal declarations of libqw3 (not part of the C ABI).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/qw3.h"

namespace qw3 {

// ---------------------------------------------------------------- weights

// A Q8_0 matrix repacked at create time into tiles of 8 rows x kt columns.
// A tile holds the 8 rows' int8 codes ([8][kt]) followed by their f16 scales
// ([8][kt/32]): 8.5 * kt bytes, the same 34 bytes per 32 weights as the GGUF
// blocks. Tiles are stored row-group-major (every k-tile of rows 0..7, then
// rows 8..15, ...) or k-tile-major (k-tile 0 of every row group, then k-tile
// 1, ...), so the slice a kernel needs is one contiguous 16-byte-aligned
// range and streams with a single bulk copy. Rows are padded to a multiple of
// 16 with zero rows.
struct QMat {
    uint8_t *base = nullptr;
    int rows = 0;         // logical rows
    int rows_pad = 0;     // allocated rows (multiple of 16)
    int cols = 0;
    int kt = 0;           // tile width: divides cols, multiple of 32
    int ktile_major = 0;  // 0: row-group-major, 1: k-tile-major
    uint8_t *ut = nullptr;  // nullable: the same weights as bf16 hi/lo tensor-core tiles
    const uint8_t *q4 = nullptr;  // Q4_K models: the raw rows (base is then null)
    uint8_t *uq = nullptr;        // nullable: the Q8_0 weights in the tensor-core GEMM's streamed layout
};

constexpr int kRowAlign = 16;

__host__ __device__ inline size_t qm_tile_bytes(int kt) { return static_cast<size_t>(kt) * 17 / 2; }

__host__ __device__ inline size_t qm_bytes(const QMat &m) {
    return static_cast<size_t>(m.rows_pad / 8) * (m.cols / m.kt) * qm_tile_bytes(m.kt);
}

__host__ __device__ inline size_t qm_tile_offset(const QMat &m, int group, int t) {
    const size_t ngroups = static_cast<size_t>(m.rows_pad / 8), ntiles = static_cast<size_t>(m.cols / m.kt);
    const size_t idx = m.ktile_major ? static_cast<size_t>(t) * ngroups + group : static_cast<size_t>(group) * ntiles + t;
    return idx * qm_tile_bytes(m.kt);
}

// Codes of row r from column k (k and the run read must stay inside one tile).
__host__ __device__ inline const int8_t *qm_codes(const QMat &m, int r, int k) {
    const int t = k / m.kt, kk = k - t * m.kt;
    return reinterpret_cast<const int8_t *>(m.base + qm_tile_offset(m, r >> 3, t)) + (r & 7) * m.kt + kk;
}

// Scale of the 32-column block of row r that holds column k.
__host__ __device__ inline const __half *qm_scale(const QMat &m, int r, int k) {
    const int t = k / m.kt, kk = k - t * m.kt;
    return reinterpret_cast<const __half *>(m.base + qm_tile_offset(m, r >> 3, t) + 8 * static_cast<size_t>(m.kt)) +
           (r & 7) * (m.kt / 32) + kk / 32;
}

struct LayerDev {
    QMat qkv;   // rows: q (n_heads*hd), k (n_kv*hd), v (n_kv*hd); cols H
    QMat o;     // [H][n_heads*hd]
    QMat gu;    // rows interleaved: 2i = gate_i, 2i+1 = up_i; cols H
    QMat down;  // [H][I]
    float *attn_norm, *q_norm, *k_norm, *ffn_norm;
};

// ------------------------------------------------------------ GEMV params

// Output pointers of a decode step, kept in device memory so that one
// captured CUDA graph serves calls with different caller buffers.
struct DecodeIO {
    float *logits;     // nullable [B][V]
    int32_t *argmax;   // nullable [B]
    int32_t *hist;     // nullable [step][B] token history
    int32_t *unused;
};

enum GemvMode : int { GEMV_STORE = 0, GEMV_RESID = 1, GEMV_SWIGLU = 2, GEMV_ARGMAX = 3 };

struct GemvArgs {
    QMat W;                   // row-group-major tiles
    int N, K;                 // logical rows, cols
    int B;                    // activation rows (1..4)
    const float *x;           // [B][K] input
    const float *norm_w;      // [K] RMSNorm weight, nullptr = no norm prologue
    float eps;
    float *y;                 // STORE: [B][N]; RESID: [B][N] += ; SWIGLU: [B][N/2]
    // ARGMAX mode
    unsigned long long *argmax_key;  // [B] packed (value, index) keys, reset to 0
    unsigned int *done_counter;      // CTA arrival counter, reset by the last CTA
    const DecodeIO *io;              // nullable: output pointers read on the device
    int32_t *argmax_out;             // used when io == nullptr (nullable) [B]
    int32_t *next_token;             // nullable [B]: written with the argmax
    int32_t *step_ctr;               // nullable: incremented by the last CTA
    int32_t *pos_inc;                // nullable [B]: +1 by the last CTA
    int32_t *status;                 // device status word
    unsigned long long *trace;       // nullable: 2 records of 8 u64 (first, last CTA)
    int act_q8;                      // 1: the (normalised) input rows go through a Q8_0 round trip
};

struct AttnDecodeArgs {
    const float *qkv;     // [B][(nh+2nkv)*hd] raw projections
    int qkv_stride;
    const float *q_norm, *k_norm;
    float eps;
    const float2 *rope;   // [max_seq_len][hd/2] (cos, sin)
    void *kv;             // this layer's cache: [seq][K|V][kv_head][capacity][head_dim]
    int kvtype;           // KvType: f32, IEEE half or q8_0 rows
    size_t seq_stride, kvsel_stride, head_stride;  // cache elements (bytes for q8_0)
    const int32_t *seq_ids;  // [B]
    const int32_t *pos;      // [B] position of the new token
    int nh, nkv, hd;
    float scale;
    float *out;              // [B][nh*hd]
    // several clusters per (b, g) (nsplit > cluster size): their partials
    // [B][nkv][clusters][G][hd+4] and arrival counters [B][nkv] (zero)
    float *cpart;
    unsigned int *ccnt;
    int32_t *status;
    unsigned long long *trace;  // nullable: 2 records of 8 u64 (first, last CTA)
};

// ---------------------------------------------------------------- helpers

#define QW3_CUDA_TRY(expr)                                   \
    do {                                                     \
        cudaError_t _e = (expr);                             \
        if (_e != cudaSuccess) return ::qw3::cuda_fail(_e, #expr, __FILE__, __LINE__); \
    } while (0)

int cuda_fail(cudaError_t e, const char *what, const char *file, int line);
void set_thread_error(const std::string &msg);
const std::string &thread_error();

int num_sms();

// Set the dynamic shared-memory limits of every kernel instantiation; called
// once per process before any launch or graph capture.
cudaError_t configure_gemv();
cudaError_t configure_attention();
cudaError_t configure_misc();

// launchers (return cudaError_t of the launch)
cudaError_t launch_quantize(const float *x, int64_t nblocks, uint8_t *out, int32_t *status, cudaStream_t s);
cudaError_t launch_dequantize(const uint8_t *blocks, int64_t nblocks, float *y, cudaStream_t s);
cudaError_t launch_repack(const uint8_t *raw, int rows, int cols, const QMat &dst,
                          int dst_row0, int dst_row_stride, cudaStream_t s);
// Raw GGUF Q8_0 GEMV (the boundary entries): y[b][r] = sum_k W[r][k] x[b][k];
// q8act: x re-quantized to Q8_0 per 32-block, integer block dots (needs
// cols % 256 == 0 and 16-byte aligned W and x).
cudaError_t launch_gemv_raw(const uint8_t *W, int rows, int cols, const float *x, int B, float *y, bool q8act,
                            cudaStream_t s);

cudaError_t launch_gemv(const GemvArgs &a, int mode, bool pdl, cudaStream_t s);
// largest B * K the decode GEMV stages (activations live in shared memory)
constexpr int kGemvMaxBK = 16384;
// nsplit splits of each (sequence, kv head) in clusters of csize CTAs
// (csize divides nsplit; nsplit / csize <= 8 clusters merge through cpart)
cudaError_t launch_attn_decode(const AttnDecodeArgs &a, int B, int nsplit, int csize, bool pdl, cudaStream_t s);
// largest split count (= cluster size) of the decode attention kernel for
// (head_dim, group) on the current device such that `units` clusters (one per
// kv head and sequence) run at once
int attn_decode_max_nsplit(int hd, int G, int units);
cudaError_t launch_embed(const int32_t *tokens, int n, const QMat &E, float *x, bool pdl, cudaStream_t s,
                         unsigned long long *trace = nullptr);

// prefill / batched path
cudaError_t launch_rmsnorm_rows(const float *x, int M, int K, const float *w, float eps, float *y,
                                cudaStream_t s);
// Workspace of the split-K tensor-core GEMM: partial tiles [split][M][N].
struct GemmSplitK {
    float *ws = nullptr;
    size_t ws_floats = 0;
};

// Dense contraction C[M][N] = A[M][K] . W[N][K]^T with the GEMV epilogue
// modes; tensor cores (tcgen05) from kGemmTcMinRows rows, CUDA cores below.
// apack: scratch for the packed activations (apack_bytes(M, K)); nullptr
// keeps the CUDA-core path. sk (nullable): lets small-M products split K.
cudaError_t launch_gemm(const float *A, int M, int K, const QMat &W, float *C, int mode,
                        unsigned long long *argmax_key, const DecodeIO *io, cudaStream_t s,
                        int32_t *status = nullptr, uint8_t *apack = nullptr, const GemmSplitK *sk = nullptr);
constexpr int kGemmTcMinRows = 32;
bool gemm_tc_supported(int M, int K, const QMat &W);
// bytes of a weight matrix packed into fp16 hi/lo UMMA tiles plus its row factors
size_t ut_bytes(int rows, int K);
// bytes of the packed activations of a GEMM with up to `rows` rows and K columns
size_t apack_bytes(int rows, int K);
cudaError_t configure_gemm_tc();
// The Q8_0 weights of W in the layout the tensor-core GEMM streams, plus the
// row factors (tq_bytes).
size_t tq_bytes(int rows, int K);
cudaError_t launch_pack_w_q8(const QMat &W, uint8_t *dst, cudaStream_t s);
// C[M][N] = A[M][K] . W[N][K]^T on the tensor cores from a raw Q8_0 matrix
// (K % 64 == 0): the weights are packed into the streamed layout and A into
// its operand tiles inside ws (gemm_q8_raw_workspace_bytes, 16-byte aligned).
size_t gemm_q8_raw_workspace_bytes(int N, int K, int M);
cudaError_t launch_gemm_q8_raw(const uint8_t *W, int N, int K, const float *A, int M, float *C, uint8_t *ws,
                               cudaStream_t s);
// The same tiles from a raw Q4_K matrix [N][K / 256 blocks].
cudaError_t launch_pack_w_q4k(const uint8_t *W, int N, int K, uint8_t *dst, cudaStream_t s);

// ---- Q4_K weights (q4k.cu; "Model files and quantization", 11.8)
size_t q4k_row_bytes(int cols);                 // cols / 256 blocks of 144 bytes
bool q4k_gemv_fits(int B, int K);               // B <= 8, K % 256 == 0, B * K <= 49152
cudaError_t configure_q4k();
cudaError_t launch_q4k_quantize(const float *x, int64_t nblocks, uint8_t *out, int32_t *status, cudaStream_t s);
cudaError_t launch_q4k_dequantize(const uint8_t *blocks, int64_t nblocks, float *y, cudaStream_t s);
cudaError_t launch_embed_q4k(const int32_t *tokens, int M, const uint8_t *E, int H, int vocab, float *x,
                             cudaStream_t s);
// y = W xn for B rows (xn = RMSNorm(x) * norm_w when norm_w is given); mode
// GEMV_STORE / GEMV_RESID / GEMV_SWIGLU (row pairs) / GEMV_ARGMAX (y nullable
// or io->logits; packed keys max'ed into key[B]).
cudaError_t launch_gemv_q4k(const uint8_t *W, int N, int K, int B, const float *x, const float *norm_w, float eps,
                            float *y, int mode, const DecodeIO *io, unsigned long long *key, bool pdl,
                            cudaStream_t s);
cudaError_t launch_gemm_tc(const float *A, int M, int K, const QMat &W, float *C, int mode,
                           unsigned long long *argmax_key, const DecodeIO *io, int32_t *status, uint8_t *apack,
                           cudaStream_t s, const GemmSplitK *sk = nullptr);
// KV cache pointers below are the byte address of the layer's (or the
// sequence's) first element; strides are in cache elements (bytes for a
// q8_0 cache); kvtype (KvType) selects f32, IEEE half or q8_0 rows.
cudaError_t launch_qk_rope_append(float *qkv, int M, int qkv_stride, const float *q_norm,
                                  const float *k_norm, float eps, const float2 *rope,
                                  const int32_t *row_seq, int seq0, const int32_t *row_pos, int pos0,
                                  void *kv_layer, size_t seq_stride, size_t kvsel_stride,
                                  size_t head_stride, int nh, int nkv, int hd, int kvtype, cudaStream_t s);
cudaError_t launch_attn_prefill(const float *qkv, int M, int qkv_stride, const void *kv_seq,
                                size_t kvsel_stride, size_t head_stride, int pos0, int nh, int nkv, int hd,
                                float scale, float *out, int kvtype, cudaStream_t s);
// Causal prefill attention on tensor cores (attn_prefill_tc.cu): packs the
// sequence's K/V of the layer into kvpack (attn_prefill_tc_pack_bytes) and
// runs one CTA per (128-query tile, head); for chunks of >= 128 rows.
constexpr int kAttnPrefillTcMinRows = 128;
size_t attn_prefill_tc_pack_bytes(int hd, int nkv, int max_seq_len);
cudaError_t configure_attn_prefill_tc();
cudaError_t launch_attn_prefill_tc(const float *qkv, int M, int qkv_stride, const void *kv_seq, size_t kvsel_stride,
                                   size_t head_stride, int pos0, int nh, int nkv, int hd, float scale, float *out,
                                   uint8_t *kvpack, int32_t *status, int kvtype, cudaStream_t s);
// In-place Q8_0 round trip (q8_0_roundtrip4) of M rows of K values (K a
// multiple of 32): the input of a linear layer in the q8_0 activation mode.
cudaError_t launch_q8act_rows(float *x, int M, int K, cudaStream_t s);
// Greedy argmax of each of M logits rows [M][V] (lowest index among equal
// maxima); a NaN records QW3_ERR_NONFINITE.
cudaError_t launch_argmax_rows(const float *logits, int M, int V, int32_t *out, int32_t *status, cudaStream_t s);
cudaError_t launch_argmax_finalize(unsigned long long *key, int B, const DecodeIO *io,
                                   int32_t *next_token, int32_t *step_ctr, int32_t *pos_inc,
                                   int32_t *status, cudaStream_t s);
cudaError_t launch_copy_kv_rows(const void *kv_layer_seq, size_t kvsel_stride, size_t head_stride,
                                int pos0, int n, int nkv, int hd, float *k_out, float *v_out, int kvtype,
                                cudaStream_t s);

}  // namespace qw3

// ------------------------------------------------------------ device PTX

#ifdef __CUDACC__
namespace qw3 {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase: gives up after ~1 s and returns false.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait with cluster-scope acquire: for phases completed by peers of
// the cluster (remote arrives, st.async bytes).
__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Asynchronous stores into a peer CTA's shared memory (shared::cluster
// addresses from dsmem_map); each completes its bytes on the peer's mbarrier.
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float a, float b, float c, float d, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar) : "memory");
}

__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
                 ::"r"(addr), "f"(a), "f"(b), "r"(bar) : "memory");
}

// 1-D bulk copy global -> shared (TMA), completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch controls (no-ops without the launch attribute).
// ---- thread-block clusters: rank, the hardware cluster barrier (every
// thread of every CTA of the cluster arrives; release/acquire order shared
// memory across the cluster), and loads from a peer CTA's shared memory.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void hw_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of the cluster barrier, for work between them.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t dsmem_map(const void *local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
    return r;
}

__device__ __forceinline__ float dsmem_ld(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- KV cache element (f32, or IEEE half for a QW3_FLAG_KV_F16 model)
__device__ __forceinline__ float kv_f32(float v) { return v; }
__device__ __forceinline__ float kv_f32(__half v) { return __half2float(v); }
template <typename KT>
__device__ __forceinline__ KT kv_cvt(float v);
template <>
__device__ __forceinline__ float kv_cvt<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half kv_cvt<__half>(float v) { return __float2half_rn(v); }

// ---- q8_0 KV cache ("The LLM stack", 13.4; "A transformer from scratch",
// 12.4): a cached (position, kv head) row of head_dim values is head_dim/32
// Q8_0 blocks (f16 scale, 32 int8 codes: 34 bytes), so a q8_0 cache is
// addressed in bytes and a row is kv_row<kvq8, HD>() of them.
struct kvq8 {
    uint8_t b;
};
enum KvType : int { KV_F32 = 0, KV_F16 = 1, KV_Q8 = 2 };
template <typename KT>
struct kv_is_q8 {
    static constexpr bool value = false;
};
template <>
struct kv_is_q8<kvq8> {
    static constexpr bool value = true;
};
// Elements of type KT in one cached row of head_dim HD.
template <typename KT, int HD>
__host__ __device__ constexpr int kv_row() { return kv_is_q8<KT>::value ? HD / 32 * 34 : HD; }
inline size_t kv_row_units(int kvtype, int hd) { return kvtype == KV_Q8 ? static_cast<size_t>(hd) / 32 * 34 : hd; }
inline size_t kv_unit_bytes(int kvtype) { return kvtype == KV_F32 ? 4 : (kvtype == KV_F16 ? 2 : 1); }

// Value d of a cached row (any element type).
template <int HD>
__device__ __forceinline__ float kv_elem(const float *row, int d) { return row[d]; }
template <int HD>
__device__ __forceinline__ float kv_elem(const __half *row, int d) { return __half2float(row[d]); }
template <int HD>
__device__ __forceinline__ float kv_elem(const kvq8 *row, int d) {
    const uint8_t *blk = &row->b + (d >> 5) * 34;
    const float sc = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(blk)));
    return sc * static_cast<float>(static_cast<int8_t>(blk[2 + (d & 31)]));
}

// ---- Q4_K block decode ("Model files and quantization", 11.8; layout in q4k.cu)
__device__ __forceinline__ float q4k_half(const uint8_t *p) {
    return __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t *>(p)));
}

// (d * sc_j, dmin * m_j) of sub-block j of a block.
__device__ __forceinline__ void q4k_sub(const uint8_t *blk, int j, float &d1, float &m1) {
    const uint8_t *s = blk + 4;
    int sc, m;
    if (j < 4) {
        sc = s[j] & 63;
        m = s[j + 4] & 63;
    } else {
        sc = (s[j + 4] & 0xF) | ((s[j - 4] >> 6) << 4);
        m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
    d1 = q4k_half(blk) * static_cast<float>(sc);
    m1 = q4k_half(blk + 2) * static_cast<float>(m);
}

// Value t (0..255) of a block.
__device__ __forceinline__ float q4k_value(const uint8_t *blk, int t) {
    float d1, m1;
    q4k_sub(blk, t >> 5, d1, m1);
    const uint8_t byte = blk[16 + 32 * (t >> 6) + (t & 31)];
    const int q = ((t >> 5) & 1) ? (byte >> 4) : (byte & 0xF);
    return fmaf(d1, static_cast<float>(q), -m1);
}


// ---- fp16 hi/lo operands of the tensor-core products
// A row (of an activation matrix, a weight matrix, a query, a key) whose
// largest magnitude is amax is multiplied by the power of two 2^t that brings
// amax into [2^14, 2^15); each scaled value x then splits exactly enough into
// fp16 parts hi = rn(x), lo = rn(x - hi) (22 significant bits, no overflow:
// fp16 holds up to 65504), and the product's f32 result is multiplied by the
// inverse powers afterwards (exact). t is clamped to [-100, 100] so that both
// 2^t and 2^-t are normal f32; amax = 0 gives t = 0.
__device__ __forceinline__ int f16_row_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;   // floor(log2 amax), normal amax
    return max(-100, min(100, 14 - e));
}
__device__ __forceinline__ float pow2_f32(int t) { return __uint_as_float(static_cast<uint32_t>(127 + t) << 23); }

// hi/lo fp16 parts of 8 (already scaled) values as two uint4, value j in
// halfword j.
__device__ __forceinline__ void split8_f16(const float (&v)[8], uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 p = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        const float2 pf = __half22float2(p);
        const __half2 r = __floats2half2_rn(v[2 * i] - pf.x, v[2 * i + 1] - pf.y);
        h[i] = *reinterpret_cast<const uint32_t *>(&p);
        l[i] = *reinterpret_cast<const uint32_t *>(&r);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Q8_0 encoding of a row spread over a warp, lane holding values
// [lane * E, lane * E + E) (E = HD / 32): 32 / E consecutive lanes hold one
// 32-value block. The 11.7 encoder: d = amax / 127, inv = d ? 1 / d : 0,
// q = clamp(round(v * inv), +-127), halves away from zero, d kept as f16.
// All 32 lanes call it.
template <int HD>
__device__ __forceinline__ void q8_encode_lanes(const float (&v)[HD / 32], int (&q)[HD / 32], __half &dh) {
    constexpr int E = HD / 32, L = 32 / E;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
    for (int o = 1; o < L; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const float inv = (d == 0.0f) ? 0.0f : __fdiv_rn(1.0f, d);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float p = __fmul_rn(v[e], inv);
        q[e] = isnan(p) ? 0 : static_cast<int>(fminf(fmaxf(roundf(p), -127.0f), 127.0f));
    }
    dh = __float2half_rn(d);
}

// Store a warp's row (lane layout as q8_encode_lanes) as Q8_0 blocks at row:
// the first lane of each block writes its f16 scale, every lane its codes
// (2-byte stores: a block's codes start 2 bytes into it). All 32 lanes call it.
template <int HD>
__device__ __forceinline__ void q8_store_lanes(kvq8 *row, const float (&v)[HD / 32], int lane) {
    constexpr int E = HD / 32, L = 32 / E;
    int q[E];
    __half dh;
    q8_encode_lanes<HD>(v, q, dh);
    uint8_t *blk = &row->b + (lane / L) * 34;
    if (lane % L == 0) *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(dh);
    uint16_t *cp = reinterpret_cast<uint16_t *>(blk + 2 + (lane % L) * E);
#pragma unroll
    for (int h = 0; h < E / 2; ++h)
        cp[h] = static_cast<uint16_t>((q[2 * h] & 0xff) | ((q[2 * h + 1] & 0xff) << 8));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Order-preserving map of f32 to u32 (larger float -> larger unsigned).
__device__ __forceinline__ uint32_t float_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_key(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// (value, index) packed so that u64 max picks the largest value and, among
// equal values, the lowest index.
__device__ __forceinline__ unsigned long long argmax_pack(float v, int idx) {
    return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(idx));
}

// Trace record of one CTA: 8 u64 words, see qw3_debug_read_trace.
constexpr int kTraceWords = 8;

__device__ __forceinline__ unsigned long long *trace_slot(unsigned long long *trace) {
    if (!trace) return nullptr;
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) return trace;
    if (blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1)
        return trace + kTraceWords;
    return nullptr;
}

__device__ __forceinline__ uint32_t smid() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void record_status(int32_t *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---- activation digit planes (decode GEMVs)
//
// A GEMV input vector enters the decode GEMVs as three int8 digit planes per
// 32-value block: x = s * (h + m / 254 + l / 254^2) with s = max|x| / 127 and
// |h|, |m|, |l| <= 127, which represents x to within s / (2 * 254^2), about
// 6e-8 of the block's largest value (the size of an f32 rounding). The dot
// of 16 int8 codes with 16 such values is then 12 exact int8 dot products
// (dp4a) and one f32 combination. Layout: plane q of values [16c, 16c + 16)
// is the uint4 at planes[3c + q]; s of values [32b, 32b + 32) is scales[b].

// Digit planes of v (|v| <= 127 s), packed one byte per value.
__device__ __forceinline__ void digit_planes(float v, float inv_s, int &h, int &m, int &l) {
    const float t = v * inv_s;
    const float th = rintf(t);
    const float r1 = (t - th) * 254.0f;
    const float tm = rintf(r1);
    const float r2 = (r1 - tm) * 254.0f;
    h = static_cast<int>(fminf(fmaxf(th, -127.0f), 127.0f));
    m = static_cast<int>(fminf(fmaxf(tm, -127.0f), 127.0f));
    l = static_cast<int>(fminf(fmaxf(rintf(r2), -127.0f), 127.0f));
}

// Digit planes of four values at once, packed one byte per value into the
// three plane words (value j in byte j). inv_s = 1 / s with s >= max|v| / 127
// (any such s: the digits represent v / s). Rounding to nearest by the 1.5 *
// 2^23 shift, exact for |t| < 2^22; every digit lies in [-127, 127] because
// |t| <= 127 (1 + 2^-23) and each residual is at most 0.5 * 254.
__device__ __forceinline__ void digit_planes4(const float (&v)[4], float inv_s, uint32_t &ph, uint32_t &pm,
                                              uint32_t &pl) {
    constexpr float kShift = 12582912.0f;   // 1.5 * 2^23
    uint32_t bh[4], bm[4], bl[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float t = v[j] * inv_s;
        const float sh = __fadd_rn(t, kShift);
        const float r1 = __fmul_rn(__fsub_rn(t, __fsub_rn(sh, kShift)), 254.0f);
        const float sm = __fadd_rn(r1, kShift);
        const float r2 = __fmul_rn(__fsub_rn(r1, __fsub_rn(sm, kShift)), 254.0f);
        const float sl = __fadd_rn(r2, kShift);
        bh[j] = __float_as_uint(sh);
        bm[j] = __float_as_uint(sm);
        bl[j] = __float_as_uint(sl);
    }
    // the low byte of each shifted float is the digit in two's complement
    ph = __byte_perm(__byte_perm(bh[0], bh[1], 0x0040), __byte_perm(bh[2], bh[3], 0x0040), 0x5410);
    pm = __byte_perm(__byte_perm(bm[0], bm[1], 0x0040), __byte_perm(bm[2], bm[3], 0x0040), 0x5410);
    pl = __byte_perm(__byte_perm(bl[0], bl[1], 0x0040), __byte_perm(bl[2], bl[3], 0x0040), 0x5410);
}

__device__ __forceinline__ uint32_t pack4_s8(int a, int b, int c, int d) {
    return (static_cast<uint32_t>(a) & 0xffu) | ((static_cast<uint32_t>(b) & 0xffu) << 8) |
           ((static_cast<uint32_t>(c) & 0xffu) << 16) | ((static_cast<uint32_t>(d) & 0xffu) << 24);
}

// Q8_0 round trip of activations ("Model files and quantization": the 11.7
// encoder applied per row per call, 11.9): 8 consecutive lanes hold one
// 32-value block, 4 values each; every value becomes f32(f16(d)) * q, the
// value the integer block dot multiplies (d = amax / 127, q = the encoder's
// code). A dot over these values is the pages' sum of d_w * d_a * i32 dots up
// to f32 rounding. All 32 lanes of the warp call it; a NaN stays NaN and an
// infinity turns its block into NaN.
__device__ __forceinline__ float4 q8_0_roundtrip4(float4 u) {
    float amax = fmaxf(fmaxf(fabsf(u.x), fabsf(u.y)), fmaxf(fabsf(u.z), fabsf(u.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float d = __fdiv_rn(amax, 127.0f);
    const float inv = (d == 0.0f) ? 0.0f : __fdiv_rn(1.0f, d);
    const float dq = __half2float(__float2half_rn(d));
    auto rt = [&](float v) {
        if (isnan(v)) return v;
        const float p = __fmul_rn(v, inv);
        const float q = isnan(p) ? 0.0f : fminf(fmaxf(roundf(p), -127.0f), 127.0f);
        return dq * q;
    };
    return make_float4(rt(u.x), rt(u.y), rt(u.z), rt(u.w));
}

// sum over 16 codes w of q * (h + m / 254 + l / 254^2), planes P[0..2]
__device__ __forceinline__ float pdot16(const uint4 w, const uint4 *P) {
    int a = __dp4a(static_cast<int>(w.x), static_cast<int>(P[0].x), 0);
    a = __dp4a(static_cast<int>(w.y), static_cast<int>(P[0].y), a);
    a = __dp4a(static_cast<int>(w.z), static_cast<int>(P[0].z), a);
    a = __dp4a(static_cast<int>(w.w), static_cast<int>(P[0].w), a);
    int b = __dp4a(static_cast<int>(w.x), static_cast<int>(P[1].x), 0);
    b = __dp4a(static_cast<int>(w.y), static_cast<int>(P[1].y), b);
    b = __dp4a(static_cast<int>(w.z), static_cast<int>(P[1].z), b);
    b = __dp4a(static_cast<int>(w.w), static_cast<int>(P[1].w), b);
    int c = __dp4a(static_cast<int>(w.x), static_cast<int>(P[2].x), 0);
    c = __dp4a(static_cast<int>(w.y), static_cast<int>(P[2].y), c);
    c = __dp4a(static_cast<int>(w.z), static_cast<int>(P[2].z), c);
    c = __dp4a(static_cast<int>(w.w), static_cast<int>(P[2].w), c);
    return fmaf(static_cast<float>(c), 1.0f / 64516.0f, fmaf(static_cast<float>(b), 1.0f / 254.0f, static_cast<float>(a)));
}

}  // namespace qw3
#endif
