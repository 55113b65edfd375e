// Host side of libqw3: the C ABI declared in include/qw3.h.
//
// The forward pass follows "A transformer from scratch" (Fucina course
// ch. 12), sections 12.3-12.6, with the Qwen3 deltas of minfer's "Qwen3
// Support Plan (dense)", section 2: embedding gather, per layer
// [RMSNorm -> QKV -> per-head Q/K RMSNorm -> NeoX RoPE -> KV append -> causal
// GQA -> o_proj + residual -> RMSNorm -> gate/up -> SwiGLU -> down + residual],
// final RMSNorm, lm_head on the last row, greedy argmax.
//
// Decode (B <= 4 rows): one GEMV kernel per projection with fused norm
// prologues and residual/SwiGLU/argmax epilogues, one split-K attention kernel
// per layer; the step is captured once per B as a CUDA graph whose kernels
// are chained with programmatic dependent launch. Larger batches and prefill
// use the tiled GEMM path.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "qw3_internal.cuh"
#include "decode_step.cuh"

namespace qw3 {

namespace {
thread_local std::string g_err;
}

void set_thread_error(const std::string &msg) { g_err = msg; }
const std::string &thread_error() { return g_err; }

int cuda_fail(cudaError_t e, const char *what, const char *file, int line) {
    char buf[512];
    snprintf(buf, sizeof buf, "%s failed: %s (%s:%d)", what, cudaGetErrorString(e), file, line);
    set_thread_error(buf);
    if (e == cudaErrorMemoryAllocation) return QW3_ERR_OOM;
    return QW3_ERR_CUDA;
}

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

namespace {

std::once_flag g_cfg_once;
cudaError_t g_cfg_err = cudaSuccess;

cudaError_t configure_all() {
    std::call_once(g_cfg_once, [] {
        cudaError_t e = configure_gemv();
        if (e == cudaSuccess) e = configure_attention();
        if (e == cudaSuccess) e = configure_misc();
        if (e == cudaSuccess) e = configure_step();
        if (e == cudaSuccess) e = configure_gemm_tc();
        if (e == cudaSuccess) e = configure_q4k();
        if (e == cudaSuccess) e = configure_attn_prefill_tc();
        g_cfg_err = e;
    });
    return g_cfg_err;
}

// Device allocations go through here so that tests can make the n-th one
// fail (QW3_FAULT_ALLOC_AT=n) and check that create cleans up.
int g_alloc_count = 0;
int g_alloc_fail_at = -1;

cudaError_t dev_alloc(void **p, size_t bytes) {
    ++g_alloc_count;
    if (g_alloc_fail_at > 0 && g_alloc_count == g_alloc_fail_at) {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

}  // namespace qw3

using namespace qw3;

struct qw3_model {
    qw3_config cfg{};
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    cudaStream_t cap_stream = nullptr;
    std::string err;

    std::vector<void *> allocs;

    std::vector<LayerDev> layers;
    QMat embd, out;
    float *out_norm = nullptr;
    float2 *rope = nullptr;

    void *kv = nullptr;    // f32, IEEE half or q8_0 rows (kvtype)
    int kvtype = KV_F32;
    bool act_q8 = false;   // linear inputs through a Q8_0 round trip
    bool q4k = false;      // Q4_K weights: raw rows per matrix (QMat::q4), tensor-core tiles, no Q8_0 tiles
    uint8_t *emb4 = nullptr, *out4 = nullptr;
    size_t head_stride = 0, kvsel_stride = 0, seq_stride = 0, layer_stride = 0;
    std::vector<int32_t> seq_len;

    // decode scratch
    int qkv_w = 0;
    float *x = nullptr, *h = nullptr, *qkv = nullptr, *o = nullptr, *act = nullptr;
    unsigned int *done_counter = nullptr;
    unsigned long long *argmax_key = nullptr;
    int32_t *d_tok = nullptr, *d_pos = nullptr, *d_seq = nullptr, *d_step = nullptr, *d_status = nullptr;
    DecodeIO *d_io = nullptr;
    int attn_max_split = 8;   // largest decode-attention cluster (splits per kv head)
    int attn_long_c = 0;      // cluster size of the batch-1 long-context split (0: none)
    float *attn_cpart = nullptr;          // cluster partials of the long-context split
    unsigned int *attn_ccnt = nullptr;    // their arrival counters

    // prefill scratch
    float *px = nullptr, *ph = nullptr, *pqkv = nullptr, *po = nullptr, *pact = nullptr;
    uint8_t *apack = nullptr;   // tensor-core GEMM input, packed (nullptr: CUDA-core GEMM only)
    uint8_t *kvpack = nullptr;  // K/V operand tiles of the tensor-core prefill attention (nullptr: CUDA cores)
    GemmSplitK gsk;             // split-K workspace of the small-M tensor-core GEMMs

    std::map<int, cudaGraphExec_t> graphs;

    // QW3_FLAG_TRACE: per-kernel timestamp records of the latest decode step
    unsigned long long *trace = nullptr;
    int trace_kernels = 0;

    // persistent batch-1 decode-step kernel (decode_step.cu)
    bool step = false;
    StepParams sp{};
    int step_trace_words = 0;
};

namespace {
// Address of (layer, seq)'s block of the KV cache.
void *kv_at(const qw3_model *m, int layer, int seq) {
    const size_t e = static_cast<size_t>(layer) * m->layer_stride + static_cast<size_t>(seq) * m->seq_stride;
    return static_cast<uint8_t *>(m->kv) + e * kv_unit_bytes(m->kvtype);
}

// A linear layer through the GEMM; in the q8_0 activation mode its input
// rows (a scratch buffer no later step reads) first take their Q8_0 round
// trip.
cudaError_t lin_gemm(qw3_model *m, float *A, int M, int K, const QMat &W, float *C, GemvMode mode,
                     unsigned long long *argmax_key, const DecodeIO *io, cudaStream_t s) {
    if (m->act_q8)
        if (cudaError_t e = launch_q8act_rows(A, M, K, s); e != cudaSuccess) return e;
    return launch_gemm(A, M, K, W, C, mode, argmax_key, io, s, m->d_status, m->apack, &m->gsk);
}
}  // namespace

namespace {

int fail(qw3_model *m, int code, const std::string &msg) {
    if (m) m->err = msg;
    set_thread_error(msg);
    return code;
}

int cuda_err(qw3_model *m, cudaError_t e, const char *what) {
    const int code = (e == cudaErrorMemoryAllocation) ? QW3_ERR_OOM : QW3_ERR_CUDA;
    return fail(m, code, std::string(what) + ": " + cudaGetErrorString(e));
}

#define M_TRY(m, expr)                                        \
    do {                                                      \
        cudaError_t _e = (expr);                              \
        if (_e != cudaSuccess) return cuda_err((m), _e, #expr); \
    } while (0)

cudaError_t model_alloc(qw3_model *m, void **p, size_t bytes) {
    cudaError_t e = dev_alloc(p, bytes < 256 ? 256 : bytes);
    if (e == cudaSuccess) m->allocs.push_back(*p);
    return e;
}

void free_all(qw3_model *m) {
    for (auto &kv : m->graphs) cudaGraphExecDestroy(kv.second);
    m->graphs.clear();
    for (void *p : m->allocs) cudaFree(p);
    m->allocs.clear();
    if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
    m->cap_stream = nullptr;
    if (m->own_stream && m->stream) cudaStreamDestroy(m->stream);
    m->stream = nullptr;
}

// Tile width of the repacked layout: the whole row up to 3072 columns; wider
// rows are cut into the widest tiles of at most 2048 columns (a multiple of
// 256 that divides the row; 17 KB tiles), so that the decode GEMV's
// shared-memory ring holds two stages or more at two CTAs per SM.
int tile_width(int cols) {
    if (cols <= 3072) return cols;
    for (int kt = 2048; kt >= 256; kt -= 256)
        if (cols % kt == 0) return kt;
    int kt = cols;
    while (kt > 2048 && kt % 2 == 0 && (kt / 2) % 32 == 0) kt /= 2;
    return kt;
}

QMat qmat_shape(int rows, int cols, int kt = 0, int ktile_major = 0) {
    QMat q;
    q.rows = rows;
    q.cols = cols;
    q.rows_pad = static_cast<int>(align_up(static_cast<size_t>(rows), kRowAlign));
    q.kt = kt ? kt : tile_width(cols);
    q.ktile_major = ktile_major;
    return q;
}

size_t qmat_bytes(int rows, int cols) { return align_up(qm_bytes(qmat_shape(rows, cols)), 256); }

void qmat_place(QMat &q, uint8_t *&cursor, int rows, int cols) {
    q = qmat_shape(rows, cols);
    q.base = cursor;
    cursor += align_up(qm_bytes(q), 256);
}

// Copy (if on the host) and repack one raw Q8_0 matrix into rows
// dst_row0 + r * dst_stride of q.
int repack_into(qw3_model *m, const QMat &q, const void *raw, int rows, int cols, int dst_row0, int dst_stride,
                bool on_device, uint8_t *staging) {
    if (!raw) return fail(m, QW3_ERR_INVALID_ARG, "null weight pointer");
    if (on_device && (reinterpret_cast<uintptr_t>(raw) & 1u))
        return fail(m, QW3_ERR_INVALID_ARG, "Q8_0 blocks must be 2-byte aligned");
    const size_t bytes = static_cast<size_t>(rows) * (cols / 32) * 34;
    const uint8_t *src = static_cast<const uint8_t *>(raw);
    if (!on_device) {
        M_TRY(m, cudaMemcpyAsync(staging, raw, bytes, cudaMemcpyHostToDevice, m->stream));
        src = staging;
    }
    M_TRY(m, launch_repack(src, rows, cols, q, dst_row0, dst_stride, m->stream));
    if (!on_device) M_TRY(m, cudaStreamSynchronize(m->stream));
    return QW3_OK;
}

// Device address of a raw Q8_0 matrix: the caller's buffer, or a copy in the
// staging buffer (synchronous) when the weights are in host memory.
int raw_on_device(qw3_model *m, const void *raw, int rows, int cols, bool on_device, uint8_t *staging,
                  const uint8_t **out) {
    if (!raw) return fail(m, QW3_ERR_INVALID_ARG, "null weight pointer");
    if (on_device) {
        if (reinterpret_cast<uintptr_t>(raw) & 1u) return fail(m, QW3_ERR_INVALID_ARG, "Q8_0 blocks must be 2-byte aligned");
        *out = static_cast<const uint8_t *>(raw);
        return QW3_OK;
    }
    const size_t bytes = static_cast<size_t>(rows) * (cols / 32) * 34;
    M_TRY(m, cudaStreamSynchronize(m->stream));
    M_TRY(m, cudaMemcpyAsync(staging, raw, bytes, cudaMemcpyHostToDevice, m->stream));
    *out = staging;
    return QW3_OK;
}

int copy_f32(qw3_model *m, float *dst, const float *src, size_t n, bool on_device) {
    if (!src) return fail(m, QW3_ERR_INVALID_ARG, "null norm weight pointer");
    M_TRY(m, cudaMemcpyAsync(dst, src, n * 4, on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice,
                             m->stream));
    if (!on_device) M_TRY(m, cudaStreamSynchronize(m->stream));
    return QW3_OK;
}

int validate_config(const qw3_config *c, std::string &why) {
    auto bad = [&](const char *w) { why = w; return QW3_ERR_SHAPE; };
    if (c->vocab <= 0 || c->hidden <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 ||
        c->head_dim <= 0 || c->intermediate <= 0)
        return bad("every config size must be positive");
    if (c->hidden % 32) return bad("hidden must be a multiple of 32");
    if (c->intermediate % 32) return bad("intermediate must be a multiple of 32");
    if ((c->n_heads * c->head_dim) % 32) return bad("n_heads*head_dim must be a multiple of 32");
    if (c->n_heads % c->n_kv_heads) return bad("n_heads must be a multiple of n_kv_heads");
    if (c->n_kv_heads > 64) return bad("n_kv_heads must be at most 64");
    if (c->head_dim % 2) return bad("head_dim must be even");
    if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
    const int group = c->n_heads / c->n_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return bad("n_heads/n_kv_heads must be 1, 2, 4 or 8");
    if (c->max_seqs <= 0 || c->max_seq_len <= 0 || c->max_prefill <= 0)
        return bad("max_seqs, max_seq_len and max_prefill must be positive");
    if (!(c->rms_eps >= 0.0f) || !(c->rope_theta > 0.0f)) return bad("rms_eps must be >= 0 and rope_theta > 0");
    if (c->hidden > 16384 || c->intermediate > 65536) return bad("hidden or intermediate too large");
    if ((c->flags & QW3_FLAG_KV_F16) && (c->flags & QW3_FLAG_KV_Q8)) return bad("one KV cache type at most");
    if (c->flags & QW3_FLAG_WEIGHTS_Q4_K) {
        if (c->hidden % 256 || c->intermediate % 256 || (c->n_heads * c->head_dim) % 256)
            return bad("Q4_K weights need hidden, intermediate and n_heads*head_dim multiples of 256");
        if (c->flags & QW3_FLAG_ACT_Q8) return bad("the Q8_0 activation mode takes Q8_0 weights");
    }
    return QW3_OK;
}

int pick_nsplit(int B, int nkv, int cap) {
    const int sms = num_sms();
    const int units = B * nkv;
    int ns = units >= sms ? (4 * sms + units - 1) / units : (sms + units - 1) / units;
    if (ns > cap) ns = cap;
    if (ns < 1) ns = 1;
    return ns;
}

// The decode GEMV path stages B activation rows of up to max(H, I, n_heads*hd)
// floats in shared memory; larger batches use the tiled GEMM path.
// Batch-1 decode at contexts of this capacity or more splits each kv head's
// positions over kAttnLongClusters clusters.
constexpr int kAttnLongCtx = 4096;
constexpr int kAttnLongClusters = 4;

bool use_gemv(const qw3_config &c, int B) {
    const int kmax = std::max(c.hidden, std::max(c.intermediate, c.n_heads * c.head_dim));
    if (c.flags & QW3_FLAG_WEIGHTS_Q4_K) return q4k_gemv_fits(B, kmax);
    return B <= 4 && B * kmax <= kGemvMaxBK;
}

// Attention arguments of layer l for the decode step.
AttnDecodeArgs attn_args(qw3_model *m, int l) {
    const qw3_config &c = m->cfg;
    const LayerDev &L = m->layers[l];
    AttnDecodeArgs at{};
    at.qkv = m->qkv; at.qkv_stride = m->qkv_w; at.q_norm = L.q_norm; at.k_norm = L.k_norm; at.eps = c.rms_eps;
    at.rope = m->rope; at.kv = kv_at(m, l, 0); at.kvtype = m->kvtype;
    at.seq_stride = m->seq_stride; at.kvsel_stride = m->kvsel_stride; at.head_stride = m->head_stride;
    at.seq_ids = m->d_seq; at.pos = m->d_pos; at.nh = c.n_heads; at.nkv = c.n_kv_heads; at.hd = c.head_dim;
    at.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.head_dim)));
    at.out = m->o; at.status = m->d_status; at.cpart = m->attn_cpart; at.ccnt = m->attn_ccnt;
    return at;
}

// One decode step of a Q4_K model for B rows the Q4_K GEMV takes: every
// projection streams the raw Q4_K rows (norms fused as prologues, SwiGLU over
// the interleaved gate/up pairs), the lm_head keeps packed argmax keys that
// k_argmax_finalize turns into tokens.
int enqueue_decode_q4k(qw3_model *m, int B, int nsplit, int csize, cudaStream_t s) {
    const qw3_config &c = m->cfg;
    const int H = c.hidden, I = c.intermediate, qw = c.n_heads * c.head_dim;
    const float eps = c.rms_eps;
    // programmatic dependent launch measured slower here (1360 against 1300
    // us per 0.6B token): a waiting GEMV's shared memory crowds the running one
    const bool pdl = false;
    M_TRY(m, launch_embed_q4k(m->d_tok, B, m->emb4, H, c.vocab, m->x, s));
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerDev &L = m->layers[l];
        M_TRY(m, launch_gemv_q4k(L.qkv.q4, m->qkv_w, H, B, m->x, L.attn_norm, eps, m->qkv, GEMV_STORE, nullptr,
                                 nullptr, pdl, s));
        M_TRY(m, launch_attn_decode(attn_args(m, l), B, nsplit, csize, pdl, s));
        M_TRY(m, launch_gemv_q4k(L.o.q4, H, qw, B, m->o, nullptr, eps, m->x, GEMV_RESID, nullptr, nullptr, pdl, s));
        M_TRY(m, launch_gemv_q4k(L.gu.q4, 2 * I, H, B, m->x, L.ffn_norm, eps, m->act, GEMV_SWIGLU, nullptr, nullptr,
                                 pdl, s));
        M_TRY(m, launch_gemv_q4k(L.down.q4, H, I, B, m->act, nullptr, eps, m->x, GEMV_RESID, nullptr, nullptr, pdl,
                                 s));
    }
    M_TRY(m, launch_gemv_q4k(m->out4, c.vocab, H, B, m->x, m->out_norm, eps, nullptr, GEMV_ARGMAX, m->d_io,
                             m->argmax_key, pdl, s));
    M_TRY(m, launch_argmax_finalize(m->argmax_key, B, m->d_io, m->d_tok, m->d_step, m->d_pos, m->d_status, s));
    return QW3_OK;
}

// Enqueue one decode step for B rows on stream s: inputs d_tok/d_seq/d_pos,
// outputs through d_io; afterwards d_tok holds the argmax and d_pos moved by 1.
int enqueue_decode(qw3_model *m, int B, cudaStream_t s) {
    const qw3_config &c = m->cfg;
    const bool pdl = !(c.flags & QW3_FLAG_NO_PDL);
    const int H = c.hidden, hd = c.head_dim, nh = c.n_heads, nkv = c.n_kv_heads, I = c.intermediate;
    const int qw = nh * hd;
    int nsplit = pick_nsplit(B, nkv, m->attn_max_split), csize = nsplit;
    if (B == 1 && m->attn_long_c > 0) {
        // long contexts at batch 1: kAttnLongClusters clusters per kv head,
        // merged in global memory (more CTAs stream the cache than one
        // cluster holds)
        csize = m->attn_long_c;
        nsplit = csize * kAttnLongClusters;
    }
    const bool gv = use_gemv(c, B);
    if (m->q4k && gv) return enqueue_decode_q4k(m, B, nsplit, csize, s);
    int kidx = 0;
    auto tr = [&]() -> unsigned long long * {
        if (!m->trace) return nullptr;
        const int i = kidx++;
        return i < m->trace_kernels ? m->trace + static_cast<size_t>(i) * 2 * kTraceWords : nullptr;
    };
    if (m->q4k) M_TRY(m, launch_embed_q4k(m->d_tok, B, m->emb4, H, c.vocab, m->x, s));
    else M_TRY(m, launch_embed(m->d_tok, B, m->embd, m->x, pdl && gv, s, tr()));
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerDev &L = m->layers[l];
        if (gv) {
            GemvArgs a{};
            a.act_q8 = m->act_q8;
            a.W = L.qkv; a.N = L.qkv.rows; a.K = H; a.B = B;
            a.x = m->x; a.norm_w = L.attn_norm; a.eps = c.rms_eps; a.y = m->qkv; a.status = m->d_status;
            a.trace = tr();
            M_TRY(m, launch_gemv(a, GEMV_STORE, pdl, s));
        } else {
            M_TRY(m, launch_rmsnorm_rows(m->x, B, H, L.attn_norm, c.rms_eps, m->h, s));
            M_TRY(m, lin_gemm(m, m->h, B, H, L.qkv, m->qkv, GEMV_STORE, nullptr, nullptr, s));
        }
        AttnDecodeArgs at{};
        at.qkv = m->qkv; at.qkv_stride = m->qkv_w; at.q_norm = L.q_norm; at.k_norm = L.k_norm; at.eps = c.rms_eps;
        at.rope = m->rope; at.kv = kv_at(m, l, 0); at.kvtype = m->kvtype;
        at.seq_stride = m->seq_stride; at.kvsel_stride = m->kvsel_stride; at.head_stride = m->head_stride;
        at.seq_ids = m->d_seq; at.pos = m->d_pos; at.nh = nh; at.nkv = nkv; at.hd = hd;
        at.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(hd)));
        at.out = m->o; at.status = m->d_status; at.cpart = m->attn_cpart; at.ccnt = m->attn_ccnt;
        at.trace = tr();
        M_TRY(m, launch_attn_decode(at, B, nsplit, csize, pdl && gv, s));
        if (gv) {
            GemvArgs a{};
            a.act_q8 = m->act_q8;
            a.W = L.o; a.N = H; a.K = qw; a.B = B; a.x = m->o; a.norm_w = nullptr;
            a.eps = c.rms_eps; a.y = m->x; a.status = m->d_status;
            a.trace = tr();
            M_TRY(m, launch_gemv(a, GEMV_RESID, pdl, s));
            GemvArgs g{};
            g.act_q8 = m->act_q8;
            g.W = L.gu; g.N = 2 * I; g.K = H; g.B = B; g.x = m->x; g.norm_w = L.ffn_norm;
            g.eps = c.rms_eps; g.y = m->act; g.status = m->d_status;
            g.trace = tr();
            M_TRY(m, launch_gemv(g, GEMV_SWIGLU, pdl, s));
            GemvArgs dn{};
            dn.act_q8 = m->act_q8;
            dn.W = L.down; dn.N = H; dn.K = I; dn.B = B; dn.x = m->act; dn.norm_w = nullptr;
            dn.eps = c.rms_eps; dn.y = m->x; dn.status = m->d_status;
            dn.trace = tr();
            M_TRY(m, launch_gemv(dn, GEMV_RESID, pdl, s));
        } else {
            M_TRY(m, lin_gemm(m, m->o, B, qw, L.o, m->x, GEMV_RESID, nullptr, nullptr, s));
            M_TRY(m, launch_rmsnorm_rows(m->x, B, H, L.ffn_norm, c.rms_eps, m->h, s));
            M_TRY(m, lin_gemm(m, m->h, B, H, L.gu, m->act, GEMV_SWIGLU, nullptr, nullptr, s));
            M_TRY(m, lin_gemm(m, m->act, B, I, L.down, m->x, GEMV_RESID, nullptr, nullptr, s));
        }
    }
    if (gv) {
        GemvArgs a{};
            a.act_q8 = m->act_q8;
        a.W = m->out; a.N = c.vocab; a.K = H; a.B = B; a.x = m->x; a.norm_w = m->out_norm;
        a.eps = c.rms_eps; a.y = nullptr; a.argmax_key = m->argmax_key; a.done_counter = m->done_counter;
        a.io = m->d_io; a.next_token = m->d_tok; a.step_ctr = m->d_step; a.pos_inc = m->d_pos;
        a.status = m->d_status;
        a.trace = tr();
        M_TRY(m, launch_gemv(a, GEMV_ARGMAX, pdl, s));
    } else {
        M_TRY(m, launch_rmsnorm_rows(m->x, B, H, m->out_norm, c.rms_eps, m->h, s));
        M_TRY(m, lin_gemm(m, m->h, B, H, m->out, nullptr, GEMV_ARGMAX, m->argmax_key, m->d_io, s));
        M_TRY(m, launch_argmax_finalize(m->argmax_key, B, m->d_io, m->d_tok, m->d_step, m->d_pos, m->d_status, s));
    }
    return QW3_OK;
}

// Launch one decode step: replay the captured graph for B, capturing it on
// first use, or enqueue the kernels directly when graphs are disabled.
int run_decode_step(qw3_model *m, int B) {
    if (m->cfg.flags & QW3_FLAG_NO_GRAPH) return enqueue_decode(m, B, m->stream);
    auto it = m->graphs.find(B);
    if (it == m->graphs.end()) {
        M_TRY(m, cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
        const int rc = enqueue_decode(m, B, m->cap_stream);
        cudaGraph_t g = nullptr;
        const cudaError_t e = cudaStreamEndCapture(m->cap_stream, &g);
        if (rc != QW3_OK) {
            if (g) cudaGraphDestroy(g);
            return rc;
        }
        if (e != cudaSuccess) return cuda_err(m, e, "cudaStreamEndCapture");
        cudaGraphExec_t ex = nullptr;
        const cudaError_t e2 = cudaGraphInstantiate(&ex, g, 0);
        cudaGraphDestroy(g);
        if (e2 != cudaSuccess) return cuda_err(m, e2, "cudaGraphInstantiate");
        it = m->graphs.emplace(B, ex).first;
    }
    M_TRY(m, cudaGraphLaunch(it->second, m->stream));
    return QW3_OK;
}

// ---- tensor-core GEMM (prefill, batches from kGemmTcMinRows rows): every
// layer matrix (and the lm_head when batches that large are possible) gets a
// copy in the layout the tensor-core GEMM reads: Q8_0 pieces streamed as they
// are (1.0625 bytes per weight), Q4_K decoded into fp16 hi/lo tiles (4 bytes
// per weight); each with its power-of-two row factors.
int setup_tensor_core_gemm(qw3_model *m) {
    const qw3_config &c = m->cfg;
    // a Q4_K model's prefill and batches past the GEMV's rows run here at any size
    const bool prefill_tc = c.max_prefill >= kGemmTcMinRows || m->q4k;
    const bool batch_tc = c.max_seqs >= kGemmTcMinRows || m->q4k;
    if (!prefill_tc && !batch_tc) return QW3_OK;
    const int H = c.hidden, qw = c.n_heads * c.head_dim, I = c.intermediate;
    if (H % 64 || qw % 64 || I % 64) return QW3_OK;
    auto pack = [&](QMat &q) -> int {
        uint8_t *p = nullptr;
        if (q.q4) {
            // Q4_K: fp16 hi/lo tiles (4 bytes per weight) and row factors
            M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&p), ut_bytes(q.rows, q.cols)));
            M_TRY(m, launch_pack_w_q4k(q.q4, q.rows, q.cols, p, m->stream));
            q.ut = p;
        } else {
            // Q8_0: the codes and scales in the streamed layout (1.0625 bytes per weight)
            M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&p), tq_bytes(q.rows, q.cols)));
            M_TRY(m, launch_pack_w_q8(q, p, m->stream));
            q.uq = p;
        }
        return QW3_OK;
    };
    for (int l = 0; l < c.n_layers; ++l) {
        LayerDev &L = m->layers[l];
        if (int rc = pack(L.qkv)) return rc;
        if (int rc = pack(L.o)) return rc;
        if (int rc = pack(L.gu)) return rc;
        if (int rc = pack(L.down)) return rc;
    }
    if (batch_tc) {
        if (int rc = pack(m->out)) return rc;
        if (c.tied_lm_head) {
            m->embd.ut = m->out.ut;
            m->embd.uq = m->out.uq;
        }
    }
    const int rows = std::max(c.max_prefill, c.max_seqs);
    const int kmax = std::max(H, std::max(qw, I));
    M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&m->apack), apack_bytes(rows, kmax)));
    // split-K partials of products with few output tiles (batched decode, short prefill chunks)
    m->gsk.ws_floats = static_cast<size_t>(4) << 20;
    M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&m->gsk.ws), m->gsk.ws_floats * 4));
    M_TRY(m, cudaStreamSynchronize(m->stream));
    return QW3_OK;
}

// ---- persistent batch-1 decode-step kernel: buffers and plan

// Set up the step kernel unless the model opts out or its shape is not
// covered; the per-kernel path then serves batch 1 too.
int setup_step(qw3_model *m) {
    const qw3_config &c = m->cfg;
    if ((c.flags & QW3_FLAG_PER_KERNEL) || m->kvtype != KV_F32 || m->act_q8 || m->q4k || !step_supported(c))
        return QW3_OK;
    // The step kernel wins where a layer is latency-bound (a few hundred KB
    // of weights per SM); past that a layer is bandwidth-bound and the
    // per-kernel chain, with two streaming CTAs per SM, moves it faster
    // (measured at the 8B geometry: 295 vs 402 tok/s).
    {
        const size_t layer_bytes = qm_bytes(m->layers[0].qkv) + qm_bytes(m->layers[0].o) + qm_bytes(m->layers[0].gu) +
                                   qm_bytes(m->layers[0].down);
        if (layer_bytes / static_cast<size_t>(num_sms()) > kStepMaxLayerBytesPerSm) return QW3_OK;
    }
    StepParams P{};
    P.L = c.n_layers;
    P.H = c.hidden;
    P.I = c.intermediate;
    P.V = c.vocab;
    P.nh = c.n_heads;
    P.nkv = c.n_kv_heads;
    P.hd = c.head_dim;
    P.G = c.n_heads / c.n_kv_heads;
    P.qkv_w = m->qkv_w;
    P.eps = c.rms_eps;
    P.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(c.head_dim)));
    P.embd = m->embd;
    P.out = m->out;
    P.out_norm = m->out_norm;
    // the kernel finds layer l's weights and norms at a fixed stride from layer 0's
    const size_t lstride = c.n_layers > 1 ? static_cast<size_t>(m->layers[1].qkv.base - m->layers[0].qkv.base) : 0;
    for (int l = 0; l < c.n_layers; ++l) {
        const LayerDev &L = m->layers[l], &L0 = m->layers[0];
        const size_t d = static_cast<size_t>(l) * lstride;
        auto same = [&](const void *a, const void *b) {
            return reinterpret_cast<uintptr_t>(a) == reinterpret_cast<uintptr_t>(b) + d;
        };
        if (!same(L.qkv.base, L0.qkv.base) || !same(L.o.base, L0.o.base) || !same(L.gu.base, L0.gu.base) ||
            !same(L.down.base, L0.down.base) || !same(L.attn_norm, L0.attn_norm) || !same(L.ffn_norm, L0.ffn_norm) ||
            !same(L.q_norm, L0.q_norm) || !same(L.k_norm, L0.k_norm))
            return QW3_OK;
    }
    P.L0 = m->layers[0];
    P.lstride = lstride;
    if (!step_plan(P, m->layers[0])) return QW3_OK;
    LayerDev *dl = nullptr;
    M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&dl), sizeof(LayerDev) * c.n_layers));
    M_TRY(m, cudaMemcpyAsync(dl, m->layers.data(), sizeof(LayerDev) * c.n_layers, cudaMemcpyHostToDevice, m->stream));
    P.layers = dl;
    P.rope = m->rope;
    P.kv = static_cast<float *>(m->kv);
    P.seq_stride = m->seq_stride;
    P.kvsel_stride = m->kvsel_stride;
    P.head_stride = m->head_stride;
    P.layer_stride = m->layer_stride;
    P.seq_ids = m->d_seq;
    P.pos = m->d_pos;
    P.tok = m->d_tok;
    P.step_ctr = m->d_step;
    P.io = m->d_io;
    P.argmax_key = m->argmax_key;
    P.done_counter = m->done_counter;
    P.status = m->d_status;
    P.wait_ns = (c.flags & QW3_FLAG_TEST_NO_WAIT) ? 0ull : kWaitLimitNs;
    // exchange buffers, arrival counters (zero), the epoch and the abort word
    const size_t floats = static_cast<size_t>(P.H) + P.qkv_w + static_cast<size_t>(P.nkv) * P.S * P.G * (P.hd + 2) +
                          static_cast<size_t>(P.nh) * P.hd + P.I + 64;
    float *fb = nullptr;
    M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&fb), floats * 8));
    M_TRY(m, cudaMemsetAsync(fb, 0, floats * 8, m->stream));
    auto take = [&](size_t n) {   // room for one 64-bit word per value
        float *r = fb;
        fb += (n + 3) / 4 * 8;
        return r;
    };
    P.xb = take(P.H);
    P.qkvb = take(P.qkv_w);
    P.partb = take(static_cast<size_t>(P.nkv) * P.S * P.G * (P.hd + 2));
    P.ob = take(static_cast<size_t>(P.nh) * P.hd);
    P.actb = take(P.I);
    const size_t cbytes = static_cast<size_t>(step_counters(P.nkv)) * 128 + 256;
    unsigned *ew = nullptr;
    M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&ew), cbytes));
    M_TRY(m, cudaMemsetAsync(ew, 0, cbytes, m->stream));
    const unsigned init[2] = {1u, 0u};
    M_TRY(m, cudaMemcpyAsync(ew, init, sizeof init, cudaMemcpyHostToDevice, m->stream));
    P.epoch = ew;
    P.abort_word = ew + 1;
    P.ctrs = ew + 64;
    if (c.flags & QW3_FLAG_TRACE) {
        m->step_trace_words = 2 * ((kStepPhases * c.n_layers + 2) * 4 + 64) + P.NCTA * 16 + 64;
        M_TRY(m, model_alloc(m, reinterpret_cast<void **>(&P.trace), static_cast<size_t>(m->step_trace_words) * 8));
        M_TRY(m, cudaMemsetAsync(P.trace, 0, static_cast<size_t>(m->step_trace_words) * 8, m->stream));
    }
    M_TRY(m, cudaStreamSynchronize(m->stream));
    m->sp = P;
    m->step = true;
    return QW3_OK;
}

int check_model(const qw3_model *m) { return m ? QW3_OK : QW3_ERR_INVALID_ARG; }

// Caller buffers are read and written with plain scalar accesses of their
// element type; a pointer off that alignment is rejected here instead of
// faulting on the device.
bool misaligned(const void *p, size_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; }

int check_seq(qw3_model *m, int32_t seq) {
    if (seq < 0 || seq >= m->cfg.max_seqs) return fail(m, QW3_ERR_INVALID_ARG, "sequence id out of range");
    return QW3_OK;
}

}  // namespace

extern "C" {

const char *qw3_status_string(int status) {
    switch (status) {
        case QW3_OK: return "ok";
        case QW3_ERR_INVALID_ARG: return "invalid argument";
        case QW3_ERR_SHAPE: return "invalid shape";
        case QW3_ERR_SEQ_POS: return "position does not match the sequence length";
        case QW3_ERR_KV_OVERFLOW: return "KV cache overflow";
        case QW3_ERR_NONFINITE: return "non-finite value";
        case QW3_ERR_OOM: return "out of memory";
        case QW3_ERR_CUDA: return "CUDA error";
        case QW3_ERR_TIMEOUT: return "device wait timed out";
        default: return "unknown status";
    }
}

const char *qw3_last_error(const qw3_model *m) {
    if (m) return m->err.c_str();
    return thread_error().c_str();
}

void *qw3_stream(const qw3_model *m) { return m ? static_cast<void *>(m->stream) : nullptr; }

int qw3_create(const qw3_config *cfg, const qw3_weights *w, void *cuda_stream, qw3_model **out) {
    if (!out) return fail(nullptr, QW3_ERR_INVALID_ARG, "out is null");
    *out = nullptr;
    if (!cfg || !w || !w->layers || !w->token_embd || !w->output_norm)
        return fail(nullptr, QW3_ERR_INVALID_ARG, "null config or weights");
    std::string why;
    if (int rc = validate_config(cfg, why)) return fail(nullptr, rc, why);
    if (!cfg->tied_lm_head && !w->output) return fail(nullptr, QW3_ERR_INVALID_ARG, "untied lm_head needs output");
    {
        const char *fa = getenv("QW3_FAULT_ALLOC_AT");
        g_alloc_fail_at = fa ? atoi(fa) : -1;
        g_alloc_count = 0;
    }
    if (cudaError_t e = configure_all(); e != cudaSuccess) return cuda_err(nullptr, e, "configure kernels");

    qw3_model *m = new qw3_model();
    m->cfg = *cfg;
    m->kvtype = (cfg->flags & QW3_FLAG_KV_Q8) ? KV_Q8 : ((cfg->flags & QW3_FLAG_KV_F16) ? KV_F16 : KV_F32);
    m->act_q8 = (cfg->flags & QW3_FLAG_ACT_Q8) != 0;
    m->q4k = (cfg->flags & QW3_FLAG_WEIGHTS_Q4_K) != 0;
    auto bail = [&](int rc) {
        if (m->stream) cudaStreamSynchronize(m->stream);
        const std::string msg = m->err;
        free_all(m);
        delete m;
        set_thread_error(msg);
        return rc;
    };
    if (cuda_stream) {
        m->stream = static_cast<cudaStream_t>(cuda_stream);
    } else {
        if (cudaError_t e = cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking); e != cudaSuccess)
            return bail(cuda_err(m, e, "cudaStreamCreate"));
        m->own_stream = true;
    }
    if (cudaError_t e = cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking); e != cudaSuccess)
        return bail(cuda_err(m, e, "cudaStreamCreate"));

    const qw3_config &c = m->cfg;
    const int H = c.hidden, hd = c.head_dim, nh = c.n_heads, nkv = c.n_kv_heads, I = c.intermediate, V = c.vocab;
    m->qkv_w = (nh + 2 * nkv) * hd;
    const int qw = nh * hd;

    // ---- weights: one arena, zero-filled so padding rows are zero (Q4_K
    // models keep only the norms there; their matrices are raw rows)
    const int qm = m->q4k ? 0 : 1;
    size_t wbytes = qm * (qmat_bytes(V, H) + (c.tied_lm_head ? 0 : qmat_bytes(V, H)));
    wbytes += static_cast<size_t>(c.n_layers) *
              (qm * (qmat_bytes(m->qkv_w, H) + qmat_bytes(H, qw) + qmat_bytes(2 * I, H) + qmat_bytes(H, I)) +
               align_up(static_cast<size_t>(2 * H + 2 * hd) * 4, 256) + 4 * 256);
    wbytes += align_up(static_cast<size_t>(H) * 4, 256);
    uint8_t *arena = nullptr;
    if (cudaError_t e = model_alloc(m, reinterpret_cast<void **>(&arena), wbytes); e != cudaSuccess)
        return bail(cuda_err(m, e, "weight arena"));
    if (cudaError_t e = cudaMemsetAsync(arena, 0, wbytes, m->stream); e != cudaSuccess)
        return bail(cuda_err(m, e, "memset"));
    uint8_t *cur = arena;
    const bool on_dev = w->on_device != 0;
    uint8_t *staging = nullptr;
    // Q4_K: a device buffer of `rows` raw rows per matrix, filled by plain copies
    auto q4mat = [&](QMat &q, int rows, int cols) -> uint8_t * {
        q = qmat_shape(rows, cols);
        uint8_t *p = nullptr;
        if (model_alloc(m, reinterpret_cast<void **>(&p), static_cast<size_t>(rows) * q4k_row_bytes(cols)) != cudaSuccess)
            return nullptr;
        q.q4 = p;
        return p;
    };
    auto q4copy = [&](uint8_t *dst, size_t dpitch, const void *src, int rows, int cols) -> int {
        const size_t rb = q4k_row_bytes(cols);
        if (!src) return fail(m, QW3_ERR_INVALID_ARG, "a weight pointer is NULL");
        M_TRY(m, cudaMemcpy2DAsync(dst, dpitch, src, rb, rb, rows, cudaMemcpyDefault, m->stream));
        return QW3_OK;
    };
    if (!on_dev && !m->q4k) {
        size_t biggest = static_cast<size_t>(V) * H;
        biggest = std::max(biggest, static_cast<size_t>(qw) * H);
        biggest = std::max(biggest, static_cast<size_t>(I) * H);
        biggest = biggest / 32 * 34;
        if (cudaError_t e = model_alloc(m, reinterpret_cast<void **>(&staging), biggest); e != cudaSuccess)
            return bail(cuda_err(m, e, "staging"));
    }
    if (m->q4k) {
        const size_t rbH = q4k_row_bytes(H);
        if (!(m->emb4 = q4mat(m->embd, V, H))) return bail(fail(m, QW3_ERR_OOM, "Q4_K embedding"));
        if (int rc = q4copy(m->emb4, rbH, w->token_embd, V, H)) return bail(rc);
        if (c.tied_lm_head) {
            m->out = m->embd;
            m->out4 = m->emb4;
        } else {
            if (!(m->out4 = q4mat(m->out, V, H))) return bail(fail(m, QW3_ERR_OOM, "Q4_K output"));
            if (int rc = q4copy(m->out4, rbH, w->output, V, H)) return bail(rc);
        }
    } else {
        qmat_place(m->embd, cur, V, H);
        if (int rc = repack_into(m, m->embd, w->token_embd, V, H, 0, 1, on_dev, staging)) return bail(rc);
        if (c.tied_lm_head) {
            m->out = m->embd;
        } else {
            qmat_place(m->out, cur, V, H);
            if (int rc = repack_into(m, m->out, w->output, V, H, 0, 1, on_dev, staging)) return bail(rc);
        }
    }
    m->layers.resize(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const qw3_layer_weights &lw = w->layers[l];
        LayerDev &L = m->layers[l];
        int rc = QW3_OK;
        if (m->q4k) {
            // the Q8_0 layout's row order: [q; k; v], gate/up interleaved
            const size_t rbH = q4k_row_bytes(H);
            uint8_t *pq = q4mat(L.qkv, m->qkv_w, H), *po = q4mat(L.o, H, qw);
            uint8_t *pg = q4mat(L.gu, 2 * I, H), *pd = q4mat(L.down, H, I);
            if (!pq || !po || !pg || !pd) return bail(fail(m, QW3_ERR_OOM, "Q4_K layer weights"));
            rc = q4copy(pq, rbH, lw.attn_q, qw, H);
            if (!rc) rc = q4copy(pq + static_cast<size_t>(qw) * rbH, rbH, lw.attn_k, nkv * hd, H);
            if (!rc) rc = q4copy(pq + static_cast<size_t>(qw + nkv * hd) * rbH, rbH, lw.attn_v, nkv * hd, H);
            if (!rc) rc = q4copy(po, q4k_row_bytes(qw), lw.attn_output, H, qw);
            if (!rc) rc = q4copy(pg, 2 * rbH, lw.ffn_gate, I, H);
            if (!rc) rc = q4copy(pg + rbH, 2 * rbH, lw.ffn_up, I, H);
            if (!rc) rc = q4copy(pd, q4k_row_bytes(I), lw.ffn_down, H, I);
        } else {
            qmat_place(L.qkv, cur, m->qkv_w, H);
            qmat_place(L.o, cur, H, qw);
            qmat_place(L.gu, cur, 2 * I, H);
            qmat_place(L.down, cur, H, I);
            rc = repack_into(m, L.qkv, lw.attn_q, qw, H, 0, 1, on_dev, staging);
            if (!rc) rc = repack_into(m, L.qkv, lw.attn_k, nkv * hd, H, qw, 1, on_dev, staging);
            if (!rc) rc = repack_into(m, L.qkv, lw.attn_v, nkv * hd, H, qw + nkv * hd, 1, on_dev, staging);
            if (!rc) rc = repack_into(m, L.o, lw.attn_output, H, qw, 0, 1, on_dev, staging);
            if (!rc) rc = repack_into(m, L.gu, lw.ffn_gate, I, H, 0, 2, on_dev, staging);
            if (!rc) rc = repack_into(m, L.gu, lw.ffn_up, I, H, 1, 2, on_dev, staging);
            if (!rc) rc = repack_into(m, L.down, lw.ffn_down, H, I, 0, 1, on_dev, staging);
        }
        if (rc) return bail(rc);
        float *nb = reinterpret_cast<float *>(cur);
        L.attn_norm = nb;
        L.ffn_norm = nb + align_up(H, 64);
        L.q_norm = L.ffn_norm + align_up(H, 64);
        L.k_norm = L.q_norm + align_up(hd, 64);
        cur += align_up(static_cast<size_t>(2 * align_up(H, 64) + 2 * align_up(hd, 64)) * 4, 256);
        if ((rc = copy_f32(m, L.attn_norm, lw.attn_norm, H, on_dev))) return bail(rc);
        if ((rc = copy_f32(m, L.ffn_norm, lw.ffn_norm, H, on_dev))) return bail(rc);
        if ((rc = copy_f32(m, L.q_norm, lw.attn_q_norm, hd, on_dev))) return bail(rc);
        if ((rc = copy_f32(m, L.k_norm, lw.attn_k_norm, hd, on_dev))) return bail(rc);
    }
    m->out_norm = reinterpret_cast<float *>(cur);
    cur += align_up(static_cast<size_t>(H) * 4, 256);
    if (int rc = copy_f32(m, m->out_norm, w->output_norm, H, on_dev)) return bail(rc);
    if (static_cast<size_t>(cur - arena) > wbytes) return bail(fail(m, QW3_ERR_CUDA, "internal: arena overflow"));

    // ---- RoPE table (course 12.3.4): angle p * theta^(-2i/d), f64 -> f32
    {
        const size_t n = static_cast<size_t>(c.max_seq_len) * (hd / 2);
        std::vector<float2> tab(n);
        for (int p = 0; p < c.max_seq_len; ++p)
            for (int i = 0; i < hd / 2; ++i) {
                const double inv = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / hd);
                const double ang = static_cast<double>(p) * inv;
                tab[static_cast<size_t>(p) * (hd / 2) + i] =
                    make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang)));
            }
        if (cudaError_t e = model_alloc(m, reinterpret_cast<void **>(&m->rope), n * sizeof(float2)); e != cudaSuccess)
            return bail(cuda_err(m, e, "rope table"));
        if (cudaError_t e = cudaMemcpyAsync(m->rope, tab.data(), n * sizeof(float2), cudaMemcpyHostToDevice, m->stream);
            e != cudaSuccess)
            return bail(cuda_err(m, e, "rope upload"));
        if (cudaError_t e = cudaStreamSynchronize(m->stream); e != cudaSuccess) return bail(cuda_err(m, e, "sync"));
    }

    // ---- KV cache: [layer][seq][K|V][kv_head][capacity][row] of f32 or
    // half values, or of q8_0 rows (hd/32 blocks of 34 bytes; the capacity
    // rounded up to 32 positions so every head and every 32-position tile
    // starts 16-byte aligned, and 64 bytes of tail for the last bulk copy's
    // rounding to 16 bytes)
    const size_t cap = m->kvtype == KV_Q8 ? (static_cast<size_t>(c.max_seq_len) + 31) / 32 * 32
                                          : static_cast<size_t>(c.max_seq_len);
    m->head_stride = cap * kv_row_units(m->kvtype, hd);
    m->kvsel_stride = m->head_stride * nkv;
    m->seq_stride = 2 * m->kvsel_stride;
    m->layer_stride = m->seq_stride * c.max_seqs;
    {
        const size_t bytes = m->layer_stride * c.n_layers * kv_unit_bytes(m->kvtype) + 64;
        if (cudaError_t e = model_alloc(m, reinterpret_cast<void **>(&m->kv), bytes); e != cudaSuccess)
            return bail(cuda_err(m, e, "KV cache"));
    }
    m->seq_len.assign(c.max_seqs, 0);

    // ---- decode scratch
    const int Bm = c.max_seqs;
    m->attn_max_split = attn_decode_max_nsplit(hd, nh / nkv, nkv);
    if (c.max_seq_len >= kAttnLongCtx) {
        const int lc = attn_decode_max_nsplit(hd, nh / nkv, nkv * kAttnLongClusters);
        if (lc >= 4) m->attn_long_c = lc;
    }
    auto A = [&](void **p, size_t bytes) { return model_alloc(m, p, bytes); };
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->x), static_cast<size_t>(Bm) * H * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->h), static_cast<size_t>(Bm) * H * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->qkv), static_cast<size_t>(Bm) * m->qkv_w * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->o), static_cast<size_t>(Bm) * qw * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->act), static_cast<size_t>(Bm) * I * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->done_counter), 64);
    if (e == cudaSuccess && m->attn_long_c > 0)
        e = A(reinterpret_cast<void **>(&m->attn_cpart),
              static_cast<size_t>(nkv) * kAttnLongClusters * (nh / nkv) * (hd + 4) * 4);
    if (e == cudaSuccess && m->attn_long_c > 0) e = A(reinterpret_cast<void **>(&m->attn_ccnt), 64 * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->argmax_key), static_cast<size_t>(Bm) * 8);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->d_tok), static_cast<size_t>(Bm) * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->d_pos), static_cast<size_t>(Bm) * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->d_seq), static_cast<size_t>(Bm) * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->d_step), 64);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->d_status), 64);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->d_io), sizeof(DecodeIO));
    if (e == cudaSuccess && (c.flags & QW3_FLAG_TRACE)) {
        m->trace_kernels = 2 + 5 * c.n_layers + 4;
        const size_t tb = static_cast<size_t>(m->trace_kernels) * 2 * kTraceWords * 8;
        e = A(reinterpret_cast<void **>(&m->trace), tb);
        if (e == cudaSuccess) e = cudaMemsetAsync(m->trace, 0, tb, m->stream);
    }
    // ---- prefill scratch
    const size_t P = static_cast<size_t>(c.max_prefill);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->px), P * H * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->ph), P * H * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->pqkv), P * m->qkv_w * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->po), P * qw * 4);
    if (e == cudaSuccess) e = A(reinterpret_cast<void **>(&m->pact), P * I * 4);
    if (e != cudaSuccess) return bail(cuda_err(m, e, "scratch allocation"));
    if (int rc = setup_tensor_core_gemm(m)) return bail(rc);
    if (c.max_prefill >= kAttnPrefillTcMinRows && (hd == 64 || hd == 128)) {
        e = model_alloc(m, reinterpret_cast<void **>(&m->kvpack), attn_prefill_tc_pack_bytes(hd, nkv, c.max_seq_len));
        if (e != cudaSuccess) return bail(cuda_err(m, e, "prefill attention packing buffer"));
    }
    if (int rc = setup_step(m)) return bail(rc);
    e = cudaMemsetAsync(m->done_counter, 0, 64, m->stream);
    if (e == cudaSuccess && m->attn_ccnt) e = cudaMemsetAsync(m->attn_ccnt, 0, 64 * 4, m->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->argmax_key, 0, static_cast<size_t>(Bm) * 8, m->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->d_step, 0, 64, m->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->d_status, 0, 64, m->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(m->d_io, 0, sizeof(DecodeIO), m->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(m->stream);
    if (e != cudaSuccess) return bail(cuda_err(m, e, "scratch init"));
    *out = m;
    return QW3_OK;
}

int qw3_destroy(qw3_model *m) {
    if (!m) return QW3_OK;
    if (m->stream) cudaStreamSynchronize(m->stream);
    free_all(m);
    delete m;
    return QW3_OK;
}

namespace {

// Append n rows of sequence seq (max_prefill rows per pass through the
// layers). Outputs: the last row's logits and argmax (nullable), or, when
// all_logits is given, every row's logits [n][V] and argmax [n] (nullable).
int forward_rows(qw3_model *m, int32_t seq, const int32_t *tokens_dev, int32_t n, float *last_logits_dev,
                 int32_t *argmax_dev, float *all_logits, int32_t *all_argmax) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    if (int rc = check_seq(m, seq)) return rc;
    if (!tokens_dev || n < 1) return fail(m, QW3_ERR_INVALID_ARG, "a forward needs n >= 1 tokens");
    if (misaligned(tokens_dev, 4) || misaligned(last_logits_dev, 4) || misaligned(argmax_dev, 4) ||
        misaligned(all_logits, 4) || misaligned(all_argmax, 4))
        return fail(m, QW3_ERR_INVALID_ARG, "device buffers must be 4-byte aligned");
    const qw3_config &c = m->cfg;
    const int len = m->seq_len[seq];
    if (static_cast<int64_t>(len) + n > c.max_seq_len)
        return fail(m, QW3_ERR_KV_OVERFLOW, "prefill would overflow the KV cache");
    const int H = c.hidden, hd = c.head_dim, nh = c.n_heads, nkv = c.n_kv_heads, I = c.intermediate;
    const int qw = nh * hd;
    const float scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(hd)));
    cudaStream_t s = m->stream;
    for (int off = 0; off < n; off += c.max_prefill) {
        const int M = std::min(c.max_prefill, n - off);
        const int pos0 = len + off;
        if (m->q4k) M_TRY(m, launch_embed_q4k(tokens_dev + off, M, m->emb4, H, c.vocab, m->px, s));
        else M_TRY(m, launch_embed(tokens_dev + off, M, m->embd, m->px, false, s));
        for (int l = 0; l < c.n_layers; ++l) {
            const LayerDev &L = m->layers[l];
            void *kvl = kv_at(m, l, 0);
            M_TRY(m, launch_rmsnorm_rows(m->px, M, H, L.attn_norm, c.rms_eps, m->ph, s));
            M_TRY(m, lin_gemm(m, m->ph, M, H, L.qkv, m->pqkv, GEMV_STORE, nullptr, nullptr, s));
            M_TRY(m, launch_qk_rope_append(m->pqkv, M, m->qkv_w, L.q_norm, L.k_norm, c.rms_eps, m->rope, nullptr, seq,
                                           nullptr, pos0, kvl, m->seq_stride, m->kvsel_stride, m->head_stride, nh,
                                           nkv, hd, m->kvtype, s));
            if (m->kvpack && M >= kAttnPrefillTcMinRows) {
                M_TRY(m, launch_attn_prefill_tc(m->pqkv, M, m->qkv_w, kv_at(m, l, seq), m->kvsel_stride,
                                                m->head_stride, pos0, nh, nkv, hd, scale, m->po, m->kvpack,
                                                m->d_status, m->kvtype, s));
            } else {
                M_TRY(m, launch_attn_prefill(m->pqkv, M, m->qkv_w, kv_at(m, l, seq), m->kvsel_stride, m->head_stride,
                                             pos0, nh, nkv, hd, scale, m->po, m->kvtype, s));
            }
            M_TRY(m, lin_gemm(m, m->po, M, qw, L.o, m->px, GEMV_RESID, nullptr, nullptr, s));
            M_TRY(m, launch_rmsnorm_rows(m->px, M, H, L.ffn_norm, c.rms_eps, m->ph, s));
            M_TRY(m, lin_gemm(m, m->ph, M, H, L.gu, m->pact, GEMV_SWIGLU, nullptr, nullptr, s));
            M_TRY(m, lin_gemm(m, m->pact, M, I, L.down, m->px, GEMV_RESID, nullptr, nullptr, s));
        }
        if (all_logits) {
            // final norm of every row, the lm_head over all of them, each row's argmax
            float *lg = all_logits + static_cast<size_t>(off) * c.vocab;
            M_TRY(m, launch_rmsnorm_rows(m->px, M, H, m->out_norm, c.rms_eps, m->ph, s));
            M_TRY(m, lin_gemm(m, m->ph, M, H, m->out, lg, GEMV_STORE, nullptr, nullptr, s));
            if (all_argmax) M_TRY(m, launch_argmax_rows(lg, M, c.vocab, all_argmax + off, m->d_status, s));
        } else if (off + M == n && (last_logits_dev || argmax_dev) && m->q4k) {
            M_TRY(m, launch_gemv_q4k(m->out4, c.vocab, H, 1, m->px + static_cast<size_t>(M - 1) * H, m->out_norm,
                                     c.rms_eps, last_logits_dev, GEMV_ARGMAX, nullptr, m->argmax_key, false, s));
            M_TRY(m, launch_argmax_finalize(m->argmax_key, 1, nullptr, argmax_dev, nullptr, nullptr, m->d_status, s));
        } else if (off + M == n && (last_logits_dev || argmax_dev)) {
            GemvArgs a{};
            a.act_q8 = m->act_q8;
            a.W = m->out; a.N = c.vocab; a.K = H; a.B = 1;
            a.x = m->px + static_cast<size_t>(M - 1) * H; a.norm_w = m->out_norm; a.eps = c.rms_eps;
            a.y = last_logits_dev; a.argmax_key = m->argmax_key; a.done_counter = m->done_counter; a.io = nullptr;
            a.argmax_out = argmax_dev; a.status = m->d_status;
            M_TRY(m, launch_gemv(a, GEMV_ARGMAX, false, s));
        }
    }
    m->seq_len[seq] = len + n;
    return QW3_OK;
}

}  // namespace

int qw3_prefill(qw3_model *m, int32_t seq, const int32_t *tokens_dev, int32_t n, float *last_logits_dev,
                int32_t *argmax_dev) {
    return forward_rows(m, seq, tokens_dev, n, last_logits_dev, argmax_dev, nullptr, nullptr);
}

int qw3_forward_all_logits(qw3_model *m, int32_t seq, const int32_t *tokens_dev, int32_t n, float *logits_dev,
                           int32_t *argmax_dev) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    if (!logits_dev) return fail(m, QW3_ERR_INVALID_ARG, "all-logits forward needs a logits buffer");
    return forward_rows(m, seq, tokens_dev, n, nullptr, nullptr, logits_dev, argmax_dev);
}

int qw3_decode(qw3_model *m, int32_t B, const int32_t *seqs_host, const int32_t *tokens_dev, const int32_t *pos_host,
               float *logits_dev, int32_t *argmax_dev) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    const qw3_config &c = m->cfg;
    if (B < 1 || B > c.max_seqs) return fail(m, QW3_ERR_INVALID_ARG, "batch must be in [1, max_seqs]");
    if (!tokens_dev || !pos_host) return fail(m, QW3_ERR_INVALID_ARG, "null tokens or positions");
    if (misaligned(tokens_dev, 4) || misaligned(logits_dev, 4) || misaligned(argmax_dev, 4))
        return fail(m, QW3_ERR_INVALID_ARG, "device buffers must be 4-byte aligned");
    std::vector<int32_t> seqs(B), pos(B);
    std::vector<char> seen(c.max_seqs, 0);
    for (int b = 0; b < B; ++b) {
        const int sq = seqs_host ? seqs_host[b] : b;
        if (sq < 0 || sq >= c.max_seqs) return fail(m, QW3_ERR_INVALID_ARG, "sequence id out of range");
        if (seen[sq]) return fail(m, QW3_ERR_INVALID_ARG, "duplicate sequence id in batch");
        seen[sq] = 1;
        if (pos_host[b] != m->seq_len[sq]) return fail(m, QW3_ERR_SEQ_POS, "pos != current sequence length");
        if (m->seq_len[sq] + 1 > c.max_seq_len) return fail(m, QW3_ERR_KV_OVERFLOW, "decode would overflow the KV cache");
        seqs[b] = sq;
        pos[b] = pos_host[b];
    }
    DecodeIO io{logits_dev, argmax_dev, nullptr, nullptr};
    M_TRY(m, cudaMemcpyAsync(m->d_seq, seqs.data(), B * 4, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_pos, pos.data(), B * 4, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_io, &io, sizeof io, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_tok, tokens_dev, B * 4, cudaMemcpyDeviceToDevice, m->stream));
    if (m->step && B == 1) {
        M_TRY(m, launch_step(m->sp, m->stream));
    } else if (int rc = run_decode_step(m, B)) {
        return rc;
    }
    for (int b = 0; b < B; ++b) m->seq_len[seqs[b]] += 1;
    return QW3_OK;
}

int qw3_generate_greedy(qw3_model *m, int32_t B, const int32_t *seqs_host, int32_t n_steps,
                        const int32_t *first_tokens_dev, int32_t *out_tokens_dev) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    const qw3_config &c = m->cfg;
    if (B < 1 || B > c.max_seqs) return fail(m, QW3_ERR_INVALID_ARG, "batch must be in [1, max_seqs]");
    if (n_steps < 0 || !first_tokens_dev || (n_steps > 0 && !out_tokens_dev))
        return fail(m, QW3_ERR_INVALID_ARG, "bad generate arguments");
    if (misaligned(first_tokens_dev, 4) || misaligned(out_tokens_dev, 4))
        return fail(m, QW3_ERR_INVALID_ARG, "device buffers must be 4-byte aligned");
    if (n_steps == 0) return QW3_OK;
    std::vector<int32_t> seqs(B), pos(B);
    std::vector<char> seen(c.max_seqs, 0);
    for (int b = 0; b < B; ++b) {
        const int sq = seqs_host ? seqs_host[b] : b;
        if (sq < 0 || sq >= c.max_seqs) return fail(m, QW3_ERR_INVALID_ARG, "sequence id out of range");
        if (seen[sq]) return fail(m, QW3_ERR_INVALID_ARG, "duplicate sequence id in batch");
        seen[sq] = 1;
        if (static_cast<int64_t>(m->seq_len[sq]) + n_steps > c.max_seq_len)
            return fail(m, QW3_ERR_KV_OVERFLOW, "generation would overflow the KV cache");
        seqs[b] = sq;
        pos[b] = m->seq_len[sq];
    }
    DecodeIO io{nullptr, nullptr, out_tokens_dev, nullptr};
    const int32_t zero = 0;
    M_TRY(m, cudaMemcpyAsync(m->d_seq, seqs.data(), B * 4, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_pos, pos.data(), B * 4, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_io, &io, sizeof io, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_step, &zero, 4, cudaMemcpyHostToDevice, m->stream));
    M_TRY(m, cudaMemcpyAsync(m->d_tok, first_tokens_dev, B * 4, cudaMemcpyDeviceToDevice, m->stream));
    for (int sidx = 0; sidx < n_steps; ++sidx) {
        if (m->step && B == 1) {
            M_TRY(m, launch_step(m->sp, m->stream));
        } else if (int rc = run_decode_step(m, B)) {
            return rc;
        }
    }
    for (int b = 0; b < B; ++b) m->seq_len[seqs[b]] += n_steps;
    return QW3_OK;
}

int qw3_reset(qw3_model *m, int32_t seq) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    if (int rc = check_seq(m, seq)) return rc;
    m->seq_len[seq] = 0;
    return QW3_OK;
}

int qw3_truncate(qw3_model *m, int32_t seq, int32_t keep_len) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    if (int rc = check_seq(m, seq)) return rc;
    if (keep_len < 0) return fail(m, QW3_ERR_INVALID_ARG, "keep_len must be >= 0");
    if (keep_len < m->seq_len[seq]) m->seq_len[seq] = keep_len;
    return QW3_OK;
}

int qw3_seq_len(const qw3_model *m, int32_t seq, int32_t *len_out) {
    if (!m || !len_out) return QW3_ERR_INVALID_ARG;
    if (seq < 0 || seq >= m->cfg.max_seqs) return QW3_ERR_INVALID_ARG;
    *len_out = m->seq_len[seq];
    return QW3_OK;
}

int qw3_debug_read_kv(qw3_model *m, int32_t layer, int32_t seq, int32_t pos0, int32_t n, float *k_out_dev,
                      float *v_out_dev) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    if (int rc = check_seq(m, seq)) return rc;
    const qw3_config &c = m->cfg;
    if (layer < 0 || layer >= c.n_layers || pos0 < 0 || n < 0 || static_cast<int64_t>(pos0) + n > c.max_seq_len ||
        !k_out_dev || !v_out_dev || misaligned(k_out_dev, 4) || misaligned(v_out_dev, 4))
        return fail(m, QW3_ERR_INVALID_ARG, "bad KV read range");
    M_TRY(m, launch_copy_kv_rows(kv_at(m, layer, seq), m->kvsel_stride, m->head_stride, pos0, n, c.n_kv_heads,
                                 c.head_dim, k_out_dev, v_out_dev, m->kvtype, m->stream));
    return QW3_OK;
}

int qw3_debug_read_trace(qw3_model *m, uint64_t *out_host, int32_t max_records, int32_t *n_out) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    if (!n_out || max_records < 0 || (max_records > 0 && !out_host))
        return fail(m, QW3_ERR_INVALID_ARG, "bad trace arguments");
    *n_out = 0;
    if (!m->trace) return fail(m, QW3_ERR_INVALID_ARG, "model was created without QW3_FLAG_TRACE");
    const bool stp = m->step && m->sp.trace;
    const int avail = stp ? m->step_trace_words / kTraceWords : 2 * m->trace_kernels;
    const int n = std::min(max_records, avail);
    M_TRY(m, cudaStreamSynchronize(m->stream));
    M_TRY(m, cudaMemcpy(out_host, stp ? m->sp.trace : m->trace, static_cast<size_t>(n) * kTraceWords * 8,
                        cudaMemcpyDeviceToHost));
    *n_out = n;
    return QW3_OK;
}

int qw3_decode_plan(const qw3_model *m, int32_t B, int32_t *persistent, int32_t *launches_per_step) {
    if (!m || !persistent || !launches_per_step || B < 1 || B > m->cfg.max_seqs) return QW3_ERR_INVALID_ARG;
    const qw3_config &c = m->cfg;
    if (m->step && B == 1) {
        *persistent = 1;
        *launches_per_step = 1;
        return QW3_OK;
    }
    *persistent = 0;
    *launches_per_step = use_gemv(c, B) ? ((c.flags & QW3_FLAG_WEIGHTS_Q4_K) ? 3 : 2) + 5 * c.n_layers
                                        : 4 + 7 * c.n_layers;
    return QW3_OK;
}

int qw3_sync(qw3_model *m) {
    if (check_model(m)) return QW3_ERR_INVALID_ARG;
    M_TRY(m, cudaStreamSynchronize(m->stream));
    int32_t st = 0;
    M_TRY(m, cudaMemcpy(&st, m->d_status, 4, cudaMemcpyDeviceToHost));
    if (st != 0) {
        M_TRY(m, cudaMemset(m->d_status, 0, 4));
        return fail(m, st, std::string("device reported: ") + qw3_status_string(st));
    }
    return QW3_OK;
}

int qw3_q8_0_quantize(const float *x_dev, int64_t n, void *blocks_dev, int32_t *status_dev, void *stream) {
    if (n < 0 || (n > 0 && (!x_dev || !blocks_dev))) return fail(nullptr, QW3_ERR_INVALID_ARG, "bad quantize arguments");
    if (n % 32) return fail(nullptr, QW3_ERR_SHAPE, "n must be a multiple of 32");
    if (misaligned(x_dev, 4) || misaligned(blocks_dev, 2) || misaligned(status_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "x must be 4-byte, blocks 2-byte aligned");
    QW3_CUDA_TRY(launch_quantize(x_dev, n / 32, static_cast<uint8_t *>(blocks_dev), status_dev,
                                 static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

int qw3_q8_0_dequantize(const void *blocks_dev, int64_t n, float *y_dev, void *stream) {
    if (n < 0 || (n > 0 && (!y_dev || !blocks_dev))) return fail(nullptr, QW3_ERR_INVALID_ARG, "bad dequantize arguments");
    if (n % 32) return fail(nullptr, QW3_ERR_SHAPE, "n must be a multiple of 32");
    if (misaligned(blocks_dev, 2) || misaligned(y_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "blocks must be 2-byte, y 4-byte aligned");
    QW3_CUDA_TRY(launch_dequantize(static_cast<const uint8_t *>(blocks_dev), n / 32, y_dev,
                                   static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

int qw3_q4_k_quantize(const float *x_dev, int64_t n, void *blocks_dev, int32_t *status_dev, void *stream) {
    if (n < 0 || (n > 0 && (!x_dev || !blocks_dev))) return fail(nullptr, QW3_ERR_INVALID_ARG, "bad quantize arguments");
    if (n % 256) return fail(nullptr, QW3_ERR_SHAPE, "n must be a multiple of 256");
    if (misaligned(x_dev, 16) || misaligned(blocks_dev, 16) || misaligned(status_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "x and blocks must be 16-byte aligned");
    QW3_CUDA_TRY(launch_q4k_quantize(x_dev, n / 256, static_cast<uint8_t *>(blocks_dev), status_dev,
                                     static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

int qw3_q4_k_dequantize(const void *blocks_dev, int64_t n, float *y_dev, void *stream) {
    if (n < 0 || (n > 0 && (!y_dev || !blocks_dev))) return fail(nullptr, QW3_ERR_INVALID_ARG, "bad dequantize arguments");
    if (n % 256) return fail(nullptr, QW3_ERR_SHAPE, "n must be a multiple of 256");
    if (misaligned(blocks_dev, 2) || misaligned(y_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "blocks must be 2-byte, y 4-byte aligned");
    QW3_CUDA_TRY(launch_q4k_dequantize(static_cast<const uint8_t *>(blocks_dev), n / 256, y_dev,
                                       static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

int qw3_q4_k_gemv(const void *W_dev, int32_t rows, int32_t cols, const float *x_dev, int32_t B, float *y_dev,
                  void *stream) {
    if (!W_dev || !x_dev || !y_dev || rows < 0 || cols < 0 || B < 1 || B > 8)
        return fail(nullptr, QW3_ERR_INVALID_ARG, "bad gemv arguments");
    if (cols % 256 || !q4k_gemv_fits(B, cols)) return fail(nullptr, QW3_ERR_SHAPE, "cols % 256 and B * cols <= 49152");
    if (misaligned(W_dev, 16) || misaligned(x_dev, 16) || misaligned(y_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "W and x must be 16-byte, y 4-byte aligned");
    if (rows == 0) return QW3_OK;
    QW3_CUDA_TRY(configure_all());   // the kernel's shared-memory limit
    QW3_CUDA_TRY(launch_gemv_q4k(static_cast<const uint8_t *>(W_dev), rows, cols, B, x_dev, nullptr, 0.0f, y_dev,
                                 GEMV_STORE, nullptr, nullptr, false, static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

int qw3_q8_0_gemv(const void *W_dev, int32_t rows, int32_t cols, const float *x_dev, int32_t B, float *y_dev,
                  void *stream) {
    if (!W_dev || !x_dev || !y_dev || rows < 0 || cols < 0 || B < 1 || B > 8)
        return fail(nullptr, QW3_ERR_INVALID_ARG, "bad gemv arguments");
    if (cols % 32) return fail(nullptr, QW3_ERR_SHAPE, "cols must be a multiple of 32");
    if (misaligned(W_dev, 2) || misaligned(x_dev, 4) || misaligned(y_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "W must be 2-byte, x and y 4-byte aligned");
    if (rows == 0) return QW3_OK;
    QW3_CUDA_TRY(launch_gemv_raw(static_cast<const uint8_t *>(W_dev), rows, cols, x_dev, B, y_dev, false,
                                 static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

int64_t qw3_q8_0_gemm_workspace_bytes(int32_t rows, int32_t cols, int32_t M) {
    if (rows < 0 || cols < 0 || M < 0 || cols % 64) return -1;
    return static_cast<int64_t>(gemm_q8_raw_workspace_bytes(rows, cols, M));
}

int qw3_q8_0_gemm(const void *W_dev, int32_t rows, int32_t cols, const float *x_dev, int32_t M, float *y_dev,
                  void *workspace_dev, int64_t workspace_bytes, void *stream) {
    if (!W_dev || !x_dev || !y_dev || rows < 0 || cols < 0 || M < 0)
        return fail(nullptr, QW3_ERR_INVALID_ARG, "bad gemm arguments");
    if (cols % 64) return fail(nullptr, QW3_ERR_SHAPE, "cols must be a multiple of 64");
    if (misaligned(W_dev, 2) || misaligned(x_dev, 16) || misaligned(y_dev, 4) || misaligned(workspace_dev, 16))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "W must be 2-byte, x and the workspace 16-byte, y 4-byte aligned");
    if (rows == 0 || M == 0) return QW3_OK;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cols == 0) {
        QW3_CUDA_TRY(cudaMemsetAsync(y_dev, 0, static_cast<size_t>(M) * rows * sizeof(float), s));
        return QW3_OK;
    }
    if (!workspace_dev || workspace_bytes < 0 ||
        static_cast<uint64_t>(workspace_bytes) < gemm_q8_raw_workspace_bytes(rows, cols, M))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "workspace too small");
    QW3_CUDA_TRY(configure_all());
    QW3_CUDA_TRY(launch_gemm_q8_raw(static_cast<const uint8_t *>(W_dev), rows, cols, x_dev, M, y_dev,
                                    static_cast<uint8_t *>(workspace_dev), s));
    return QW3_OK;
}

int qw3_q8_0_gemv_q8act(const void *W_dev, int32_t rows, int32_t cols, const float *x_dev, int32_t B, float *y_dev,
                        void *stream) {
    if (!W_dev || !x_dev || !y_dev || rows < 0 || cols < 0 || B < 1 || B > 8)
        return fail(nullptr, QW3_ERR_INVALID_ARG, "bad gemv arguments");
    if (cols % 256) return fail(nullptr, QW3_ERR_SHAPE, "cols must be a multiple of 256");
    if (static_cast<int64_t>(B) * cols > 49152) return fail(nullptr, QW3_ERR_SHAPE, "B * cols must be <= 49152");
    if (misaligned(W_dev, 16) || misaligned(x_dev, 16) || misaligned(y_dev, 4))
        return fail(nullptr, QW3_ERR_INVALID_ARG, "W and x must be 16-byte, y 4-byte aligned");
    if (rows == 0) return QW3_OK;
    QW3_CUDA_TRY(launch_gemv_raw(static_cast<const uint8_t *>(W_dev), rows, cols, x_dev, B, y_dev, true,
                                 static_cast<cudaStream_t>(stream)));
    return QW3_OK;
}

}  // extern "C"
