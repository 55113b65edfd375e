/*
 * qw3.h -- C ABI of libqw3: the forward pass of a Qwen3-style dense decoder
 * whose linear weights are GGUF Q8_0 blocks, on one NVIDIA GB300 (sm_103a).
 *
 * What is computed (page titles and sections):
 *   "A transformer from scratch" (Fucina course ch. 12)
 *     12.3    forward pass: embedding gather, L x (attention block + FFN
 *             block), final RMSNorm, lm_head on the last row only
 *     12.3.1  embedding rows dequantised on the fly; tied lm_head reuses the
 *             embedding table when there is no output weight
 *     12.3.2  RMSNorm y = x / sqrt(mean(x^2) + eps) * w
 *     12.3.3  Q/K/V projections; q is n_heads*head_dim wide, k and v
 *             n_kv_heads*head_dim wide
 *     12.3.4  NeoX ("half") RoPE, angle p / theta^(2i/d) for pair (i, i+d/2)
 *     12.3.5  grouped-query causal attention, kv head = h / (n_heads/n_kv),
 *             scale 1/sqrt(head_dim)
 *     12.3.6  SwiGLU FFN down(silu(gate x) * up x)
 *     12.3.7  residual adds
 *     12.4    KV cache: K stored after norm and RoPE, V as projected; the new
 *             rows are written at the current length, which moves once per
 *             call; pos must equal the length, and rows must fit
 *     12.6    greedy decoding (argmax, lowest index on ties)
 *   minfer "Qwen3 Support Plan (dense)"
 *     1       tensor inventory; 2.1 head_dim decoupled from hidden/n_heads;
 *     2.2     per-head Q/K RMSNorm (length head_dim) before RoPE
 *   "Model files and quantization" (Fucina course ch. 11)
 *     11.7    Q8_0: blocks of 32, f16 scale d then 32 int8 q (34 bytes),
 *             value = d * q; encoder d = max|x| / 127, q = round(x * (1/d))
 *     11.10   non-finite encoder input is an error
 *
 * Conventions
 *   - Every function returns an int status (enum qw3_status); 0 is success.
 *   - "_dev" pointers are CUDA device pointers; "_host" pointers are host
 *     memory read during the call. The caller owns every buffer it passes.
 *     Buffers are accessed with plain loads and stores of their element
 *     type: f32/int32 buffers must be 4-byte aligned, Q8_0 blocks 2-byte
 *     aligned (QW3_ERR_INVALID_ARG otherwise).
 *   - Q8_0 matrices are [rows][cols/32] blocks in GGUF order (row-major,
 *     blocks along the input dimension), 34 bytes per block, so a matrix of
 *     rows x cols takes rows*cols/32*34 bytes. cols must be a multiple of 32.
 *   - Activations, norm weights, logits and the KV cache are float32.
 *   - Model calls run asynchronously on the model's stream; host-side
 *     validation happens before anything is enqueued, and an error leaves
 *     every sequence length unchanged. Device-side conditions (NaN logits, a
 *     bounded wait that timed out) are recorded in a status word that
 *     qw3_sync() returns and clears.
 *   - Not thread-safe per model: calls on one qw3_model must not overlap.
 */
#ifndef QW3_H
#define QW3_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QW3_API __attribute__((visibility("default")))
#else
#define QW3_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum qw3_status {
    QW3_OK = 0,
    QW3_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad count or id */
    QW3_ERR_SHAPE = 2,        /* a size the format or model cannot take     */
    QW3_ERR_SEQ_POS = 3,      /* pos != current sequence length (12.4)      */
    QW3_ERR_KV_OVERFLOW = 4,  /* rows would not fit in the KV cache (12.4)  */
    QW3_ERR_NONFINITE = 5,    /* NaN/inf encoder input, or NaN logits       */
    QW3_ERR_OOM = 6,          /* a device or host allocation failed         */
    QW3_ERR_CUDA = 7,         /* a CUDA runtime call failed                 */
    QW3_ERR_TIMEOUT = 8       /* a bounded device-side wait expired         */
};

/* Model geometry and capacities (course 12.1: the nine integers of Config). */
typedef struct qw3_config {
    int32_t vocab;          /* V                                            */
    int32_t hidden;         /* H, multiple of 32                            */
    int32_t n_layers;       /* L                                            */
    int32_t n_heads;        /* query heads                                  */
    int32_t n_kv_heads;     /* key/value heads, <= 64; n_heads % n_kv_heads == 0 */
    int32_t head_dim;       /* 64 or 128                                    */
    int32_t intermediate;   /* FFN width, multiple of 32                    */
    float rms_eps;          /* 1e-6 for Qwen3                               */
    float rope_theta;       /* 1e6 for Qwen3                                */
    int32_t tied_lm_head;   /* 1: lm_head is token_embd                     */
    int32_t max_seqs;       /* number of sequence slots (KV caches)         */
    int32_t max_seq_len;    /* KV capacity per sequence, in positions       */
    int32_t max_prefill;    /* largest chunk one prefill pass processes;
                               longer prompts run in chunks of this size   */
    int32_t flags;          /* QW3_FLAG_* bits                              */
} qw3_config;

#define QW3_FLAG_NO_GRAPH 0x1  /* launch decode kernels directly, no CUDA graph */
#define QW3_FLAG_NO_PDL   0x2  /* no programmatic dependent launch               */
#define QW3_FLAG_TRACE    0x4  /* record timestamps of decode steps          */
#define QW3_FLAG_PER_KERNEL 0x8 /* batch-1 decode through the per-kernel
                                  chain (one launch per projection and
                                  attention) instead of the persistent
                                  decode-step kernel                          */
#define QW3_FLAG_TEST_NO_WAIT 0x10 /* testing only: a wait on another CTA's
                                  data in the decode-step kernel gives up at
                                  its first miss (QW3_ERR_TIMEOUT) instead
                                  of after 1 s                                */
#define QW3_FLAG_KV_F16 0x20     /* KV cache in IEEE half (the default cache
                                  type of "A transformer from scratch",
                                  12.4) instead of f32: half the cache bytes;
                                  keys and values are rounded to nearest
                                  even when appended. Batch-1 decode then
                                  runs the per-kernel chain.                  */
#define QW3_FLAG_KV_Q8  0x80     /* KV cache as q8_0 rows ("The LLM stack",
                                  13.4): each (position, kv head) row is
                                  head_dim/32 Q8_0 blocks (11.7 encoder) at
                                  34 bytes per 32 values. A decode step
                                  quantises the query once per head and scores
                                  with the integer block dots (to f32
                                  rounding); prefill and the all-logits
                                  forward read the dequantised rows. Not with
                                  QW3_FLAG_KV_F16. Batch-1 decode runs the
                                  per-kernel chain.                           */
#define QW3_FLAG_WEIGHTS_Q4_K 0x100 /* every linear weight (the embedding and
                                  output included) is given as Q4_K blocks
                                  ("Model files and quantization", 11.8:
                                  144 bytes per 256 values, GGUF layout)
                                  instead of Q8_0; hidden, intermediate and
                                  n_heads*head_dim must be multiples of 256.
                                  Decode of up to 8 rows streams the Q4_K
                                  rows; prefill and larger batches run the
                                  tensor-core GEMMs on tiles packed from
                                  them. Not with QW3_FLAG_ACT_Q8.             */
#define QW3_FLAG_ACT_Q8 0x40     /* every linear layer takes its input rows
                                  re-quantized to Q8_0 per 32-block on the
                                  fly ("Model files and quantization", 11.9:
                                  dynamic activations, integer block dots)
                                  instead of f32. Batch-1 decode then runs
                                  the per-kernel chain.                       */

/* One decoder layer (minfer section 1). Q8_0 matrices [out][in]:
 *   attn_q [n_heads*head_dim][H], attn_k and attn_v [n_kv_heads*head_dim][H],
 *   attn_output [H][n_heads*head_dim], ffn_gate and ffn_up [I][H],
 *   ffn_down [H][I]. Norm weights f32: attn_norm [H], attn_q_norm and
 *   attn_k_norm [head_dim], ffn_norm [H]. */
typedef struct qw3_layer_weights {
    const void *attn_q, *attn_k, *attn_v, *attn_output;
    const void *ffn_gate, *ffn_up, *ffn_down;
    const float *attn_norm, *attn_q_norm, *attn_k_norm, *ffn_norm;
} qw3_layer_weights;

/* token_embd and output are Q8_0 [V][H]; output is ignored (may be NULL)
 * when tied_lm_head. output_norm is f32 [H]. layers is a host array of
 * n_layers entries. on_device: 1 if every weight pointer is device memory,
 * 0 if host memory. */
typedef struct qw3_weights {
    const void *token_embd;
    const void *output;
    const float *output_norm;
    const qw3_layer_weights *layers;
    int32_t on_device;
} qw3_weights;

typedef struct qw3_model qw3_model;

/* Validate cfg (shapes as above, plus the head_dim checks of minfer 2.1),
 * copy and repack every weight into device storage owned by the model (the
 * caller may free its buffers when this returns), allocate the KV caches
 * (max_seqs x max_seq_len positions, f32) and the RoPE table. cuda_stream is
 * a cudaStream_t the model will run on; NULL makes the model create its own.
 * On error *out is NULL and nothing is leaked. */
QW3_API int qw3_create(const qw3_config *cfg, const qw3_weights *weights,
               void *cuda_stream, qw3_model **out);

/* Wait for outstanding work and free everything the model owns. NULL is ok. */
QW3_API int qw3_destroy(qw3_model *m);

/* Prefill (course 12.3 with seq = n): append n tokens to sequence `seq` at
 * positions len..len+n-1 and, when requested, return the last row's logits
 * (last_logits_dev, f32 [V]) and its argmax (argmax_dev, int32 [1]); both are
 * nullable. tokens_dev: int32 [n], each in [0, V). n >= 1 and len + n must
 * not exceed max_seq_len (QW3_ERR_KV_OVERFLOW). */
QW3_API int qw3_prefill(qw3_model *m, int32_t seq, const int32_t *tokens_dev, int32_t n,
                float *last_logits_dev, int32_t *argmax_dev);

/* All-logits forward ("A transformer from scratch", 12.3.7 and 12.5: the
 * step that returns logits for every appended row, the shape a speculative
 * verify needs): append n tokens to sequence `seq` exactly as qw3_prefill
 * does and return every appended row's logits in logits_dev (f32 [n][V],
 * required) and, when argmax_dev (int32 [n]) is not NULL, each row's greedy
 * argmax (lowest index among equal maxima). Row i is the prediction after
 * token i. Errors as qw3_prefill; nothing is appended on an error. */
QW3_API int qw3_forward_all_logits(qw3_model *m, int32_t seq, const int32_t *tokens_dev, int32_t n,
                                   float *logits_dev, int32_t *argmax_dev);

/* One decode step for B sequences at once (course 12.5, batch decode: one
 * pass over the weights, RoPE positions, KV appends and attention per
 * sequence). seqs_host: int32 [B] distinct slot ids, NULL means 0..B-1.
 * tokens_dev: int32 [B]. pos_host: int32 [B], pos_host[b] must equal the
 * current length of sequence seqs[b] (QW3_ERR_SEQ_POS). logits_dev: nullable
 * f32 [B][V]. argmax_dev: nullable int32 [B]. Each sequence grows by one. */
QW3_API int qw3_decode(qw3_model *m, int32_t B, const int32_t *seqs_host,
               const int32_t *tokens_dev, const int32_t *pos_host,
               float *logits_dev, int32_t *argmax_dev);

/* n_steps greedy decode steps for B sequences without host round trips
 * (course 12.6). Step 0 feeds first_tokens_dev[b] (int32 [B]) at the current
 * length of seqs[b]; step s feeds the argmax of step s-1. out_tokens_dev
 * receives int32 [n_steps][B] argmax ids. Each sequence grows by n_steps. */
QW3_API int qw3_generate_greedy(qw3_model *m, int32_t B, const int32_t *seqs_host,
                        int32_t n_steps, const int32_t *first_tokens_dev,
                        int32_t *out_tokens_dev);

/* Sequence bookkeeping (course 12.4): reset sets the length to 0, truncate
 * to min(len, keep_len); neither touches device memory. */
QW3_API int qw3_reset(qw3_model *m, int32_t seq);
QW3_API int qw3_truncate(qw3_model *m, int32_t seq, int32_t keep_len);
QW3_API int qw3_seq_len(const qw3_model *m, int32_t seq, int32_t *len_out);

/* Copy positions [pos0, pos0+n) of one layer's cache for `seq` into
 * k_out_dev and v_out_dev, each f32 [n][n_kv_heads][head_dim] (the pages'
 * [seq, kv_head, d] layout). Enqueued on the model's stream. */
QW3_API int qw3_debug_read_kv(qw3_model *m, int32_t layer, int32_t seq, int32_t pos0,
                      int32_t n, float *k_out_dev, float *v_out_dev);

/* Timestamps recorded when the model was created with QW3_FLAG_TRACE, in
 * records of 8 u64.
 * Per-kernel decode path (QW3_FLAG_PER_KERNEL at batch 1; B > 1 always): the
 * most recent step; for each kernel, in launch order, two records (its first
 * and its last CTA): entry, after the wait for the previous kernel, after the
 * prologue, after the weight/KV stream, exit, two kernel-specific words, SM
 * id (%globaltimer ns).
 * Persistent step kernel (batch 1, the default): the most recent step, as a
 * flat array of u64 words. With P = 6 * n_layers + 2 phases, for the first
 * and then the last CTA, 4 * P + 64 words: per phase (0 = step start, 6 l + k
 * for phase k = 1..6 of layer l, P - 1 = lm_head) inputs staged, first weight
 * chunk in, dot products done, outputs published (SM cycle counter), then the
 * issue and the take times of the first 32 ring chunks; after both, 16 words
 * per CTA for layer 1 (%globaltimer ns).
 * out_host receives min(max_records, available) records; *n_out is the
 * number written. Synchronises the model's stream. */
QW3_API int qw3_debug_read_trace(qw3_model *m, uint64_t *out_host, int32_t max_records, int32_t *n_out);

/* How decode calls of batch B run: *persistent = 1 when they use the
 * persistent decode-step kernel (one cooperative launch per step; then
 * *launches_per_step = 1), else 0 and *launches_per_step kernels per step. */
QW3_API int qw3_decode_plan(const qw3_model *m, int32_t B, int32_t *persistent,
                            int32_t *launches_per_step);

/* Block until the model's stream is idle; return and clear the first
 * device-side status recorded since the last call (QW3_ERR_NONFINITE for NaN
 * logits, QW3_ERR_TIMEOUT for an expired bounded wait), else QW3_OK. */
QW3_API int qw3_sync(qw3_model *m);

/* The model's stream as a cudaStream_t. */
QW3_API void *qw3_stream(const qw3_model *m);

QW3_API const char *qw3_status_string(int status);
/* Detail of the last error on this model (never NULL). */
QW3_API const char *qw3_last_error(const qw3_model *m);

/* ---- standalone Q8_0 entries on caller device buffers ----------------- */

/* Encode n f32 values (n % 32 == 0, else QW3_ERR_SHAPE) into n/32 Q8_0
 * blocks at blocks_dev (n/32*34 bytes), course 11.7: per block amax, d =
 * amax/127 (f32), inv_d = d ? 1/d : 0, q = clamp(round(x*inv_d), +-127) with
 * halves rounded away from zero, d stored as IEEE f16 (nearest even). A block
 * holding NaN or inf is written as all-zero bytes and, if status_dev is not
 * NULL, *status_dev is set to QW3_ERR_NONFINITE (the caller zeroes it first).
 * Asynchronous on `stream`. */
QW3_API int qw3_q8_0_quantize(const float *x_dev, int64_t n, void *blocks_dev,
                      int32_t *status_dev, void *stream);

/* Decode n values (n % 32 == 0) of Q8_0 blocks to f32: y = f32(d) * q. */
QW3_API int qw3_q8_0_dequantize(const void *blocks_dev, int64_t n, float *y_dev, void *stream);

/* y[b][r] = sum_k W[r][k] * x[b][k] for a raw Q8_0 matrix W [rows][cols/32]
 * (GGUF layout), x f32 [B][cols], y f32 [B][rows]; f32 accumulation.
 * 1 <= B <= 8, cols % 32 == 0. When cols % 256 == 0 and W and x are 16-byte
 * aligned (every row then starts 16-byte aligned) each row streams with
 * 128-bit loads; otherwise a slower path with 2-byte loads runs. */
QW3_API int qw3_q8_0_gemv(const void *W_dev, int32_t rows, int32_t cols,
                  const float *x_dev, int32_t B, float *y_dev, void *stream);

/* The pages' quantized matmul ("Model files and quantization", 11.9, the
 * dotBlocks step): each row x[b] is first encoded to Q8_0 per 32-block by
 * the 11.7 encoder (d = amax/127, codes rounded half away from zero, d kept
 * as f16), then y[b][r] = sum over blocks of (d_w * d_x) * (i32 dot of the
 * 32 weight and activation codes), f32. A block of x holding NaN or inf
 * makes the rows it touches NaN. Arguments as qw3_q8_0_gemv; cols % 256 == 0,
 * B * cols <= 49152, W and x 16-byte aligned (QW3_ERR_SHAPE /
 * QW3_ERR_INVALID_ARG otherwise). Asynchronous on `stream`. */
QW3_API int qw3_q8_0_gemv_q8act(const void *W_dev, int32_t rows, int32_t cols,
                        const float *x_dev, int32_t B, float *y_dev, void *stream);

/* ---- Q4_K ("Model files and quantization", 11.8) ------------------------
 * Block: 256 values in 144 bytes: f16 d, f16 dmin, 12 bytes packing eight
 * 6-bit sub-scales sc_j and eight 6-bit sub-mins m_j (GGUF layout), 128
 * bytes of 4-bit codes; value i of sub-block j = i/32 is
 * (d*sc_j)*q - dmin*m_j in f32. */

/* Encode n values (n % 256 == 0) to Q4_K. The pages give no encoding
 * algorithm; this one: per 32-value sub-block lo = min(0, min x),
 * S = (max x - lo)/15, O = -lo; d = max S/63, dmin = max O/63 as f16; sub-
 * scales, sub-mins (0..63) and codes (0..15) rounded half away from zero.
 * A block holding NaN or inf is written as zero bytes and, if status_dev is
 * not NULL, *status_dev = QW3_ERR_NONFINITE. x and blocks 16-byte aligned. */
QW3_API int qw3_q4_k_quantize(const float *x_dev, int64_t n, void *blocks_dev,
                      int32_t *status_dev, void *stream);

/* Decode n values (n % 256 == 0) of Q4_K blocks to f32. */
QW3_API int qw3_q4_k_dequantize(const void *blocks_dev, int64_t n, float *y_dev, void *stream);

/* y[b][r] = sum_k W[r][k] * x[b][k] for a raw Q4_K matrix W [rows][cols/256]
 * (GGUF layout), x f32 [B][cols], y f32 [B][rows]; f32 accumulation (a
 * sub-block adds d1 * sum(q x) - m1 * sum(x)). 1 <= B <= 8, cols % 256 == 0,
 * B * cols <= 49152; W and x 16-byte aligned. Asynchronous on `stream`. */
QW3_API int qw3_q4_k_gemv(const void *W_dev, int32_t rows, int32_t cols,
                  const float *x_dev, int32_t B, float *y_dev, void *stream);

/* ---- no-allocation variant ------------------------------------------- */

/* The same product as qw3_q8_0_gemv (y[b][r] = sum_k W[r][k] x[b][k], raw
 * Q8_0 blocks, f32 accumulation), computed split-K: the K range of each
 * 8-row group is spread over several CTAs whose partial sums the last CTA of
 * the group adds in a fixed order. The pages have no counterpart of this
 * call; it serves callers that must not allocate device memory during a
 * call (a serving loop whose memory a caching allocator has fully reserved,
 * or one that cannot take cudaFree's device-wide synchronisation).
 *
 * No allocation: the scratch (65536 row-group arrival counters and 1048576
 * f32 partial sums, 4.25 MiB) is a static device array of the library,
 * limiting rows to 524288 and B*rows to 1048576 (QW3_ERR_SHAPE beyond).
 * The counters must be zero when a call starts: static storage starts at
 * zero and every call leaves them at zero.
 * The first call on each device looks up the scratch address
 * (cudaGetSymbolAddress, which can load the module) and keeps it for the
 * life of the process; make that first call before any stream capture, and
 * do not call this entry on a device after cudaDeviceReset (the kept
 * address belongs to the context that was reset).
 * Calls that overlap on one device (two streams, or two threads without
 * ordering) share the scratch and race: order them on one stream.
 * Arguments as qw3_q8_0_gemv, except that x_dev must be 8-byte aligned.
 * rows == 0 is a no-op; cols == 0 writes zeros. Asynchronous on `stream`. */
QW3_API int qw3_q8_0_gemv_splitk_noalloc(const void *W_dev, int32_t rows, int32_t cols,
                                         const float *x_dev, int32_t B, float *y_dev,
                                         void *stream);

/* ---- The dense contraction on the tensor cores ----------------------------
 * The product prefill and large batches run ("A transformer from scratch",
 * 12.3: every linear layer applies to all rows of a chunk at once), as one
 * call: y[m][r] = sum_k W[r][k] * x[m][k] for raw Q8_0 W [rows][cols/32
 * blocks] ("Model files and quantization", 11.6) and f32 x [M][cols], y f32
 * [M][rows]. tcgen05 MMAs on fp16 hi/lo operand pairs, each row of W and of x
 * first multiplied by its own power of two (largest magnitude into
 * [2^14, 2^15)); f32 accumulation; results within f32 reassociation error of
 * the exact product.
 *
 * Returns the workspace bytes qw3_q8_0_gemm needs for these sizes, or -1 if
 * a size is negative or cols % 64 != 0. */
QW3_API int64_t qw3_q8_0_gemm_workspace_bytes(int32_t rows, int32_t cols, int32_t M);

/* W 2-byte aligned, x and the workspace 16-byte aligned, y 4-byte aligned;
 * workspace_bytes at least qw3_q8_0_gemm_workspace_bytes(rows, cols, M)
 * (QW3_ERR_INVALID_ARG otherwise; QW3_ERR_SHAPE if cols % 64 != 0). The
 * caller owns every buffer; the workspace must not be used by another call
 * until this one has completed on `stream`. rows == 0 or M == 0 is a no-op;
 * cols == 0 writes zeros. Asynchronous on `stream`. */
QW3_API int qw3_q8_0_gemm(const void *W_dev, int32_t rows, int32_t cols, const float *x_dev,
                          int32_t M, float *y_dev, void *workspace_dev, int64_t workspace_bytes,
                          void *stream);

#ifdef __cplusplus
}
#endif
#endif /* QW3_H */
