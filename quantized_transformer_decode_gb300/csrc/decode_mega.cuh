// Parameters of the persistent batch-1 decode kernel (decode_mega.cu).
#pragma once

#include "qw3_internal.cuh"

namespace qw3 {

struct MegaParams {
    // Per-layer weights in the layouts the kernel streams; layer l of each
    // array sits at base + l * stride (bytes).
    const uint8_t *qkv0;      // rows grouped per KV head g: [G query heads | k | v], tiles 8 x H, row-group-major
    const uint8_t *o0;        // W_o, tiles 8 x (G*head_dim), k-tile-major (one k-tile per KV head group)
    const uint8_t *down0;     // W_down, column-partitioned over the NC clusters (see k_repack_colpart)
    size_t mstride;
    const uint8_t *gu0;       // gate/up rows interleaved (2i gate, 2i+1 up), tiles 8 x H, row-group-major
    const float *attn_norm0, *q_norm0, *k_norm0, *ffn_norm0;
    size_t wstride;
    QMat embd, out;           // token embedding, lm_head (row-group-major, kt = H)
    const float *out_norm;
    const float2 *rope;       // [max_seq_len][hd/2] (cos, sin)
    float *kv;                // [layer][seq][K|V][kv_head][capacity][hd]
    size_t seq_stride, kvsel_stride, head_stride, layer_stride;  // floats
    int L, H, I, V, hd, G;
    int NA;                   // attention clusters (= n_kv_heads)
    int NC;                   // all clusters (FFN, lm_head)
    int CS;                   // CTAs per cluster
    int NCTA;                 // NC * CS
    int RG, RPC;              // QKV rows per KV head group, per CTA
    int ORPC;                 // o_proj / down rows per CTA (H / CS)
    int o_groups;             // H / 8
    int act_units;            // I / 32
    int maxpos;               // score slots per head (>= positions per CTA + 1)
    int o_act_cap;            // capacity (values) of the channel plane buffer
    float eps, scale;
    int seq, pos0, n_steps;
    const int32_t *first_token;   // device [1]
    int32_t *hist;                // nullable device [n_steps]
    float *logits;                // nullable device [V] (written every step)
    int32_t *argmax_out;          // nullable device [1] (last step)
    float *opart;                 // [NA][H] o_proj partials
    float *dpart;                 // [NC][H] down partials
    unsigned int *gctr;           // grid arrival counter, zero at launch
    unsigned long long *key;      // [2] argmax keys, zero at launch
    int32_t *status;
    unsigned long long *trace;    // nullable: timeline of two CTAs (last step) + per-CTA wait totals
    uint32_t SB;                  // ring slot bytes
    int NS;                       // ring slots
    // shared-memory layout (byte offsets)
    uint32_t o_bar, o_x, o_xn, o_wbuf, o_qkvpub, o_qkv, o_scores, o_apub, o_vred, o_oall, o_guout, o_actpub, o_act, o_red,
        o_ring;
};

constexpr int kMegaMaxSmem = 227 * 1024;
constexpr int kMegaCS = 8;

size_t mega_smem_bytes(const MegaParams &P);
cudaError_t configure_mega();
bool mega_supported_heads(int hd, int G);
cudaError_t mega_max_clusters(const MegaParams &P, int *n);
cudaError_t launch_mega(const MegaParams &P, cudaStream_t s);
cudaError_t launch_repack_colpart(const uint8_t *raw, int rows, int cols, int NC, uint8_t *dst, cudaStream_t s);

}  // namespace qw3
