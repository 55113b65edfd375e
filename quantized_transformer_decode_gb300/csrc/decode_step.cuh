// Parameters of the persistent batch-1 decode-step kernel (decode_step.cu).
#pragma once

#include "qw3_internal.cuh"

namespace qw3 {

// One launch computes one greedy decode step at batch 1: the embedding of
// the current token, every layer, the final norm, the lm_head and the argmax
// ("A transformer from scratch", 12.3-12.6). Its CTAs (one per SM, all
// resident: cooperative launch) hand activation vectors to each other
// through global f32 buffers guarded by arrival counters.
struct StepParams {
    // model shape
    int L, H, I, V, nh, nkv, hd, G, qkv_w;
    float eps, scale;
    const LayerDev *layers;     // device array [L]
    LayerDev L0;                // layer 0; layer l's matrices and norms sit lstride bytes further per layer
    size_t lstride;
    QMat embd, out;             // token embedding; lm_head (== embd when tied)
    const float *out_norm;
    const float2 *rope;         // [max_seq_len][hd/2] (cos, sin)
    float *kv;                  // [layer][seq][K|V][kv_head][capacity][hd]
    size_t seq_stride, kvsel_stride, head_stride, layer_stride;   // floats
    // step state (device memory)
    const int32_t *seq_ids;     // [1]
    int32_t *pos;               // [1]: position of the new token; +1 at the end
    int32_t *tok;               // [1]: token in, argmax out
    int32_t *step_ctr;          // history index (incremented at the end)
    const DecodeIO *io;         // logits / argmax / history outputs
    unsigned *epoch;            // step epoch (scopes the abort word); +1 at the end
    unsigned *abort_word;       // == epoch once a wait on other CTAs gave up
    unsigned long long *argmax_key;
    unsigned *done_counter;
    int32_t *status;
    // exchange buffers (f32) and their arrival counters (128 bytes apart:
    // x [8 split], o [8], act [8], qkv per kv head, partials per kv head;
    // zero at the start of every step)
    float *xb;                  // [H] residual stream
    float *qkvb;                // [qkv_w]
    float *partb;               // [nkv * S][G][hd + 2] attention partials
    float *ob;                  // [nh * hd] attention output
    float *actb;                // [I] SwiGLU output
    unsigned *ctrs;             // [24 + 2 nkv][32]
    unsigned cnt_x[8], cnt_o[8], cnt_act[8];   // writers behind each split counter
    unsigned cnt_qkv[64];       // projection writers of each kv head's rows
    uint64_t wait_ns;           // limit of a wait on another CTA's data
    unsigned long long *trace;  // nullable: [2 CTAs][phases][2] timestamps
    // plan
    int NCTA;                   // CTAs (one per SM)
    int S;                      // attention units per kv head
    int LC;                     // activation columns per lane in a dot task (8 or 16)
    int NS;                     // ring slots
    uint32_t SB;                // ring slot bytes
    int CP;                     // cached positions per KV chunk
    int kmax;                   // widest activation vector (max of H, I, nh * hd)
    uint32_t o_misc, o_xown, o_planes, o_scales, o_red, o_ring;   // shared-memory offsets
    uint32_t smem;
};

constexpr int kStepConsumerWarps = 16;
// Largest per-SM share of one layer's weights for which batch-1 decode uses
// the step kernel (0.6B geometry: ~110 KB; 8B: ~1.4 MB).
constexpr size_t kStepMaxLayerBytesPerSm = 512 * 1024;
constexpr int kStepThreads = (kStepConsumerWarps + 1) * 32;

// Phases per layer (trace records).
constexpr int kStepPhases = 6;
// Arrival counters of a model with nkv kv heads.
inline int step_counters(int nkv) { return 24 + 2 * nkv; }

// True when the persistent step kernel supports the model's shape.
bool step_supported(const qw3_config &c);
// Fill the plan part of P (NCTA, S, LC, ring, shared-memory layout) for the
// current device from the shape fields and layer 0's matrices (every layer
// has the same); false if the layout does not fit.
bool step_plan(StepParams &P, const LayerDev &L0);
cudaError_t configure_step();
cudaError_t launch_step(const StepParams &P, cudaStream_t s);

}  // namespace qw3
