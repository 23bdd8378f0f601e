// Host-side plumbing shared by the translation units of the library: workspace
// layout, launch geometry and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace pi {

// Workspace regions, byte offsets from the workspace base (all 256-aligned).
struct WsLayout {
    size_t ctrl;      // WsCtrl
    size_t status;    // scan tile status words, one per 32 neurons
    size_t h;         // predictor hidden [batch][rank] fp32
    size_t idx;       // internal active list [d_ff] int32
    size_t nact;      // internal active count (int32)
    size_t candb;     // one-kernel layer step: candidate biases [d_ff] fp32
    size_t qent;      // one-kernel layer step: work-queue entries [d_ff] u64
    size_t fcount;    // one-kernel layer step: per-CTA active counts [1024] u32
    size_t act;       // union path: activations, [ceil(d_ff/16)][4][8][4] fp32 (mma B-operand order)
    size_t xf;        // union path: x as fp16 hi/lo mma fragments, [ceil(d_model/32)][2][32][4] u32
    size_t uctl;      // union path: x exponents int[8], max |a| bits u32[8], h exponents int[8]
    size_t xfh;       // union path: h as fp16 hi/lo mma fragments, [ceil(rank/32)][2][32][4] u32
    size_t umask;     // union path: predicted union mask bytes [d_ff]
    size_t zbuf;      // union path: per-tile partial sums [ceil(d_ff/16)][2][16][8] fp32 (kept zero)
    size_t ucnt;      // union path: per-tile arrival counts [ceil(d_ff/16)] u32 (kept zero)
    size_t total;
};

WsLayout ws_layout(int d_model, int d_ff, int rank, int batch);
size_t compact_ws_bytes(int n);

int sm_count();  // of the current device (cached per device)

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- predictor + compaction (predict.cu) ------------------------------------------
struct PredParams {
    const void *p2;
    const float *p_bias;
    const float *h;
    int B, r, F;
    float tau;
    int prefix;           // neurons [0, prefix) are active whatever their logits
    float *logits;        // [B][F] or null
    uint8_t *mask;        // [F] or null
    int *idx;
    int *n_active;
    int cap;
    WsCtrl *ctrl;
    unsigned long long *status;
    float *y;             // when non-null: y = b_down + residual is written here
    const float *residual;
    const float *b_down;
    int d;
};

cudaError_t launch_pred_hidden(int ptype, const void *p1, const float *x, int B, int d, int r, float *h,
                               const void *p2, size_t p2_bytes, const float *p_bias, const float *b_act, int F,
                               cudaStream_t s);
cudaError_t launch_pred_logits(int ptype, const PredParams &p, cudaStream_t s);
cudaError_t launch_compact(const uint8_t *mask, int n, int *idx, int *count, int cap, WsCtrl *ctrl,
                           unsigned long long *status, cudaStream_t s);

// ---- sparse FFN (sparse_ffn.cu, union_mma.cu) --------------------------------------
struct SparseParams {
    const uint8_t *w_act;   // gate (gated) or up (non-gated)
    const uint8_t *w_up;    // up, gated only
    const uint8_t *w_down;
    const float *b_act;
    const float *x;         // [B][d]
    const int *idx;
    const int *n_active;
    float *y;               // [B][d], already holding b_down + residual
    WsCtrl *ctrl;
    float *act_ws;          // union path: activations in fragment order
    uint32_t *xf;           // union path: x fragments
    int *uexp;              // union path: per-token exponents of x [8]
    unsigned *amax;         // union path: per-token max |a| (float bits) [8]
    float *zbuf;            // union path: per-tile partial sums
    unsigned *ucnt;         // union path: per-tile arrival counts
    int xf_ready;           // union path: xf already holds x's fragments (skip the prep kernel)
    int d, F, act, B;
    // The same up kernel also runs the batched predictor (idx and n_active null:
    // every row of w_act in order, F rows of d weights):
    float *out_h;           // hidden epilogue: h [B][F]
    const float *p_bias;    // logits epilogue
    float tau;
    int prefix;             // logits epilogue: neurons [0, prefix) always in the mask
    float *out_logits;      // logits epilogue: [B][F] or null
    uint8_t *out_mask;      // logits epilogue: union mask bytes [F]
};

// Batched (2..8 tokens) predictor on tensor cores, fp16 predictor weights.
struct UnionPredArgs {
    const void *p1, *p2;
    const float *p_bias;
    float tau;
    int prefix;             // neurons [0, prefix) always in the mask
    const float *x;
    int B, d, r, F;
    float *h;               // [B][r]
    float *logits;          // [B][F] or null
    uint8_t *mask;          // [F]
    uint32_t *xf_x, *xf_h;  // operand fragments of x and of h
    int *uexp_x, *uexp_h;
    unsigned *amax;
    float *zbuf;
    unsigned *ucnt;
    WsCtrl *ctrl;
};
cudaError_t launch_pred_union(const UnionPredArgs &a, cudaStream_t s);

cudaError_t launch_sparse_b1(int wtype, int gated, const SparseParams &p, cudaStream_t s);
cudaError_t launch_sparse_union(int wtype, int gated, const SparseParams &p, cudaStream_t s);

// ---- one token through one layer in one kernel (layer_fused.cu) -------------------
struct LayerB1Args {
    int wtype, ptype, gated, act;
    const void *p1, *p2;
    const float *p_bias;
    float tau;
    int r;
    const void *w_up, *w_gate, *w_down;
    const float *b_act, *b_down;
    const float *x, *residual;
    const float *x_prev, *y_prev;  // chained input (x unused): x = (x_prev + y_prev) / rms, written to x_out
    float *x_out;
    float *y;
    int *idx_out, *n_active;
    int *cand;              // [F] workspace
    float *cand_bias;       // [F] workspace
    unsigned long long *qent;  // [F] workspace
    float *h;               // [r] workspace
    unsigned *status;       // [#SMs] workspace
    WsCtrl *ctrl;
    int d, F;
    int prefix;             // neurons [0, prefix) always active (no predictor rows read for them)
};
bool fused_layer_supported(int wtype, int ptype, int d, int F, int r, int prefix);
cudaError_t launch_layer_b1(const LayerB1Args &a, cudaStream_t s);

// ---- small kernels (aux.cu) ------------------------------------------------------
cudaError_t launch_init_y(float *y, const float *b_down, const float *residual, int B, int d,
                          int *iota_idx, int *iota_n, int iota_count, cudaStream_t s);
cudaError_t launch_quantize_q4_0(const void *src, int src_type, int64_t rows, int64_t cols, void *dst,
                                 cudaStream_t s);
cudaError_t launch_fire_counts(int wtype, const void *w, const float *b, const float *X, int T, int d, int F,
                               int *counts, cudaStream_t s);
cudaError_t launch_permute_rows(const void *src, void *dst, int64_t rows, int64_t row_bytes, const int *perm,
                                cudaStream_t s);
cudaError_t launch_rms_residual(const float *x, const float *y, int B, int d, float *out, cudaStream_t s);

}  // namespace pi
