// internal.h -- host-side declarations shared by the sffn translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "sffn.h"

namespace sffn {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }
// Every workspace starts with a control block of kControlBytes:
//   byte 0  int32  device error word (any entry point)
//   byte 4  uint32 decode grid barrier: arrivals, never reset (wraps)
//   byte 8  uint32 decode grid barrier: arrivals before the current call
// Only decode writes bytes 4 .. 11; a zero-filled control block is a valid
// start, and every call leaves it valid for the next one.
constexpr size_t kControlBytes = 16;
constexpr size_t kCtlBar = 4;

// SM count of the current device (cached per device).
int device_sm_count();
// Opt-in shared memory per block of the current device (cached per device).
int device_smem_optin();
// Opt a kernel into more than 48 KB of dynamic shared memory (once per device).
cudaError_t set_max_smem(const void *kernel, int bytes);

// Launch with programmatic stream serialisation (PDL) so the kernel may begin
// while its predecessor drains; kernels call griddepcontrol.wait before they
// touch any memory written earlier in the stream.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Decode
// ---------------------------------------------------------------------------

struct DecodePlan {
    int nb;       // tokens
    int d, F;
    int C, R;     // gate kernel: C CTAs, each owning R consecutive neurons (a "chunk")
    int G2;       // up/down kernel CTAs (one partial output per CTA)
    int nlists;   // nb per-token lists (+1 union list when nb > 1)
    int list_u;   // index of the list the up/down kernel walks
    // workspace offsets (bytes)
    size_t off_err, off_cnt, off_lidx, off_lh, off_aeff, off_uval, off_score, off_mask, off_part, total;
};

DecodePlan make_decode_plan(int B, int d, int F);

// Every host-side check sffn_decode makes before it looks at the workspace, in
// the same order and with the same status codes.
sffn_status validate_decode_call(const void *x, int B, const sffn_ffn_weights *w, int mode, int score, float param,
                                 const void *out, const int32_t *active_idx, const int32_t *n_active);

struct DecodeCall {
    const void *x;
    const sffn_ffn_weights *w;
    int B, mode, score;
    float param;
    void *out;
    int32_t *active_idx, *n_active;
    void *ws;
    float *scores_only;  // non-null: sffn_gate_scores (write scores, nothing else)
    const int32_t *core; // keep-ratio: the layer's core set (sffn_decode_tiered), or null
    int n_core;
};

sffn_status run_decode(const DecodeCall &c, const DecodePlan &p, cudaStream_t s);
// Tensor-core decode (decode_tc.cu): int4-g64 at any B and bf16 with B >= 2,
// exact or threshold-on-gate-score rules; and the dense layer (dense = true).
bool decode_tc_shape_ok(const sffn_ffn_weights *w, const DecodePlan &p);
bool decode_tc_eligible(const DecodeCall &c, const DecodePlan &p);
sffn_status run_decode_tc(const DecodeCall &c, const DecodePlan &p, cudaStream_t s, bool dense);
// One-token int4 decode on the CUDA cores (decode_q1.cu); dense = every neuron.
bool decode_q1_eligible(const DecodeCall &c, const DecodePlan &p, bool dense);
// Gate-and-up scores (with a_j and u_j) of one token with int4-g64 weights
// (decode_q1.cu): the keep-ratio rule's first step.
bool scores_q1_eligible(const sffn_ffn_weights *w, const DecodePlan &p);
cudaError_t run_scores_q1(const sffn_ffn_weights *w, const void *x, const DecodePlan &p, float *score, float *aeff,
                          float *uval, cudaStream_t s);
sffn_status run_decode_q1(const DecodeCall &c, const DecodePlan &p, cudaStream_t s, bool dense);
sffn_status run_down_norms(const sffn_ffn_weights *w, float *norms, cudaStream_t s);
// One-token finish over per-chunk partials and lists in the workspace (part
// [C, d], cnt [C], lidx [C, R]): the fixed-order reduction and the list writes.
sffn_status run_reduce_chunks(const DecodeCall &c, const DecodePlan &p, cudaStream_t s);
// Core set of a keep-ratio tier from calibration scores (tiers.cu).
size_t tier_core_workspace(int N, int F);
sffn_status run_tier_core_set(const float *scores, int N, int F, int k, int c, int32_t *core, void *ws,
                              cudaStream_t s);
// MoE routing and block budget (moe.cu).
constexpr int kMoeMaxExperts = 512;   // router width
constexpr int kMoeMaxK = 8;           // experts per token
constexpr int kMoeMaxBlocks = 8192;   // budget blocks per sequence
constexpr int kMoeMaxBuckets = 8;
struct MoeRouteArgs {
    const float *logits;  // [T, E]
    int T, E, cap, kmax;
    float mass;
    int n_buckets;
    int buckets[kMoeMaxBuckets];  // ascending
    int32_t *k_out, *experts;     // [T], [T, kmax]
    float *weights;               // [T, kmax]
};
sffn_status run_moe_route(const MoeRouteArgs &a, cudaStream_t s);
size_t moe_budget_workspace(int L, int d);
sffn_status run_moe_block_budget(const void *y_attn, int L, int d, float mass, float min_ratio, float max_ratio,
                                 int block, int32_t *token_idx, int32_t *n_tokens, int32_t *ranges,
                                 int32_t *n_ranges, void *ws, cudaStream_t s);
// Decode with the low-rank gate predictor (predict.cu): one token, bf16 / fp32.
sffn_status run_decode_predicted(const DecodeCall &c, const DecodePlan &p, const float *factor_a,
                                 const float *factor_b, int rank, float alpha, cudaStream_t s);

// ---------------------------------------------------------------------------
// Token selection / prefill
// ---------------------------------------------------------------------------

struct SelectPlan {
    int L, d;
    size_t off_err, off_norms, off_flag, off_state, off_hist, off_cmax, total;
};
SelectPlan make_select_plan(int L, int d);
sffn_status run_token_select(const void *y_attn, int L, int d, float mass_thresh, int recent_n, int min_keep,
                             int32_t *sel_idx, int32_t *n_sel, void *ws, const SelectPlan &p, cudaStream_t s);

struct PrefillPlan {
    int L, d, F;
    size_t off_err, off_ysel, off_h, total;
};
PrefillPlan make_prefill_plan(int L, int d, int F);
sffn_status run_prefill(const void *x, const void *y_attn, int L, const sffn_ffn_weights *w, const int32_t *sel_idx,
                        const int32_t *n_sel, void *out, void *ws, const PrefillPlan &p, cudaStream_t s);

}  // namespace sffn
