// api.cu -- extern "C" entry points of libsffn.so: argument validation,
// workspace layout and dispatch to the kernels.  See include/sffn.h.
#include <math.h>
#include <mutex>

#include "common.cuh"
#include <cmath>

#include "internal.h"

namespace sffn {

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
int g_smem_optin[kMaxDevices];
std::mutex g_mu;

struct SmemEntry {
    const void *fn;
    int dev;
    int bytes;
};
SmemEntry g_smem[512];
int g_nsmem = 0;
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

int device_smem_optin() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_optin[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
        g_smem_optin[dev] = n;
    }
    return g_smem_optin[dev];
}

// The attribute is set whatever the size: a kernel's static shared memory
// counts against the same 48 KB default as its dynamic shared memory.
cudaError_t set_max_smem(const void *kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_nsmem; ++i)
        if (g_smem[i].fn == kernel && g_smem[i].dev == dev && g_smem[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < g_nsmem; ++i)
        if (g_smem[i].fn == kernel && g_smem[i].dev == dev) {
            g_smem[i].bytes = bytes;
            return cudaSuccess;
        }
    if (g_nsmem < 512) g_smem[g_nsmem++] = {kernel, dev, bytes};
    return cudaSuccess;
}

}  // namespace sffn

using namespace sffn;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared checks of the weight struct.  `need_norms`: score-based modes.
sffn_status check_weights(const sffn_ffn_weights *w, bool need_norms) {
    if (!w) return SFFN_ERR_INVALID_ARG;
    if (w->wdtype < SFFN_F32 || w->wdtype > SFFN_INT4_G64) return SFFN_ERR_INVALID_ARG;
    if (w->act != SFFN_ACT_RELU && w->act != SFFN_ACT_SILU) return SFFN_ERR_INVALID_ARG;
    if (w->d_model < 8 || w->d_model > 8192 || w->d_ff < 1 || w->d_ff > 65536) return SFFN_ERR_SHAPE;
    if (w->d_model % 8 != 0) return SFFN_ERR_SHAPE;
    if (w->wdtype == SFFN_INT4_G64 && w->d_model % 64 != 0) return SFFN_ERR_SHAPE;
    if (!w->w_gate || !w->w_up || !w->w_downT) return SFFN_ERR_INVALID_ARG;
    if (!aligned16(w->w_gate) || !aligned16(w->w_up) || !aligned16(w->w_downT)) return SFFN_ERR_ALIGNMENT;
    if (w->wdtype == SFFN_INT4_G64) {
        if (!w->s_gate || !w->s_up || !w->s_downT) return SFFN_ERR_INVALID_ARG;
        if (!aligned16(w->s_gate) || !aligned16(w->s_up) || !aligned16(w->s_downT)) return SFFN_ERR_ALIGNMENT;
    }
    if (need_norms && !w->down_norms) return SFFN_ERR_INVALID_ARG;
    if (w->b_gate && !aligned16(w->b_gate)) return SFFN_ERR_ALIGNMENT;
    if (w->down_norms && !aligned16(w->down_norms)) return SFFN_ERR_ALIGNMENT;
    return SFFN_OK;
}

sffn_status check_ws(void *ws, size_t bytes, size_t need) {
    if (!ws) return SFFN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return SFFN_ERR_WORKSPACE;
    if (bytes < need) return SFFN_ERR_WORKSPACE;
    return SFFN_OK;
}

sffn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA; }

sffn_status check_decode_args(const void *x, int B, const sffn_ffn_weights *w, int mode, int score, float param) {
    if (!x) return SFFN_ERR_INVALID_ARG;
    if (mode < SFFN_MODE_EXACT || mode > SFFN_MODE_KEEP_RATIO) return SFFN_ERR_INVALID_ARG;
    if (score != SFFN_SCORE_GATE && score != SFFN_SCORE_GATE_UP) return SFFN_ERR_INVALID_ARG;
    sffn_status st = check_weights(w, mode != SFFN_MODE_EXACT);
    if (st != SFFN_OK) return st;
    if (B < 1 || B > 8) return SFFN_ERR_SHAPE;
    if (w->d_model > 4096) return SFFN_ERR_SHAPE;
    if (!aligned16(x)) return SFFN_ERR_ALIGNMENT;
    if (mode == SFFN_MODE_THRESHOLD && !(param >= 0.f) ) return SFFN_ERR_INVALID_ARG;
    if (mode == SFFN_MODE_KEEP_RATIO && !(param > 0.f && param <= 1.f)) return SFFN_ERR_INVALID_ARG;
    if (w->wdtype == SFFN_INT4_G64) {
        if (w->d_model % 512 != 0) return SFFN_ERR_SHAPE;  // a row's scales: a 16-byte multiple
    }
    return SFFN_OK;
}

}  // namespace

namespace sffn {

sffn_status validate_decode_call(const void *x, int B, const sffn_ffn_weights *w, int mode, int score, float param,
                                 const void *out, const int32_t *active_idx, const int32_t *n_active) {
    sffn_status st = check_decode_args(x, B, w, mode, score, param);
    if (st != SFFN_OK) return st;
    if (!out || !active_idx || !n_active) return SFFN_ERR_INVALID_ARG;
    if (!aligned16(out)) return SFFN_ERR_ALIGNMENT;
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    return SFFN_OK;
}

}  // namespace sffn

extern "C" {

const char *sffn_status_string(sffn_status s) {
    switch (s) {
    case SFFN_OK: return "ok";
    case SFFN_ERR_INVALID_ARG: return "invalid argument";
    case SFFN_ERR_SHAPE: return "unsupported shape";
    case SFFN_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case SFFN_ERR_UNSUPPORTED: return "unsupported combination or device";
    case SFFN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SFFN_ERR_CUDA: return "CUDA error";
    case SFFN_ERR_TIMEOUT: return "device-side wait timed out";
    case SFFN_ERR_DEVICE: return "device-side contract violation";
    }
    return "unknown status";
}

size_t sffn_workspace_size(int which, int n, const sffn_ffn_weights *w) {
    if (which == 0) {
        if (!w || n < 1 || n > 8 || w->d_model < 8 || w->d_ff < 1 || w->d_ff > 65536) return 0;
        if (device_sm_count() <= 0) return 0;
        return make_decode_plan(n, w->d_model, w->d_ff).total;
    }
    if (which == 1) {
        if (n < 1 || n > (1 << 20)) return 0;
        return make_select_plan(n, w ? w->d_model : 0).total;
    }
    if (which == 2) {
        if (!w || n < 1 || n > (1 << 20)) return 0;
        return make_prefill_plan(n, w->d_model, w->d_ff).total;
    }
    return 0;
}

sffn_status sffn_down_norms(const sffn_ffn_weights *w, float *norms, sffn_stream_t stream) {
    sffn_status st = check_weights(w, false);
    if (st != SFFN_OK) return st;
    if (!norms) return SFFN_ERR_INVALID_ARG;
    st = run_down_norms(w, norms, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_decode(const void *x, int B, const sffn_ffn_weights *w, int mode, int score, float param, void *out,
                        int32_t *active_idx, int32_t *n_active, void *workspace, size_t ws_bytes,
                        sffn_stream_t stream) {
    sffn_status st = validate_decode_call(x, B, w, mode, score, param, out, active_idx, n_active);
    if (st != SFFN_OK) return st;
    DecodePlan p = make_decode_plan(B, w->d_model, w->d_ff);
    st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    DecodeCall c = {};
    c.x = x;
    c.w = w;
    c.B = B;
    c.mode = mode;
    c.score = score;
    c.param = param;
    c.out = out;
    c.active_idx = active_idx;
    c.n_active = n_active;
    c.ws = workspace;
    c.scores_only = nullptr;
    st = run_decode(c, p, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_decode_dense(const void *x, int B, const sffn_ffn_weights *w, void *out, void *workspace,
                              size_t ws_bytes, sffn_stream_t stream) {
    sffn_status st = check_decode_args(x, B, w, SFFN_MODE_EXACT, SFFN_SCORE_GATE, 0.f);
    if (st != SFFN_OK) return st;
    if (!out) return SFFN_ERR_INVALID_ARG;
    if (!aligned16(out)) return SFFN_ERR_ALIGNMENT;
    if (w->wdtype != SFFN_BF16 && w->wdtype != SFFN_INT4_G64) return SFFN_ERR_UNSUPPORTED;
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    DecodePlan p = make_decode_plan(B, w->d_model, w->d_ff);
    DecodeCall c = {};
    c.x = x;
    c.w = w;
    c.B = B;
    c.mode = SFFN_MODE_EXACT;
    c.out = out;
    c.ws = workspace;
    const bool q1 = decode_q1_eligible(c, p, true);
    if (!q1 && !decode_tc_shape_ok(w, p)) return SFFN_ERR_UNSUPPORTED;
    st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    st = q1 ? run_decode_q1(c, p, (cudaStream_t)stream, true) : run_decode_tc(c, p, (cudaStream_t)stream, true);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_decode_predicted(const void *x, const sffn_ffn_weights *w, const float *factor_a,
                                  const float *factor_b, int rank, float alpha, void *out, int32_t *active_idx,
                                  int32_t *n_active, void *workspace, size_t ws_bytes, sffn_stream_t stream) {
    sffn_status st = check_decode_args(x, 1, w, SFFN_MODE_EXACT, SFFN_SCORE_GATE, 0.f);
    if (st != SFFN_OK) return st;
    if (!out || !active_idx || !n_active) return SFFN_ERR_INVALID_ARG;
    if (!aligned16(out)) return SFFN_ERR_ALIGNMENT;
    if (w->wdtype != SFFN_BF16 && w->wdtype != SFFN_F32) return SFFN_ERR_UNSUPPORTED;
    if (!(alpha >= 0.f)) return SFFN_ERR_INVALID_ARG;  // also rejects NaN
    if (!std::isinf(alpha)) {
        if (!factor_a || !factor_b) return SFFN_ERR_INVALID_ARG;
        if (rank < 1 || rank > w->d_ff || rank > 4096) return SFFN_ERR_SHAPE;
        if (!aligned16(factor_b)) return SFFN_ERR_ALIGNMENT;
    }
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    DecodePlan p = make_decode_plan(1, w->d_model, w->d_ff);
    st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    DecodeCall c = {};
    c.x = x;
    c.w = w;
    c.B = 1;
    c.mode = SFFN_MODE_EXACT;
    c.score = SFFN_SCORE_GATE;
    c.out = out;
    c.active_idx = active_idx;
    c.n_active = n_active;
    c.ws = workspace;
    st = run_decode_predicted(c, p, factor_a, factor_b, rank, alpha, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_decode_tiered(const void *x, int B, const sffn_ffn_weights *w, int score, float keep_ratio,
                               const int32_t *core_idx, int n_core, void *out, int32_t *active_idx, int32_t *n_active,
                               void *workspace, size_t ws_bytes, sffn_stream_t stream) {
    sffn_status st = validate_decode_call(x, B, w, SFFN_MODE_KEEP_RATIO, score, keep_ratio, out, active_idx, n_active);
    if (st != SFFN_OK) return st;
    if (n_core < 0 || n_core > w->d_ff) return SFFN_ERR_SHAPE;
    if (n_core > 0 && !core_idx) return SFFN_ERR_INVALID_ARG;
    DecodePlan p = make_decode_plan(B, w->d_model, w->d_ff);
    st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    DecodeCall c = {};
    c.x = x;
    c.w = w;
    c.B = B;
    c.mode = SFFN_MODE_KEEP_RATIO;
    c.score = score;
    c.param = keep_ratio;
    c.out = out;
    c.active_idx = active_idx;
    c.n_active = n_active;
    c.ws = workspace;
    c.core = n_core > 0 ? core_idx : nullptr;
    c.n_core = n_core;
    st = run_decode(c, p, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

size_t sffn_tier_core_workspace_size(int n_calib, int d_ff) {
    if (n_calib < 1 || n_calib > (1 << 16) || d_ff < 1 || d_ff > 65536) return 0;
    return tier_core_workspace(n_calib, d_ff);
}

sffn_status sffn_tier_core_set(const float *calib_scores, int n_calib, int d_ff, int k, int n_core, int32_t *core_idx,
                               void *workspace, size_t ws_bytes, sffn_stream_t stream) {
    if (!calib_scores || (n_core > 0 && !core_idx)) return SFFN_ERR_INVALID_ARG;
    if (n_calib < 1 || n_calib > (1 << 16) || d_ff < 1 || d_ff > 65536) return SFFN_ERR_SHAPE;
    if (k < 1 || k > d_ff || n_core < 0 || n_core > d_ff) return SFFN_ERR_INVALID_ARG;
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    sffn_status st = check_ws(workspace, ws_bytes, tier_core_workspace(n_calib, d_ff));
    if (st != SFFN_OK) return st;
    st = run_tier_core_set(calib_scores, n_calib, d_ff, k, n_core, core_idx, workspace, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

int sffn_moe_progressive_k(int layer) {
    // depth ranges and their expert counts; past the last range its count holds
    static const int kRanges[3][3] = {{0, 15, 6}, {16, 39, 5}, {40, 60, 4}};
    if (layer < 0) return -1;
    for (const auto &r : kRanges)
        if (layer >= r[0] && layer <= r[1]) return r[2];
    return kRanges[2][2];
}

sffn_status sffn_moe_route(const float *logits, int T, int E, int cap, float mass, const int32_t *buckets,
                           int n_buckets, int kmax, int32_t *k_out, int32_t *experts, float *weights,
                           sffn_stream_t stream) {
    if (!logits || !k_out || !experts || !weights || !buckets) return SFFN_ERR_INVALID_ARG;
    if (T < 0 || E < 1 || E > kMoeMaxExperts) return SFFN_ERR_SHAPE;
    if (cap < 1 || cap > E || cap > kMoeMaxK || kmax < cap || kmax > kMoeMaxK) return SFFN_ERR_SHAPE;
    if (n_buckets < 1 || n_buckets > kMoeMaxBuckets || !(mass == mass)) return SFFN_ERR_INVALID_ARG;
    MoeRouteArgs a = {};
    for (int i = 0; i < n_buckets; ++i) {
        if (buckets[i] < 1 || buckets[i] > kMoeMaxK || (i > 0 && buckets[i] <= buckets[i - 1]))
            return SFFN_ERR_INVALID_ARG;
        a.buckets[i] = buckets[i];
    }
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    if (T == 0) return SFFN_OK;
    a.logits = logits;
    a.T = T;
    a.E = E;
    a.cap = cap;
    a.kmax = kmax;
    a.mass = mass;
    a.n_buckets = n_buckets;
    a.k_out = k_out;
    a.experts = experts;
    a.weights = weights;
    sffn_status st = run_moe_route(a, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

size_t sffn_moe_budget_workspace_size(int L, int d_model) {
    if (L < 1 || L > (1 << 20) || d_model < 8 || d_model > 65536 || d_model % 8 != 0) return 0;
    return moe_budget_workspace(L, d_model);
}

sffn_status sffn_moe_block_budget(const void *y_attn, int L, int d_model, float mass, float min_ratio,
                                  float max_ratio, int block, int32_t *token_idx, int32_t *n_tokens, int32_t *ranges,
                                  int32_t *n_ranges, void *workspace, size_t ws_bytes, sffn_stream_t stream) {
    if (!y_attn || !token_idx || !n_tokens || !ranges || !n_ranges) return SFFN_ERR_INVALID_ARG;
    if (L < 1 || L > (1 << 20) || d_model < 8 || d_model > 65536 || d_model % 8 != 0) return SFFN_ERR_SHAPE;
    if (block < 1 || (L + block - 1) / block > kMoeMaxBlocks) return SFFN_ERR_SHAPE;
    if (!(mass == mass) || !(min_ratio >= 0.f) || !(max_ratio <= 1.f) || !(min_ratio <= max_ratio))
        return SFFN_ERR_INVALID_ARG;
    if (!aligned16(y_attn)) return SFFN_ERR_ALIGNMENT;
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    sffn_status st = check_ws(workspace, ws_bytes, moe_budget_workspace(L, d_model));
    if (st != SFFN_OK) return st;
    st = run_moe_block_budget(y_attn, L, d_model, mass, min_ratio, max_ratio, block, token_idx, n_tokens, ranges,
                              n_ranges, workspace, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_gate_scores(const void *x, int B, const sffn_ffn_weights *w, int score, float *scores,
                             void *workspace, size_t ws_bytes, sffn_stream_t stream) {
    sffn_status st = check_decode_args(x, B, w, SFFN_MODE_THRESHOLD, score, 0.f);
    if (st != SFFN_OK) return st;
    if (!scores) return SFFN_ERR_INVALID_ARG;
    if (device_sm_count() <= 0) return SFFN_ERR_CUDA;
    DecodePlan p = make_decode_plan(B, w->d_model, w->d_ff);
    st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    DecodeCall c = {};
    c.x = x;
    c.w = w;
    c.B = B;
    c.mode = SFFN_MODE_KEEP_RATIO;
    c.score = score;
    c.ws = workspace;
    c.scores_only = scores;
    st = run_decode(c, p, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_token_select(const void *y_attn, int L, int d_model, float mass_thresh, int recent_n, int min_keep,
                              int32_t *sel_idx, int32_t *n_sel, void *workspace, size_t ws_bytes,
                              sffn_stream_t stream) {
    if (!y_attn || !sel_idx || !n_sel) return SFFN_ERR_INVALID_ARG;
    if (L < 1 || L > (1 << 20) || d_model < 8 || d_model > 65536 || d_model % 8 != 0) return SFFN_ERR_SHAPE;
    if (recent_n < 0 || min_keep < 1 || !(mass_thresh == mass_thresh)) return SFFN_ERR_INVALID_ARG;
    if (!aligned16(y_attn)) return SFFN_ERR_ALIGNMENT;
    SelectPlan p = make_select_plan(L, d_model);
    sffn_status st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    st = run_token_select(y_attn, L, d_model, mass_thresh, recent_n, min_keep, sel_idx, n_sel, workspace, p,
                          (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_prefill(const void *x, const void *y_attn, int L, const sffn_ffn_weights *w, const int32_t *sel_idx,
                         const int32_t *n_sel, void *out, void *workspace, size_t ws_bytes, sffn_stream_t stream) {
    if (!x || !y_attn || !sel_idx || !n_sel || !out) return SFFN_ERR_INVALID_ARG;
    sffn_status st = check_weights(w, false);
    if (st != SFFN_OK) return st;
    if ((w->wdtype != SFFN_BF16 && w->wdtype != SFFN_INT4_G64) || w->act != SFFN_ACT_SILU || w->b_gate)
        return SFFN_ERR_UNSUPPORTED;
    if (L < 1 || L > (1 << 20) || w->d_model % 64 != 0 || w->d_ff % 128 != 0) return SFFN_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(y_attn) || !aligned16(out)) return SFFN_ERR_ALIGNMENT;
    PrefillPlan p = make_prefill_plan(L, w->d_model, w->d_ff);
    st = check_ws(workspace, ws_bytes, p.total);
    if (st != SFFN_OK) return st;
    st = run_prefill(x, y_attn, L, w, sel_idx, n_sel, out, workspace, p, (cudaStream_t)stream);
    if (st == SFFN_OK) st = cuda_status(cudaGetLastError());
    return st;
}

sffn_status sffn_read_device_error(void *workspace, int32_t *code, sffn_stream_t stream) {
    if (!workspace || !code) return SFFN_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(code, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    // clears the whole control block: the error word and the decode grid
    // barrier's two counters (left inconsistent only by a call that recorded a
    // timeout at the barrier)
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, kControlBytes, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

}  // extern "C"
