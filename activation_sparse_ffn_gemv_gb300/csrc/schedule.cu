// schedule.cu -- the per-layer sparsity schedule of a multi-layer token-selective
// prefill, and a driver that runs a stack of layers on one stream.
//
// RedKnot write-up ("Token 選擇性稀疏 FFN", the three-tier SparseFFNSchedule and
// the FFN presets table): shallow layers (layer < dense_until) run the dense FFN,
// middle layers select tokens with mass_thresh, deep layers (layer >=
// deep_layer_start) with mass_thresh_deep.  A dense layer is a selection with
// mass 1, which keeps every token, so the prefill kernels serve every tier.
// Host code only: the layers' kernels are those of sffn_token_select and
// sffn_prefill, enqueued back to back without a host synchronisation (the whole
// stack can be captured in one CUDA graph).
#include <climits>

#include "internal.h"

namespace {

// The write-up's presets table: (dense_until, mass_thresh, recent_n).
struct PresetRow {
    int dense_until;
    float mass_thresh;
    int recent_n;
};
constexpr PresetRow kPresets[4] = {
    {3, 0.3f, 64},    // speed
    {20, 0.5f, 128},  // balanced
    {32, 0.7f, 128},  // quality
    {80, 1.0f, 128},  // dense (equivalent to the dense FFN)
};

bool schedule_ok(const sffn_ffn_schedule *s) {
    return s && s->dense_until >= 0 && s->deep_layer_start >= 0 && s->recent_n >= 0 && s->min_keep >= 1 &&
           s->mass_thresh >= 0.f && s->mass_thresh_deep >= 0.f;
}

}  // namespace

extern "C" {

sffn_status sffn_schedule_preset(int preset, sffn_ffn_schedule *out) {
    if (!out || preset < SFFN_PRESET_SPEED || preset > SFFN_PRESET_DENSE) return SFFN_ERR_INVALID_ARG;
    const PresetRow &r = kPresets[preset];
    out->dense_until = r.dense_until;
    out->deep_layer_start = INT_MAX;  // the presets name no deep tier
    out->mass_thresh = r.mass_thresh;
    out->mass_thresh_deep = r.mass_thresh;
    out->recent_n = r.recent_n;
    out->min_keep = 1;
    return SFFN_OK;
}

float sffn_schedule_mass(const sffn_ffn_schedule *s, int layer) {
    if (!schedule_ok(s) || layer < 0) return -1.f;
    if (layer < s->dense_until) return 1.f;
    if (layer >= s->deep_layer_start) return s->mass_thresh_deep;
    return s->mass_thresh;
}

size_t sffn_prefill_layers_workspace_size(int L, const sffn_ffn_weights *w) {
    if (!w || L < 1 || L > (1 << 20) || w->d_model < 8) return 0;
    const size_t sel = sffn::make_select_plan(L, w->d_model).total;
    const size_t pf = sffn::make_prefill_plan(L, w->d_model, w->d_ff).total;
    const size_t call = sffn::align_up(sel > pf ? sel : pf);
    return call + sffn::align_up((size_t)L * w->d_model * 2);  // + one bf16 [L, d_model] buffer
}

sffn_status sffn_prefill_layers(const void *x, const void *const *y_attn, int L, int n_layers,
                                const sffn_ffn_weights *w, const sffn_ffn_schedule *s, int first_layer, void *out,
                                int32_t *sel_idx, int32_t *n_sel, void *workspace, size_t ws_bytes,
                                sffn_stream_t stream) {
    if (!x || !y_attn || !w || !s || !out || !sel_idx || !n_sel) return SFFN_ERR_INVALID_ARG;
    if (!schedule_ok(s) || first_layer < 0) return SFFN_ERR_INVALID_ARG;
    if (n_layers < 1 || L < 1 || L > (1 << 20)) return SFFN_ERR_SHAPE;
    if (x == out) return SFFN_ERR_INVALID_ARG;
    // one workspace region serves each layer's selection and prefill in turn
    // (the control block at its start stays valid across entry points); the
    // largest layer sizes it
    size_t need = 0;
    for (int i = 0; i < n_layers; ++i) {
        if (!y_attn[i]) return SFFN_ERR_INVALID_ARG;
        if (w[i].d_model != w[0].d_model) return SFFN_ERR_SHAPE;
        const size_t n = sffn_prefill_layers_workspace_size(L, &w[i]);
        if (n == 0) return SFFN_ERR_SHAPE;
        if (n > need) need = n;
    }
    const size_t ping_bytes = sffn::align_up((size_t)L * w[0].d_model * 2);
    const size_t call_bytes = need - ping_bytes;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & (sffn::kAlign - 1)) != 0 || ws_bytes < need)
        return SFFN_ERR_WORKSPACE;
    void *ping = static_cast<char *>(workspace) + call_bytes;
    // layer i writes `out` when (n_layers - 1 - i) is even, else the ping
    // buffer, so the last layer ends in `out` and no layer reads its own output
    const void *in = x;
    for (int i = 0; i < n_layers; ++i) {
        void *dst = ((n_layers - 1 - i) % 2 == 0) ? out : ping;
        const float mass = sffn_schedule_mass(s, first_layer + i);
        sffn_status st = sffn_token_select(y_attn[i], L, w[i].d_model, mass, s->recent_n, s->min_keep,
                                           sel_idx + (size_t)i * L, n_sel + i, workspace, call_bytes, stream);
        if (st != SFFN_OK) return st;
        st = sffn_prefill(in, y_attn[i], L, &w[i], sel_idx + (size_t)i * L, n_sel + i, dst, workspace, call_bytes,
                          stream);
        if (st != SFFN_OK) return st;
        in = dst;
    }
    return SFFN_OK;
}

}  // extern "C"
