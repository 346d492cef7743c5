// prefill.cu -- token selection and token-selective prefill (sm_103a).
#include "common.cuh"
#include "internal.h"

namespace sffn {

PrefillPlan make_prefill_plan(int L, int d, int F) {
    PrefillPlan p = {};
    p.L = L;
    p.d = d;
    p.F = F;
    size_t o = 0;
    p.off_err = o; o = align_up(o + sizeof(int32_t));
    p.off_ysel = o; o = align_up(o + sizeof(uint16_t) * (size_t)L * d);
    p.off_h = o; o = align_up(o + sizeof(uint16_t) * (size_t)L * F);
    p.total = o;
    return p;
}

sffn_status run_prefill(const void *, const void *, int, const sffn_ffn_weights *, const int32_t *, const int32_t *,
                        void *, void *, const PrefillPlan &, cudaStream_t) {
    return SFFN_ERR_UNSUPPORTED;
}

}  // namespace sffn
