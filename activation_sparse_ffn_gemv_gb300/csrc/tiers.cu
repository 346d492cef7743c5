// tiers.cu -- the core set of a keep-ratio tier from calibration scores
// (sm_103a).
//
// WiSparse write-up (kwkr.cn/news/623085, sec. 2.2, the paragraph after the
// score definition): to switch less online, count over a calibration set how
// often each column of a layer is in a token's top-k at the tier, and keep the
// most frequent columns as a guaranteed base ("core") set; each token then
// completes its selection with the largest scores outside the core
// (sffn_decode_tiered, the keep-ratio kernel with a forced set).  Read as: the
// core of size c is the c columns with the largest counts, count ties to the
// lower index, stored ascending.
//   k_topk_masks   one CTA per calibration token: its top-k (ties to the lower
//                  index) as mask words
//   k_col_counts   per column, the number of tokens whose mask holds it
//   k_core_list    one CTA: the top-c of the counts, ascending
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace sffn {

namespace {

constexpr int kTierThreads = 1024;
constexpr int kTierStage = 40960;  // keys staged in shared memory up to this many columns

// Stage n keys, mapping every key with the sign bit set (-0.0, or a negative
// score, which the scores never are) to 0 so that unsigned order is the order
// of the values.
SFFN_DEV void stage_score_keys(uint32_t *dst, const uint32_t *src, int n) {
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
        const uint32_t v = src[j];
        dst[j] = (v & 0x80000000u) ? 0u : v;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kTierThreads) k_topk_masks(const float *scores, int F, int k, uint32_t *masks,
                                                             uint32_t *gkeys) {
    extern __shared__ __align__(16) uint32_t tkey[];
    __shared__ unsigned hist[2048];
    __shared__ int tmp[34];
    griddep_wait();
    griddep_launch_dependents();
    const int n = blockIdx.x, nwords = (F + 31) >> 5;
    const uint32_t *src = reinterpret_cast<const uint32_t *>(scores + (size_t)n * F);
    uint32_t *key = F <= kTierStage ? tkey : gkeys + (size_t)n * F;
    stage_score_keys(key, src, F);
    const TopkCut cut = radix_topk(key, F, (unsigned)k, nullptr, hist, tmp);
    TopkChunk ch = topk_chunk(key, F, nullptr, cut, tmp);
    for (int w = ch.w0; w < ch.w1; ++w) {
        const TopkWord t = topk_word(key, F, nullptr, cut, w, ch);
        if ((threadIdx.x & 31) == 0) masks[(size_t)n * nwords + w] = t.bal;
    }
}

__global__ void __launch_bounds__(256) k_col_counts(const uint32_t *masks, int N, int F, uint32_t *counts) {
    griddep_wait();
    griddep_launch_dependents();
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= F) return;
    const int nwords = (F + 31) >> 5;
    const uint32_t *m = masks + (j >> 5);
    uint32_t c = 0;
    for (int n = 0; n < N; ++n) c += (m[(size_t)n * nwords] >> (j & 31)) & 1u;
    counts[j] = c;
}

__global__ void __launch_bounds__(kTierThreads) k_core_list(const uint32_t *counts, int F, int c, int32_t *core) {
    extern __shared__ __align__(16) uint32_t tkey[];
    __shared__ unsigned hist[2048];
    __shared__ int tmp[34];
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t *key = counts;
    if (F <= kTierStage) {
        stage_keys(tkey, counts, F);
        key = tkey;
    }
    const TopkCut cut = radix_topk(key, F, (unsigned)c, nullptr, hist, tmp);
    TopkChunk ch = topk_chunk(key, F, nullptr, cut, tmp);
    for (int w = ch.w0; w < ch.w1; ++w) {
        const TopkWord t = topk_word(key, F, nullptr, cut, w, ch);
        if (t.sel) core[t.pos] = 32 * w + (threadIdx.x & 31);
    }
}

struct TierPlan {
    size_t off_masks, off_counts, off_keys, total;
};

TierPlan make_tier_plan(int N, int F) {
    TierPlan p = {};
    const size_t nwords = (size_t)(F + 31) / 32;
    size_t o = 0;
    p.off_masks = o; o = align_up(o + sizeof(uint32_t) * (size_t)N * nwords);
    p.off_counts = o; o = align_up(o + sizeof(uint32_t) * (size_t)F);
    p.off_keys = o; o = align_up(o + (F > kTierStage ? sizeof(uint32_t) * (size_t)N * F : 0));
    p.total = o;
    return p;
}

}  // namespace

size_t tier_core_workspace(int N, int F) { return make_tier_plan(N, F).total; }

sffn_status run_tier_core_set(const float *scores, int N, int F, int k, int c, int32_t *core, void *ws,
                              cudaStream_t s) {
    const TierPlan p = make_tier_plan(N, F);
    char *w = static_cast<char *>(ws);
    uint32_t *masks = reinterpret_cast<uint32_t *>(w + p.off_masks);
    uint32_t *counts = reinterpret_cast<uint32_t *>(w + p.off_counts);
    uint32_t *gkeys = reinterpret_cast<uint32_t *>(w + p.off_keys);
    const size_t smem = F <= kTierStage ? sizeof(uint32_t) * (size_t)F : 0;
    const int smax = (int)(sizeof(uint32_t) * kTierStage);
    cudaError_t e = cudaSuccess;
    if (smem) e = set_max_smem((const void *)k_topk_masks, smax);
    if (e == cudaSuccess) e = launch_k(k_topk_masks, dim3(N), dim3(kTierThreads), smem, s, scores, F, k, masks, gkeys);
    if (e == cudaSuccess)
        e = launch_k(k_col_counts, dim3((F + 255) / 256), dim3(256), 0, s, (const uint32_t *)masks, N, F, counts);
    if (e == cudaSuccess && smem) e = set_max_smem((const void *)k_core_list, smax);
    if (e == cudaSuccess)
        e = launch_k(k_core_list, dim3(1), dim3(kTierThreads), smem, s, (const uint32_t *)counts, F, c, core);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
