// moe.cu -- adaptive expert top-K and the block token budget of an MoE layer
// (sm_103a).
//
// RedKnot write-up (bhfrc.com/news/43276, section "adaptive expert Top-K"):
//   * a progressive top-K by depth (layers 0-15: 6 experts, 16-39: 5, 40-60: 4);
//   * per token, the smallest K among the candidate buckets (3, 4, 5, 6) whose
//     top-K routing probability mass reaches 0.50 (else the layer's K);
//   * a token budget between min_full_ratio 0.10 and max_full_ratio 0.50 of the
//     tokens, taken as whole 128-token blocks chosen by a top-K so that the
//     routed rows form few contiguous ranges, all on the GPU with no host sync.
// Read as (every free choice stated): routing probabilities are the softmax of
// the router logits; experts rank by probability descending, ties to the lower
// expert index; the chosen experts' weights are their probabilities
// renormalised to sum 1; the budget's fraction is the share of tokens the
// token-selective FFN's mass rule keeps (no recent tail, no minimum), clamped
// to [min_ratio, max_ratio]; ceil(f * nblocks) blocks (at least one) with the
// largest summed importance run the MoE, ties to the lower block index.
//
//   k_moe_route     one warp per token: the token's logits in registers, the
//                   softmax in fp32, the top-cap experts by repeated warp
//                   arg-max, the bucket, and the ascending expert list
//   k_block_budget  one CTA after the token selection's norms and mass-prefix
//                   count: block sums, the top-nsel blocks (topk.cuh), the
//                   ascending token list and its contiguous ranges
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace sffn {

namespace {

constexpr int kRouteWarps = 8;
constexpr int kMaxExpertsPerLane = kMoeMaxExperts / 32;

__global__ void __launch_bounds__(32 * kRouteWarps) k_moe_route(MoeRouteArgs a) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
    if (t >= a.T) return;
    const int E = a.E;
    const float *lg = a.logits + (size_t)t * E;
    float v[kMaxExpertsPerLane];
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMaxExpertsPerLane; ++q) {
        const int e = lane + 32 * q;
        v[q] = e < E ? lg[e] : -INFINITY;
        mx = fmaxf(mx, v[q]);
    }
    mx = warp_max(mx);
    // the probabilities' normaliser
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxExpertsPerLane; ++q)
        if (lane + 32 * q < E) sum += expf(v[q] - mx);
    sum = warp_sum(sum);
    // the top-cap experts: logit descending, ties to the lower index (the order
    // of the probabilities, a monotone map of the logits); every lane ends with
    // the same lists
    int top_e[kMoeMaxK];
    float top_p[kMoeMaxK];
    bool taken[kMaxExpertsPerLane];
#pragma unroll
    for (int q = 0; q < kMaxExpertsPerLane; ++q) taken[q] = false;
#pragma unroll
    for (int i = 0; i < kMoeMaxK; ++i) {
        top_e[i] = -1;
        top_p[i] = 0.f;
        if (i >= a.cap) continue;
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < kMaxExpertsPerLane; ++q) {
            const int e = lane + 32 * q;
            if (e < E && !taken[q] && (v[q] > bv || (v[q] == bv && e < be))) {
                bv = v[q];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
#pragma unroll
        for (int q = 0; q < kMaxExpertsPerLane; ++q)
            if (lane + 32 * q == be) taken[q] = true;
        top_e[i] = be;
        top_p[i] = expf(bv - mx);  // the same value the normaliser summed
    }
    // the bucket: the smallest admissible K whose top-K mass reaches the threshold
    float cum[kMoeMaxK + 1];
    cum[0] = 0.f;
#pragma unroll
    for (int i = 0; i < kMoeMaxK; ++i) cum[i + 1] = cum[i] + top_p[i];
    int K = a.cap;
    float cumK = 0.f;
    bool found = false;
    for (int bi = 0; bi < a.n_buckets && !found; ++bi) {
        const int b = a.buckets[bi];
        if (b > a.cap) break;
        float cb = 0.f;
#pragma unroll
        for (int i = 1; i <= kMoeMaxK; ++i)
            if (i == b) cb = cum[i];
        if (cb >= a.mass * sum) {
            K = b;
            found = true;
        }
    }
#pragma unroll
    for (int i = 1; i <= kMoeMaxK; ++i)
        if (i == K) cumK = cum[i];
    // lane i < K writes the i-th chosen expert at its rank in ascending order,
    // its weight renormalised over the chosen K
    int32_t *ex = a.experts + (size_t)t * a.kmax;
    float *wt = a.weights + (size_t)t * a.kmax;
    int my_e = -1;
    float my_p = 0.f;
#pragma unroll
    for (int i = 0; i < kMoeMaxK; ++i)
        if (i == lane) {
            my_e = top_e[i];
            my_p = top_p[i];
        }
    if (lane < K) {
        int rank = 0;
#pragma unroll
        for (int i = 0; i < kMoeMaxK; ++i) rank += (i < K && top_e[i] < my_e) ? 1 : 0;
        ex[rank] = my_e;
        wt[rank] = my_p / cumK;
    } else if (lane < a.kmax) {
        ex[lane] = -1;
        wt[lane] = 0.f;
    }
    if (lane == 0) a.k_out[t] = K;
}

constexpr int kBudgetThreads = 1024;

struct BudgetArgs {
    const float *norms;       // [L] token importances
    const int32_t *n_prefix;  // tokens the mass rule keeps
    int L, block;
    float min_ratio, max_ratio;
    int32_t *token_idx, *n_tokens, *ranges, *n_ranges;
};

__global__ void __launch_bounds__(kBudgetThreads) k_block_budget(BudgetArgs a) {
    extern __shared__ __align__(16) uint32_t bkey[];  // [nblocks] block sums (float bits)
    __shared__ unsigned hist[2048];
    __shared__ int tmp[34];
    __shared__ uint32_t bmask[kMoeMaxBlocks / 32];
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = kBudgetThreads / 32;
    const int L = a.L, blk = a.block;
    const int nblocks = (L + blk - 1) / blk;
    // block sums: one warp per block
    for (int b = warp; b < nblocks; b += nw) {
        float s = 0.f;
        for (int t = b * blk + lane; t < min(L, (b + 1) * blk); t += 32) s += a.norms[t];
        s = warp_sum(s);
        if (lane == 0) bkey[b] = __float_as_uint(s);  // sums of non-negative values
    }
    __syncthreads();
    // blocks to take
    const double n = (double)min(max(*a.n_prefix, 0), L);
    double f = n / (double)L;
    f = fmin(fmax(f, (double)a.min_ratio), (double)a.max_ratio);
    int nsel = (int)ceil(f * (double)nblocks - 1e-12);
    nsel = max(1, min(nblocks, nsel));
    const TopkCut cut = radix_topk(bkey, nblocks, (unsigned)nsel, nullptr, hist, tmp);
    TopkChunk ch = topk_chunk(bkey, nblocks, nullptr, cut, tmp);
    for (int w = ch.w0; w < ch.w1; ++w) {
        const TopkWord tw = topk_word(bkey, nblocks, nullptr, cut, w, ch);
        if (lane == 0) bmask[w] = tw.bal;
        if (tw.sel) {
            // chosen block of rank tw.pos: its tokens at positions tw.pos * blk ...
            // (only the sequence's last block can be short, and it ranks last)
            const int b = 32 * w + lane;
            for (int t = b * blk; t < min(L, (b + 1) * blk); ++t) a.token_idx[(size_t)tw.pos * blk + (t - b * blk)] = t;
        }
    }
    __syncthreads();
    // contiguous ranges of chosen blocks: a range starts at a chosen block whose
    // predecessor is not chosen and ends after a chosen block whose successor is
    // not; the r-th start and the r-th end (in index order) bound range r
    const int nwords = (nblocks + 31) >> 5;
    auto starts_of = [&](int w) {
        const uint32_t m = bmask[w], prev = w > 0 ? (bmask[w - 1] >> 31) : 0u;
        return m & ~((m << 1) | prev);
    };
    auto ends_of = [&](int w) {
        const uint32_t m = bmask[w], next = w + 1 < nwords ? (bmask[w + 1] & 1u) : 0u;
        return m & ~((m >> 1) | (next << 31));
    };
    int ns = 0, ne = 0;
    for (int w = tid; w < nwords; w += kBudgetThreads) {
        ns += __popc(starts_of(w));
        ne += __popc(ends_of(w));
    }
    int total_r, total_e;
    int rs = block_excl_scan(ns, tmp, &total_r);
    int re = block_excl_scan(ne, tmp, &total_e);
    for (int w = tid; w < nwords; w += kBudgetThreads) {
        for (uint32_t m = starts_of(w); m; m &= m - 1) a.ranges[2 * rs++] = (32 * w + __ffs(m) - 1) * blk;
        for (uint32_t m = ends_of(w); m; m &= m - 1) a.ranges[2 * re++ + 1] = min(L, (32 * w + __ffs(m)) * blk);
    }
    if (tid == 0) {
        *a.n_ranges = total_r;
        // whole blocks, less the tail of a short last block when it is chosen
        const int short_by = (L % blk && bit_at(bmask, nblocks - 1)) ? blk - L % blk : 0;
        *a.n_tokens = nsel * blk - short_by;
    }
}

}  // namespace

sffn_status run_moe_route(const MoeRouteArgs &a, cudaStream_t s) {
    const int grid = (a.T + kRouteWarps - 1) / kRouteWarps;
    const cudaError_t e = launch_k(k_moe_route, dim3(grid), dim3(32 * kRouteWarps), 0, s, a);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

size_t moe_budget_workspace(int L, int d) {
    const SelectPlan p = make_select_plan(L, d);
    return align_up(p.total + align_up(sizeof(int32_t) * (size_t)L) + kAlign);
}

sffn_status run_moe_block_budget(const void *y_attn, int L, int d, float mass, float min_ratio, float max_ratio,
                                 int block, int32_t *token_idx, int32_t *n_tokens, int32_t *ranges,
                                 int32_t *n_ranges, void *ws, cudaStream_t s) {
    const SelectPlan p = make_select_plan(L, d);
    char *w = static_cast<char *>(ws);
    int32_t *sel = reinterpret_cast<int32_t *>(w + align_up(p.total));
    int32_t *n_prefix = reinterpret_cast<int32_t *>(w + align_up(p.total) + align_up(sizeof(int32_t) * (size_t)L));
    // the mass rule's prefix alone: no recent tail, no minimum
    sffn_status st = run_token_select(y_attn, L, d, mass, 0, 0, sel, n_prefix, ws, p, s);
    if (st != SFFN_OK) return st;
    BudgetArgs ba = {};
    ba.norms = reinterpret_cast<const float *>(w + p.off_norms);
    ba.n_prefix = n_prefix;
    ba.L = L;
    ba.block = block;
    ba.min_ratio = min_ratio;
    ba.max_ratio = max_ratio;
    ba.token_idx = token_idx;
    ba.n_tokens = n_tokens;
    ba.ranges = ranges;
    ba.n_ranges = n_ranges;
    const int nblocks = (L + block - 1) / block;
    const size_t smem = sizeof(uint32_t) * (size_t)nblocks;
    cudaError_t e = set_max_smem((const void *)k_block_budget, (int)(sizeof(uint32_t) * kMoeMaxBlocks));
    if (e == cudaSuccess) e = launch_k(k_block_budget, dim3(1), dim3(kBudgetThreads), smem, s, ba);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
