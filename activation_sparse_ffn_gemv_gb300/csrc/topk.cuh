// topk.cuh -- exact top-k of 32-bit keys by one CTA (sm_103a): the k largest
// keys, ties to the lower index, by a radix select over the key bits (no sort).
//
// Keys are the bit patterns of non-negative floats (whose order the unsigned
// bits keep) or plain counts.  A key set may come with a "forced" bitmask: the
// forced keys are always selected and are not candidates of the select, so the
// select takes the k largest of the others (WiSparse write-up, sec. 2.2: a
// per-layer core set plus a dynamic supplement).
//
// The CTA runs three digit passes (bits 31..21, 20..10, 9..0) with a count
// histogram in shared memory (32-bit atomic increments), which give the cut T
// (the k-th largest candidate key) and how many candidates equal to T are
// taken.  The ordered pass then gives each warp a contiguous chunk of whole
// 32-key words: a ballot over 32 consecutive keys is that word of the selection
// mask, and ballot popcounts rank the selected keys in ascending index order.
#pragma once
#include "common.cuh"

namespace sffn {

// Find, over nbins bins scanned from the top, the bin where the running count
// reaches `need`.  Returns the bin; *above = count in higher bins.
SFFN_DEV int find_cross_bin(const unsigned *hist, int nbins, unsigned need, unsigned *above, int *tmp) {
    // each thread owns up to 2 consecutive bins in descending order
    const int t = threadIdx.x;
    const int b0 = nbins - 1 - 2 * t, b1 = b0 - 1;
    const unsigned c0 = b0 >= 0 ? hist[b0] : 0u, c1 = b1 >= 0 ? hist[b1] : 0u;
    int total;
    const unsigned ex = (unsigned)block_excl_scan((int)(c0 + c1), tmp, &total);
    __shared__ int s_bin;
    __shared__ unsigned s_above;
    if (b0 >= 0 && ex < need && ex + c0 >= need) { s_bin = b0; s_above = ex; }
    if (b1 >= 0 && ex + c0 < need && ex + c0 + c1 >= need) { s_bin = b1; s_above = ex + c0; }
    __syncthreads();
    const int bin = s_bin;
    *above = s_above;
    __syncthreads();
    return bin;
}

// Copy n 32-bit keys into shared memory (sixteen loads in flight per thread:
// one memory round trip up to 16 x blockDim keys).
SFFN_DEV void stage_keys(uint32_t *dst, const uint32_t *src, int n) {
    constexpr int K = 16;
    for (int j0 = threadIdx.x; j0 < n; j0 += K * blockDim.x) {
        uint32_t v[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int j = j0 + k * blockDim.x;
            v[k] = j < n ? __ldcg(src + j) : 0u;
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const int j = j0 + k * blockDim.x;
            if (j < n) dst[j] = v[k];
        }
    }
    __syncthreads();
}

SFFN_DEV bool bit_at(const uint32_t *mask, int j) { return mask && ((mask[j >> 5] >> (j & 31)) & 1u); }

struct TopkCut {
    uint32_t T;        // the k-th largest candidate key
    unsigned take_eq;  // candidates equal to T that are taken, lowest index first
    unsigned n_eq;     // candidates equal to T (take_eq == n_eq: every one of them is taken)
};

// The cut of the k largest candidate keys (k <= the number of candidates);
// k == 0 selects no candidate.
SFFN_DEV TopkCut radix_topk(const uint32_t *key, int F, unsigned k, const uint32_t *forced, unsigned *hist,
                            int *tmp) {
    if (k == 0) return TopkCut{0xFFFFFFFFu, 0u, 0u};
    uint32_t prefix = 0, pmask = 0;
    unsigned need = k, n_eq = 0;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass], nbins = 1 << widths[pass];
        for (int i = threadIdx.x; i < nbins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < F; j += blockDim.x) {
            const uint32_t kv = key[j];
            if ((kv & pmask) == prefix && !bit_at(forced, j)) atomicAdd(&hist[(kv >> sh) & (nbins - 1)], 1u);
        }
        __syncthreads();
        unsigned above;
        const int bin = find_cross_bin(hist, nbins, need, &above, tmp);
        prefix |= (uint32_t)bin << sh;
        pmask |= (uint32_t)(nbins - 1) << sh;
        need -= above;
        if (pass == 2) n_eq = hist[bin];  // the last digit: the bin holds exactly the keys equal to T
    }
    return TopkCut{prefix, need, n_eq};
}

// This warp's chunk of 32-key words [w0, w1) for the ordered pass, with the
// number of candidates equal to T in earlier chunks and the position of its
// first selected key; total = keys selected by the whole CTA.
struct TopkChunk {
    int w0, w1;
    int eq_seen, pos, total;
};

SFFN_DEV TopkChunk topk_chunk(const uint32_t *key, int F, const uint32_t *forced, TopkCut cut, int *tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nwords = (F + 31) >> 5;
    const int wchunk = (nwords + nw - 1) / nw;
    TopkChunk c;
    c.w0 = min(nwords, warp * wchunk);
    c.w1 = min(nwords, c.w0 + wchunk);
    int gt = 0, eq = 0, fc = 0;
    for (int w = c.w0; w < c.w1; ++w) {
        const int j = 32 * w + lane;
        const bool ok = j < F;
        const uint32_t kv = ok ? key[j] : 0u;
        const bool f = ok && bit_at(forced, j);
        fc += __popc(__ballot_sync(0xffffffffu, f));
        gt += __popc(__ballot_sync(0xffffffffu, ok && !f && kv > cut.T));
        eq += __popc(__ballot_sync(0xffffffffu, ok && !f && kv == cut.T));
    }
    int tot;
    c.eq_seen = __shfl_sync(0xffffffffu, block_excl_scan(lane == 0 ? eq : 0, tmp, &tot), 0);
    const int eq_take =
        (int)min((unsigned)eq, cut.take_eq > (unsigned)c.eq_seen ? cut.take_eq - (unsigned)c.eq_seen : 0u);
    c.pos = __shfl_sync(0xffffffffu, block_excl_scan(lane == 0 ? gt + eq_take + fc : 0, tmp, &c.total), 0);
    return c;
}

// One word of the ordered pass: whether this lane's key j is selected, its
// position among the selected keys, and the word's selection ballot; advances
// the chunk's running counts.
struct TopkWord {
    bool sel;
    int pos;
    unsigned bal;
};

SFFN_DEV TopkWord topk_word(const uint32_t *key, int F, const uint32_t *forced, TopkCut cut, int w, TopkChunk &c) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int j = 32 * w + lane;
    const bool ok = j < F;
    const uint32_t kv = ok ? key[j] : 0u;
    const bool f = ok && bit_at(forced, j);
    const bool e = ok && !f && kv == cut.T;
    const unsigned ebal = __ballot_sync(0xffffffffu, e);
    const bool sel = ok && (f || kv > cut.T || (e && (unsigned)(c.eq_seen + __popc(ebal & lt)) < cut.take_eq));
    const unsigned sbal = __ballot_sync(0xffffffffu, sel);
    TopkWord r{sel, c.pos + __popc(sbal & lt), sbal};
    c.pos += __popc(sbal);
    c.eq_seen += __popc(ebal);
    return r;
}

}  // namespace sffn
