// select.cu -- token selection for the token-selective prefill (sm_103a).
//
// RedKnot (token-selective sparse FFN, bhfrc.com/news/43276): a token's
// importance is the L2 norm of its attention-output row; tokens are taken in
// decreasing importance until their importance sum covers mass_thresh of the
// total (the crossing token included); the last recent_n tokens are always
// kept, at least min_keep tokens are kept, and an all-zero importance vector or
// mass_thresh >= 1 keeps every token.  No sort and no host synchronisation:
//   token_norms  one warp per row, 128-bit loads, fp32 sum of squares (the
//                product of two bf16 values is exact in fp32); each CTA also
//                leaves its largest importance
//   mass prefix  importances are turned into 64-bit fixed point (scale from
//                the largest importance) so every mass sum is exact and order
//                independent; a radix select over the float bits (11 + 11 + 10
//                bits) with a fixed-point mass per bin finds the bin where the
//                mass from the top reaches the target, and after three passes
//                the cut value and how many keys equal to it are taken (ties go
//                to the lower index).  Up to 32768 tokens the selection CTA
//                does this itself on importances staged in shared memory;
//                longer sequences run each pass on many CTAs (mass_pass: a
//                histogram per CTA, merged in global memory, the last CTA to
//                finish finds the bin).
//   mass_select  one CTA: the selected prefix (ordered pass for the ties at the
//                cut), the recent tail, the min_keep extension (a count radix
//                select over the unselected tokens) and an ordered compaction
//                to ascending indices.  The ordered passes give each warp a
//                contiguous chunk of tokens and rank inside it with ballots.
//
// Shared-memory histograms hold a bin's mass as three 32-bit limbs of 14 bits
// per key (a key's mass is below 2^40 units, and a bin of up to 2^15 keys keeps
// each limb sum below 2^29): 32-bit shared atomics are native, where a 64-bit
// shared atomic add is not.
#include "common.cuh"
#include "internal.h"

namespace sffn {

// ---------------------------------------------------------------------------
// importance: s_t = ||y_attn[t, :]||_2
// ---------------------------------------------------------------------------

constexpr int kNormWarps = 8;
constexpr int kMaxNormCtas = 4096;  // per-CTA maxima kept for the mass passes
constexpr int kHistBins = 2048;

// State of the multi-CTA mass passes in the workspace (cleared by the norms
// kernel when they run).
struct SelState {
    unsigned long long target;  // mass the selected prefix must reach
    unsigned long long above;   // mass of the keys above the candidate bin
    unsigned long long take;    // keys equal to the cut that are taken, lowest index first
    unsigned done[3];           // CTAs finished, per pass
    int ex;                     // fixed-point exponent: every importance < 2^ex
    int mode;                   // 0: no mass prefix, 1: every token, 2: the prefix down to `cut`
    uint32_t prefix, pmask;     // radix state
    uint32_t cut;
};

__global__ void __launch_bounds__(32 * kNormWarps) k_token_norms(const void *y, int L, int d, float *s, float *cmax,
                                                                 SelState *st, unsigned long long *gmass, int clear) {
    __shared__ float s_max[kNormWarps];
    griddep_wait();
    griddep_launch_dependents();
    if (clear && blockIdx.x == 0) {  // state of the multi-CTA mass passes
        for (int i = threadIdx.x; i < 3 * kHistBins; i += blockDim.x) gmass[i] = 0ull;
        if (threadIdx.x == 0) *st = SelState{};
    }
    float wmax = 0.f;
    const int lane = threadIdx.x & 31;
    const int units = d / 8;  // 16-byte units of 8 bf16
    const size_t gw = (size_t)blockIdx.x * kNormWarps + (threadIdx.x >> 5);
    const size_t nw = (size_t)gridDim.x * kNormWarps;
    constexpr int U = 10;     // loads in flight per lane
    for (size_t t = gw; t < (size_t)L; t += nw) {
        const char *row = static_cast<const char *>(y) + t * (size_t)units * 16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        auto add = [&](const uint4 &x) {
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = bf16lo(w[q]), hi = bf16hi(w[q]);
                acc[q] = fmaf(lo, lo, acc[q]);
                acc[q] = fmaf(hi, hi, acc[q]);
            }
        };
        // whole chunks of 32 * U units load without a bounds test, then at
        // most one partial chunk
        int u0 = 0;
        for (; u0 + 32 * U <= units; u0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int i = 0; i < U; ++i) v[i] = ldg_stream(row + (size_t)(u0 + i * 32 + lane) * 16);
#pragma unroll
            for (int i = 0; i < U; ++i) add(v[i]);
        }
        if (u0 < units) {
            uint4 v[U];
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int u = u0 + i * 32 + lane;
                v[i] = u < units ? ldg_stream(row + (size_t)u * 16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < U; ++i) add(v[i]);
        }
        const float tot = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
        const float nv = sqrtf(tot);
        if (lane == 0) s[t] = nv;
        wmax = fmaxf(wmax, nv);
    }
    // this CTA's largest importance (the fixed-point scale of the mass passes)
    if (lane == 0) s_max[threadIdx.x >> 5] = wmax;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < kNormWarps; ++w) m = fmaxf(m, s_max[w]);
        cmax[blockIdx.x] = m;
    }
}

// ---------------------------------------------------------------------------
// selection helpers
// ---------------------------------------------------------------------------

constexpr int kSelectThreads = 1024;
constexpr int kPassThreads = 256;
// Up to this many importances (and their flags) are staged in shared memory,
// so that every pass of the selection reads on-chip memory.
constexpr int kStageKeys = 32768;

SFFN_DEV unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Block-wide exclusive scan of a 64-bit value per thread; *total = block sum.
SFFN_DEV unsigned long long block_excl_scan_u64(unsigned long long v, unsigned long long *scratch,
                                                unsigned long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const unsigned long long incl = warp_incl_scan_u64(v, lane);
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long w = lane < nw ? scratch[lane] : 0ull;
        const unsigned long long wi = warp_incl_scan_u64(w, lane);
        if (lane < nw) scratch[lane] = wi - w;
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    const unsigned long long r = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return r;
}

// Block-wide maximum of a non-negative float per thread.
SFFN_DEV float block_max(float v, float *scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float m = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, scratch[w]);
    __syncthreads();
    return m;
}

// Fixed-point mass of an importance v >= 0: v * 2^(40 - ex) rounded to the
// nearest integer (ties to even), from the float's bits with integer shifts
// only (no FP64 on the path).  With max importance < 2^ex every value is below
// 2^40 units.
SFFN_DEV unsigned long long fixed_mass(float v, int ex) {
    const uint32_t u = __float_as_uint(v);
    const int e = (int)((u >> 23) & 0xFFu);
    const unsigned long long m = (u & 0x7FFFFFu) | (e ? 0x800000u : 0u);  // v = m * 2^(max(e,1) - 150)
    if (m == 0ull || e == 0xFF) return 0ull;
    const int sh = (e ? e : 1) - 150 + 40 - ex;
    if (sh >= 0) return m << sh;
    const int r = -sh;
    if (r > 24) return 0ull;  // m < 2^24 <= half a unit
    const unsigned long long q = m >> r, rem = m & ((1ull << r) - 1ull), half = 1ull << (r - 1);
    return q + ((rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull);
}

// Mass of a bin from its three 14-bit limb sums.
SFFN_DEV unsigned long long limb_mass(const unsigned *hl, int bin) {
    return (unsigned long long)hl[bin] + ((unsigned long long)hl[kHistBins + bin] << 14) +
           ((unsigned long long)hl[2 * kHistBins + bin] << 28);
}

// Histogram of the digit at `sh` (nbins bins) over the keys of sv[0, L) whose
// bits under pmask equal prefix: the fixed-point mass per bin (MASS, as limbs
// in hl[3][kHistBins]) or the count per bin (!MASS, skipping keys flagged in
// `exclude`).  A warp whose 32 keys share one bin adds them up with warp
// reductions and updates the bin once; otherwise every key updates its bin.
template <bool MASS>
SFFN_DEV void radix_hist(const float *sv, int L, const uint8_t *exclude, uint32_t prefix, uint32_t pmask, int sh,
                         int nbins, int ex, unsigned *hcnt, unsigned *hl) {
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) {
        if (MASS) {
            hl[i] = 0u;
            hl[kHistBins + i] = 0u;
            hl[2 * kHistBins + i] = 0u;
        } else {
            hcnt[i] = 0u;
        }
    }
    __syncthreads();
    constexpr int U = 8;  // keys in flight per thread
    const int lane = threadIdx.x & 31;
    for (int t0 = threadIdx.x - lane; t0 < L; t0 += U * blockDim.x) {
        float v[U];
        bool ok[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int t = t0 + lane + k * blockDim.x;
            ok[k] = t < L && !(exclude && exclude[t]);
            v[k] = ok[k] ? sv[t] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t kv = __float_as_uint(v[k]);
            const int bin = ok[k] && (kv & pmask) == prefix ? (int)((kv >> sh) & (uint32_t)(nbins - 1)) : nbins;
            if (!MASS) {
                if (bin < nbins) atomicAdd(&hcnt[bin], 1u);
                continue;
            }
            const unsigned long long m = bin < nbins ? fixed_mass(v[k], ex) : 0ull;
            const unsigned l0 = (unsigned)(m & 0x3FFFu), l1 = (unsigned)((m >> 14) & 0x3FFFu),
                           l2 = (unsigned)(m >> 28);
            const int b0 = __shfl_sync(0xffffffffu, bin, 0);
            if (__all_sync(0xffffffffu, bin == b0)) {
                if (b0 < nbins) {
                    const unsigned s0 = __reduce_add_sync(0xffffffffu, l0), s1 = __reduce_add_sync(0xffffffffu, l1),
                                   s2 = __reduce_add_sync(0xffffffffu, l2);
                    if (lane == 0) {
                        atomicAdd(&hl[b0], s0);
                        atomicAdd(&hl[kHistBins + b0], s1);
                        atomicAdd(&hl[2 * kHistBins + b0], s2);
                    }
                }
            } else if (bin < nbins) {
                atomicAdd(&hl[bin], l0);
                atomicAdd(&hl[kHistBins + bin], l1);
                atomicAdd(&hl[2 * kHistBins + bin], l2);
            }
        }
    }
    __syncthreads();
}

// Ordered pass over the keys equal to `cut`, ranked by index: each warp owns a
// contiguous chunk (a multiple of 128 tokens) and ranks inside it with ballots
// after a scan of the warps' counts.  A key is in when kv > cut, or kv == cut
// and its rank is below `take`.  EXT (the min_keep extension) looks only at
// unflagged keys and only sets flags; otherwise every flag is written.
template <bool EXT>
SFFN_DEV void ordered_take(const float *sv, uint8_t *fl, int L, uint32_t cut, unsigned long long take, int *scr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int chunk = (((L + nw - 1) / nw) + 127) & ~127;
    const int c0 = min(L, warp * chunk), c1 = min(L, c0 + chunk);
    constexpr int U = 4;
    int eq = 0;
    for (int t0 = c0; t0 < c1; t0 += 32 * U) {
        bool e[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int t = t0 + 32 * k + lane;
            e[k] = t < c1 && __float_as_uint(sv[t]) == cut && (!EXT || !fl[t]);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) eq += __popc(__ballot_sync(0xffffffffu, e[k]));
    }
    int tot;
    const int wb = block_excl_scan(lane == 0 ? eq : 0, scr, &tot);
    unsigned long long seen = (unsigned long long)__shfl_sync(0xffffffffu, wb, 0);
    const unsigned lt = (1u << lane) - 1u;
    for (int t0 = c0; t0 < c1; t0 += 32 * U) {
        uint32_t kv[U];
        bool fr[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int t = t0 + 32 * k + lane;
            const bool ok = t < c1;
            kv[k] = ok ? __float_as_uint(sv[t]) : 0u;
            fr[k] = ok && (!EXT || !fl[t]);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int t = t0 + 32 * k + lane;
            const bool e = fr[k] && kv[k] == cut;
            const unsigned bal = __ballot_sync(0xffffffffu, e);
            const bool in = kv[k] > cut || (e && seen + (unsigned)__popc(bal & lt) < take);
            if (fr[k]) {
                if (EXT) {
                    if (in) fl[t] = 1;
                } else {
                    fl[t] = in ? 1 : 0;
                }
            }
            seen += (unsigned)__popc(bal);
        }
    }
    __syncthreads();
}

// Number of set flags (each flag byte is 0 or 1, so a word's popcount counts
// its flags); the flag array is padded with zero bytes to a multiple of 4.
SFFN_DEV int count_flags(const uint8_t *fl, int L, int *scr) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(fl);
    int c = 0;
    for (int i = threadIdx.x; i < (L + 3) / 4; i += blockDim.x) c += __popc(w[i]);
    int tot;
    block_excl_scan(c, scr, &tot);
    return tot;
}

// ---------------------------------------------------------------------------
// mass passes on many CTAs (sequences longer than kStageKeys)
// ---------------------------------------------------------------------------

struct PassArgs {
    const float *s;
    int L;
    const float *cmax;   // [ncmax] the norms kernel's per-CTA maxima
    int ncmax;
    float mass_thresh;
    SelState *st;
    unsigned long long *gmass;  // [3][kHistBins] fixed-point mass per bin, per pass
};

// Pass P looks at the digit at shift (21, 10, 0) of width (11, 11, 10) of the
// keys whose higher bits equal the prefix found so far.  Each CTA builds the
// pass's histogram of its slice of the tokens in shared memory and adds its
// non-empty bins to the global histogram; the last CTA to finish finds the bin,
// from the top, through which the mass reaches the target and stores the next
// prefix (after pass 0 it first forms the total and the target; after pass 2
// the cut and the number of keys equal to it that are taken).
template <int P>
__global__ void __launch_bounds__(kPassThreads) k_mass_pass(PassArgs a) {
    constexpr int sh = P == 0 ? 21 : (P == 1 ? 10 : 0);
    constexpr int nbins = P == 2 ? 1024 : 2048;
    __shared__ unsigned hl[3 * kHistBins];
    __shared__ unsigned long long scr64[33];
    __shared__ float s_red[kPassThreads / 32];
    __shared__ int s_last, s_bin;
    __shared__ unsigned long long s_above;
    griddep_wait();
    griddep_launch_dependents();
    SelState *st = a.st;
    const int tid = threadIdx.x;
    int ex = 0, mode = 2;
    uint32_t prefix = 0, pmask = 0;
    if (P == 0) {
        float mx = 0.f;
        for (int i = tid; i < a.ncmax; i += blockDim.x) mx = fmaxf(mx, a.cmax[i]);
        mx = block_max(mx, s_red);
        if (mx > 0.f) frexpf(mx, &ex);  // every importance < 2^ex
        // an all-zero importance vector (zero total mass) keeps every token
        mode = (a.mass_thresh >= 1.f || mx == 0.f) ? 1 : (a.mass_thresh > 0.f ? 2 : 0);
        if (blockIdx.x == 0 && tid == 0) {
            st->ex = ex;
            st->mode = mode;
        }
    } else {
        mode = st->mode;
        ex = st->ex;
        prefix = st->prefix;
        pmask = st->pmask;
    }
    if (mode != 2) return;  // no prefix to find (the same decision in every CTA)
    const int per = (a.L + gridDim.x - 1) / gridDim.x;
    const int t0 = min(a.L, (int)blockIdx.x * per), t1 = min(a.L, t0 + per);
    radix_hist<true>(a.s + t0, t1 - t0, nullptr, prefix, pmask, sh, nbins, ex, nullptr, hl);
    const size_t hb = (size_t)P * kHistBins;
    for (int i = tid; i < nbins; i += blockDim.x) {
        const unsigned long long m = limb_mass(hl, i);
        if (m) atomicAdd(&a.gmass[hb + i], m);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&st->done[P], 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // ---- the last CTA: every CTA's bins are in global memory
    constexpr int BPT = nbins / kPassThreads;  // bins from the top: thread i owns BPT of them
    unsigned long long mb[BPT], msum = 0;
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        mb[q] = __ldcg(&a.gmass[hb + nbins - 1 - BPT * tid - q]);
        msum += mb[q];
    }
    unsigned long long total;
    const unsigned long long before = block_excl_scan_u64(msum, scr64, &total);
    unsigned long long target, above;
    if (P == 0) {
        // mass to reach, in fixed-point units: ceil(m * T) <= T for m < 1; every
        // comparison below is an exact integer comparison
        target = (unsigned long long)ceil((double)a.mass_thresh * (double)total);
        if (target > total) target = total;
        if (target < 1ull) target = 1ull;
        above = 0ull;
    } else {
        target = st->target;
        above = st->above;
    }
    unsigned long long am = above + before;
#pragma unroll
    for (int q = 0; q < BPT; ++q) {
        if (am < target && am + mb[q] >= target) {
            s_bin = nbins - 1 - BPT * tid - q;
            s_above = am;
        }
        am += mb[q];
    }
    __syncthreads();
    if (tid == 0) {
        prefix |= (uint32_t)s_bin << sh;
        pmask |= (uint32_t)(nbins - 1) << sh;
        st->prefix = prefix;
        st->pmask = pmask;
        st->target = target;
        st->above = s_above;
        if (P == 2) {
            const uint32_t cut = prefix;
            const unsigned long long fq = fixed_mass(__uint_as_float(cut), ex);
            const unsigned long long need = target - s_above;  // >= 1
            st->cut = cut;
            st->take = fq ? (need + fq - 1) / fq : 1ull;
        }
    }
}

// ---------------------------------------------------------------------------
// the selection CTA
// ---------------------------------------------------------------------------

struct SelectArgs {
    const float *s;        // [L] importances
    const float *cmax;     // [ncmax] the norms kernel's per-CTA maxima
    int ncmax;
    int L;
    float mass_thresh;
    int recent_n, min_keep;
    uint8_t *flag;         // [L padded to 4] workspace (used when the keys are not staged)
    const SelState *st;    // the mass passes' result (when not staged)
    int staged;            // 1: keys and flags live in dynamic shared memory (L <= kStageKeys)
    int32_t *sel_idx, *n_sel;
};

__global__ void __launch_bounds__(kSelectThreads) k_mass_select(SelectArgs a) {
    extern __shared__ __align__(16) unsigned char sstage[];  // staged: [L] keys, then [L padded to 4] flags
    __shared__ unsigned hl[3 * kHistBins];
    __shared__ unsigned long long scr64[33];
    __shared__ int scr[34];
    __shared__ float s_red[32];
    __shared__ int s_bin;
    __shared__ unsigned long long s_above_mass;
    __shared__ unsigned s_above_cnt;
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.L;
    // keys and flags: shared memory when they fit (one coalesced pass, eight
    // loads in flight per thread), else the workspace
    const float *sv = a.s;
    uint8_t *fl = a.flag;
    int mode;
    uint32_t cut = 0;
    unsigned long long take = 0;
    if (!a.staged) {
        mode = a.st->mode;
        cut = a.st->cut;
        take = a.st->take;
    } else {
        float *ss = reinterpret_cast<float *>(sstage);
        for (int t0 = tid; t0 < L; t0 += 8 * blockDim.x) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int t = t0 + k * blockDim.x;
                v[k] = t < L ? a.s[t] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int t = t0 + k * blockDim.x;
                if (t < L) ss[t] = v[k];
            }
        }
        sv = ss;
        fl = sstage + (size_t)L * sizeof(float);
        // largest importance (from the norms CTAs) -> fixed-point scale: every
        // value < 2^40 units, so a sum of up to 2^20 values stays below 2^60
        float mx = 0.f;
        for (int i = tid; i < a.ncmax; i += blockDim.x) mx = fmaxf(mx, a.cmax[i]);
        mx = block_max(mx, s_red);  // its barriers also order the staging stores
        int ex = 0;
        if (mx > 0.f) frexpf(mx, &ex);  // mx < 2^ex
        // an all-zero importance vector (zero total mass) keeps every token
        mode = (a.mass_thresh >= 1.f || mx == 0.f) ? 1 : (a.mass_thresh > 0.f ? 2 : 0);
        if (mode == 2) {
            unsigned long long target = 0;
            uint32_t prefix = 0, pmask = 0;
            unsigned long long above_mass = 0;  // mass of the keys above the candidate set
            const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
            // after the first pass the keys of the crossing bin (the only ones
            // the later passes look at) are gathered into the flag area, which
            // is free until the flags are written, when they fit there
            const float *keys = sv;
            int nkeys = L;
            for (int pass = 0; pass < 3; ++pass) {
                const int nbins = 1 << widths[pass];
                if (pass == 1) {
                    const uint32_t *sk = reinterpret_cast<const uint32_t *>(sv);
                    int c = 0;
                    for (int t = tid; t < L; t += blockDim.x) c += (sk[t] & pmask) == prefix;
                    int ncand;
                    int o = block_excl_scan(c, scr, &ncand);
                    if (ncand <= ((L + 3) & ~3) / 4) {
                        uint32_t *cand = reinterpret_cast<uint32_t *>(fl);
                        for (int t = tid; t < L; t += blockDim.x)
                            if ((sk[t] & pmask) == prefix) cand[o++] = sk[t];
                        __syncthreads();
                        keys = reinterpret_cast<const float *>(cand);
                        nkeys = ncand;
                    }
                }
                radix_hist<true>(keys, nkeys, nullptr, prefix, pmask, shifts[pass], nbins, ex, nullptr, hl);
                // bins from the top: thread i owns bins nbins-1-2i and nbins-2-2i
                const int b0 = nbins - 1 - 2 * tid, b1 = b0 - 1;
                const unsigned long long m0 = b0 >= 0 ? limb_mass(hl, b0) : 0ull,
                                         m1 = b1 >= 0 ? limb_mass(hl, b1) : 0ull;
                unsigned long long psum;
                const unsigned long long am = above_mass + block_excl_scan_u64(m0 + m1, scr64, &psum);
                if (pass == 0) {
                    // mass to reach, in fixed-point units: ceil(m * T) <= T for
                    // m < 1; every comparison below is an exact integer comparison
                    target = (unsigned long long)ceil((double)a.mass_thresh * (double)psum);
                    if (target > psum) target = psum;
                    if (target < 1ull) target = 1ull;
                }
                // the first bin (from the top) through which the mass reaches the target
                if (b0 >= 0 && am < target && am + m0 >= target) {
                    s_bin = b0;
                    s_above_mass = am;
                }
                if (b1 >= 0 && am + m0 < target && am + m0 + m1 >= target) {
                    s_bin = b1;
                    s_above_mass = am + m0;
                }
                __syncthreads();
                prefix |= (uint32_t)s_bin << shifts[pass];
                pmask |= (uint32_t)(nbins - 1) << shifts[pass];
                above_mass = s_above_mass;
                __syncthreads();
            }
            cut = prefix;
            const unsigned long long fq = fixed_mass(__uint_as_float(cut), ex);
            const unsigned long long need = target - above_mass;  // >= 1
            take = fq ? (need + fq - 1) / fq : 1ull;
        }
    }
    // ---- mass prefix: mode 0 none, 1 every token, 2 down to `cut` (taking
    // `take` of the keys equal to it, lowest index first); pad bytes stay 0
    if (mode == 2) {
        for (int t = L + tid; t < ((L + 3) & ~3); t += blockDim.x) fl[t] = 0;
        ordered_take<false>(sv, fl, L, cut, take, scr);
    } else {
        for (int t = tid; t < ((L + 3) & ~3); t += blockDim.x) fl[t] = (mode == 1 && t < L) ? 1 : 0;
        __syncthreads();
    }

    // ---- the last recent_n tokens always run the FFN
    const int tail = a.recent_n < L ? a.recent_n : L;
    for (int t = L - tail + tid; t < L; t += blockDim.x) fl[t] = 1;
    __syncthreads();

    // ---- at least min(min_keep, L) tokens: extend along (s desc, t asc)
    const int nsel = count_flags(fl, L, scr);
    const int want = a.min_keep < L ? a.min_keep : L;
    if (nsel < want) {
        unsigned need = (unsigned)(want - nsel);
        unsigned *hcnt = hl;
        uint32_t prefix = 0, pmask = 0;
        const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
            const int nbins = 1 << widths[pass];
            radix_hist<false>(sv, L, fl, prefix, pmask, shifts[pass], nbins, 0, hcnt, nullptr);
            const int b0 = nbins - 1 - 2 * tid, b1 = b0 - 1;
            const unsigned c0 = b0 >= 0 ? hcnt[b0] : 0u, c1 = b1 >= 0 ? hcnt[b1] : 0u;
            int ctot;
            const unsigned exc = (unsigned)block_excl_scan((int)(c0 + c1), scr, &ctot);
            if (b0 >= 0 && exc < need && exc + c0 >= need) { s_bin = b0; s_above_cnt = exc; }
            if (b1 >= 0 && exc + c0 < need && exc + c0 + c1 >= need) { s_bin = b1; s_above_cnt = exc + c0; }
            __syncthreads();
            prefix |= (uint32_t)s_bin << shifts[pass];
            pmask |= (uint32_t)(nbins - 1) << shifts[pass];
            need -= s_above_cnt;
            __syncthreads();
        }
        ordered_take<true>(sv, fl, L, prefix, need, scr);
    }

    // ---- ordered compaction to ascending indices: each warp owns a chunk of
    // whole flag words, each lane one word (four tokens) per step; positions
    // from a warp scan of the words' popcounts
    {
        const uint32_t *fw = reinterpret_cast<const uint32_t *>(fl);
        const int nwords = (L + 3) / 4, nw = blockDim.x >> 5;
        const int chunk = (((nwords + nw - 1) / nw) + 31) & ~31;
        const int w0 = min(nwords, warp * chunk), w1 = min(nwords, w0 + chunk);
        int c = 0;
        for (int i = w0 + lane; i < w1; i += 32) c += __popc(fw[i]);
        c = (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
        int tot;
        const int wb = block_excl_scan(lane == 0 ? c : 0, scr, &tot);
        int pos = __shfl_sync(0xffffffffu, wb, 0);
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            const uint32_t wv = i < w1 ? fw[i] : 0u;
            const int n = __popc(wv);
            const int incl = warp_incl_scan(n, lane);
            int p = pos + incl - n;
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if ((wv >> (8 * b)) & 1u) a.sel_idx[p++] = 4 * i + b;
            pos += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (tid == 0) a.n_sel[0] = tot;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

SelectPlan make_select_plan(int L, int d) {
    SelectPlan p = {};
    p.L = L;
    p.d = d;
    size_t o = 0;
    p.off_err = o; o = align_up(o + kControlBytes);  // the control block
    p.off_norms = o; o = align_up(o + sizeof(float) * (size_t)L);
    p.off_flag = o; o = align_up(o + (size_t)((L + 3) & ~3));
    p.off_state = o; o = align_up(o + sizeof(SelState));
    p.off_hist = o; o = align_up(o + sizeof(unsigned long long) * 3 * kHistBins);
    p.off_cmax = o; o = align_up(o + sizeof(float) * (size_t)kMaxNormCtas);
    p.total = o;
    return p;
}

sffn_status run_token_select(const void *y_attn, int L, int d, float mass_thresh, int recent_n, int min_keep,
                             int32_t *sel_idx, int32_t *n_sel, void *ws, const SelectPlan &p, cudaStream_t s) {
    char *w = static_cast<char *>(ws);
    float *norms = reinterpret_cast<float *>(w + p.off_norms);
    float *cmax = reinterpret_cast<float *>(w + p.off_cmax);
    SelState *st = reinterpret_cast<SelState *>(w + p.off_state);
    unsigned long long *gmass = reinterpret_cast<unsigned long long *>(w + p.off_hist);
    const int sms = device_sm_count();
    int grid = (L + kNormWarps - 1) / kNormWarps;  // one row per warp while it lasts
    if (grid > kMaxNormCtas) grid = kMaxNormCtas;
    const bool staged = L <= kStageKeys;
    cudaError_t e = launch_k(k_token_norms, dim3(grid), dim3(32 * kNormWarps), 0, s, y_attn, L, d, norms, cmax, st,
                             gmass, staged ? 0 : 1);
    if (e != cudaSuccess) return SFFN_ERR_CUDA;
    if (!staged) {  // the selection CTA cannot hold the keys: the passes run on many CTAs
        PassArgs pa = {};
        pa.s = norms;
        pa.L = L;
        pa.cmax = cmax;
        pa.ncmax = grid;
        pa.mass_thresh = mass_thresh;
        pa.st = st;
        pa.gmass = gmass;
        int pgrid = (L + 2047) / 2048;
        if (pgrid > 2 * sms) pgrid = 2 * sms;
        e = launch_k(k_mass_pass<0>, dim3(pgrid), dim3(kPassThreads), 0, s, pa);
        if (e == cudaSuccess) e = launch_k(k_mass_pass<1>, dim3(pgrid), dim3(kPassThreads), 0, s, pa);
        if (e == cudaSuccess) e = launch_k(k_mass_pass<2>, dim3(pgrid), dim3(kPassThreads), 0, s, pa);
        if (e != cudaSuccess) return SFFN_ERR_CUDA;
    }
    SelectArgs a = {};
    a.s = norms;
    a.cmax = cmax;
    a.ncmax = grid;
    a.L = L;
    a.mass_thresh = mass_thresh;
    a.recent_n = recent_n;
    a.min_keep = min_keep;
    a.flag = reinterpret_cast<uint8_t *>(w + p.off_flag);
    a.st = st;
    a.sel_idx = sel_idx;
    a.n_sel = n_sel;
    a.staged = staged;
    const size_t smem = staged ? (size_t)L * sizeof(float) + (size_t)((L + 3) & ~3) : 0;
    if (staged && set_max_smem((const void *)k_mass_select, (int)(kStageKeys * (sizeof(float) + 1))) != cudaSuccess)
        return SFFN_ERR_CUDA;
    e = launch_k(k_mass_select, dim3(1), dim3(kSelectThreads), smem, s, a);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
