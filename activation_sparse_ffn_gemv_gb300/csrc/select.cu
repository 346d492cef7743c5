// select.cu -- token selection for the token-selective prefill (sm_103a).
//
// RedKnot (token-selective sparse FFN, bhfrc.com/news/43276): a token's
// importance is the L2 norm of its attention-output row; tokens are taken in
// decreasing importance until their importance sum covers mass_thresh of the
// total (the crossing token included); the last recent_n tokens are always
// kept, at least min_keep tokens are kept, and an all-zero importance vector or
// mass_thresh >= 1 keeps every token.  No sort and no host synchronisation:
//   token_norms  one warp per row, 128-bit loads, fp32 sum of squares (the
//                product of two bf16 values is exact in fp32)
//   mass_select  one CTA: importances are turned into 64-bit fixed point so
//                every mass sum is exact and order independent; a three-pass
//                radix select over the float bits (11 + 11 + 10 bits) with a
//                count and a mass per bin finds the crossing value; ties at the
//                cut go to the lower index; then the recent tail, the min_keep
//                extension (a count radix select over the unselected tokens)
//                and an ordered compaction to ascending indices.
#include "common.cuh"
#include "internal.h"

namespace sffn {

// ---------------------------------------------------------------------------
// importance: s_t = ||y_attn[t, :]||_2
// ---------------------------------------------------------------------------

constexpr int kNormWarps = 8;

__global__ void __launch_bounds__(32 * kNormWarps) k_token_norms(const void *y, int L, int d, float *s) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int units = d / 8;  // 16-byte units of 8 bf16
    const size_t gw = (size_t)blockIdx.x * kNormWarps + (threadIdx.x >> 5);
    const size_t nw = (size_t)gridDim.x * kNormWarps;
    constexpr int U = 8;      // loads in flight per lane
    for (size_t t = gw; t < (size_t)L; t += nw) {
        const char *row = static_cast<const char *>(y) + t * (size_t)units * 16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int u0 = 0; u0 < units; u0 += 32 * U) {
            uint4 v[U];
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int u = u0 + i * 32 + lane;
                v[i] = u < units ? ldg_stream(row + (size_t)u * 16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float lo = bf16lo(w[q]), hi = bf16hi(w[q]);
                    acc[q] = fmaf(lo, lo, acc[q]);
                    acc[q] = fmaf(hi, hi, acc[q]);
                }
            }
        }
        const float tot = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
        if (lane == 0) s[t] = sqrtf(tot);
    }
}

// ---------------------------------------------------------------------------
// selection
// ---------------------------------------------------------------------------

constexpr int kSelectThreads = 1024;

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

struct SelectArgs {
    const float *s;        // [L] importances
    int L;
    float mass_thresh;
    int recent_n, min_keep;
    uint8_t *flag;         // [L] workspace (used when the keys are not staged)
    int staged;            // 1: keys and flags live in dynamic shared memory (L <= kStageKeys)
    int32_t *sel_idx, *n_sel;
};

// Up to this many importances (and their flags) are staged in shared memory,
// so that every pass of the selection reads on-chip memory.
constexpr int kStageKeys = 32768;

// One radix pass over the candidate keys (kv & pmask) == prefix, flag-filtered.
// Histogram counts and (optionally) fixed-point masses per bin of the digit at `sh`.
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

template <bool MASS>
SFFN_DEV void radix_hist(const float *sv, int L, const uint8_t *exclude, uint32_t prefix, uint32_t pmask, int sh,
                         int nbins, int ex, unsigned *hcnt, unsigned long long *hmass) {
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) {
        hcnt[i] = 0;
        if (MASS) hmass[i] = 0;
    }
    __syncthreads();
    // Importances crowd into few bins, so lanes holding the same bin first add up
    // their count and mass inside the warp (match + reduce; a fixed-point mass is
    // below 2^40 and is summed as two 20-bit halves, exactly), then one lane per
    // bin updates shared memory.  The loop is warp-uniform.
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
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            const bool leader = lane == __ffs(peers) - 1;
            if (MASS) {
                const unsigned long long m = bin < nbins ? fixed_mass(v[k], ex) : 0ull;
                const unsigned lo = __reduce_add_sync(peers, (unsigned)(m & 0xFFFFFull));
                const unsigned hi = __reduce_add_sync(peers, (unsigned)(m >> 20));
                if (leader && bin < nbins) atomicAdd(&hmass[bin], ((unsigned long long)hi << 20) + lo);
            }
            if (leader && bin < nbins) atomicAdd(&hcnt[bin], (unsigned)__popc(peers));
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kSelectThreads) k_mass_select(SelectArgs a) {
    extern __shared__ __align__(16) unsigned char sstage[];  // staged: [L] keys, then [L] flags
    __shared__ unsigned hcnt[2048];
    __shared__ unsigned long long hmass[2048];
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
    if (a.staged) {
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
        __syncthreads();
    }

    // maximum importance -> fixed-point scale: every value < 2^40 units, so a
    // sum of up to 2^20 values stays below 2^60
    float mx = 0.f;
    for (int t = tid; t < L; t += blockDim.x) mx = fmaxf(mx, sv[t]);
    mx = warp_max(mx);
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    if (warp == 0) {
        float v = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0.f;
        v = warp_max(v);
        if (lane == 0) s_red[0] = v;
    }
    __syncthreads();
    mx = s_red[0];
    __syncthreads();
    int ex = 0;
    if (mx > 0.f) frexpf(mx, &ex);                     // mx < 2^ex
    unsigned long long part = 0;
    for (int t = tid; t < L; t += blockDim.x) part += fixed_mass(sv[t], ex);
    unsigned long long total;
    block_excl_scan_u64(part, scr64, &total);

    // ---- mass prefix: flag[t] = 1 for the selected prefix
    const bool all = a.mass_thresh >= 1.f || total == 0ull;
    for (int t = tid; t < L; t += blockDim.x) fl[t] = all ? 1 : 0;
    __syncthreads();
    if (!all && a.mass_thresh > 0.f) {
        // mass to reach, in fixed-point units: ceil(m * T) <= T for m < 1; all
        // comparisons below are exact integer comparisons
        unsigned long long target = (unsigned long long)ceil((double)a.mass_thresh * (double)total);
        if (target > total) target = total;
        if (target < 1ull) target = 1ull;
        uint32_t prefix = 0, pmask = 0;
        unsigned long long above_mass = 0;  // mass of the keys above the candidate set
        const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
        for (int pass = 0; pass < 3; ++pass) {
            const int nbins = 1 << widths[pass];
            radix_hist<true>(sv, L, nullptr, prefix, pmask, shifts[pass], nbins, ex, hcnt, hmass);
            // bins from the top: thread i owns bins nbins-1-2i and nbins-2-2i
            const int b0 = nbins - 1 - 2 * tid, b1 = b0 - 1;
            const unsigned long long m0 = b0 >= 0 ? hmass[b0] : 0ull, m1 = b1 >= 0 ? hmass[b1] : 0ull;
            unsigned long long dummy;
            const unsigned long long am = above_mass + block_excl_scan_u64(m0 + m1, scr64, &dummy);
            // crossing: the first bin (from the top) through which the mass reaches the target
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
        const uint32_t cut = prefix;
        const unsigned long long fq = fixed_mass(__uint_as_float(cut), ex);
        const unsigned long long need = target - above_mass;  // >= 1
        const unsigned long long take = fq ? (need + fq - 1) / fq : 1ull;
        // ordered pass over contiguous segments for the equal keys
        const int seg = (L + blockDim.x - 1) / blockDim.x;
        const int t0 = min(L, tid * seg), t1 = min(L, t0 + seg);
        int eq = 0;
        for (int t = t0; t < t1; ++t) eq += __float_as_uint(sv[t]) == cut;
        int eqtot;
        const int eqb = block_excl_scan(eq, scr, &eqtot);
        int seen = 0;
        for (int t = t0; t < t1; ++t) {
            const uint32_t kv = __float_as_uint(sv[t]);
            const bool in = kv > cut || (kv == cut && (unsigned long long)(eqb + seen) < take);
            seen += kv == cut;
            fl[t] = in ? 1 : 0;
        }
        __syncthreads();
    }

    // ---- the last recent_n tokens always run the FFN
    const int tail = a.recent_n < L ? a.recent_n : L;
    for (int t = L - tail + tid; t < L; t += blockDim.x) fl[t] = 1;
    __syncthreads();

    // ---- at least min(min_keep, L) tokens: extend along (s desc, t asc)
    int cnt_local = 0;
    for (int t = tid; t < L; t += blockDim.x) cnt_local += fl[t];
    int nsel;
    block_excl_scan(cnt_local, scr, &nsel);
    const int want = a.min_keep < L ? a.min_keep : L;
    if (nsel < want) {
        unsigned need = (unsigned)(want - nsel);
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
        const uint32_t cut = prefix;
        const int seg = (L + blockDim.x - 1) / blockDim.x;
        const int t0 = min(L, tid * seg), t1 = min(L, t0 + seg);
        int eq = 0;
        for (int t = t0; t < t1; ++t) eq += !fl[t] && __float_as_uint(sv[t]) == cut;
        int eqtot;
        const int eqb = block_excl_scan(eq, scr, &eqtot);
        int seen = 0;
        for (int t = t0; t < t1; ++t) {  // each thread updates only its own segment
            if (fl[t]) continue;
            const uint32_t kv = __float_as_uint(sv[t]);
            const bool in = kv > cut || (kv == cut && (unsigned)(eqb + seen) < need);
            seen += kv == cut;
            if (in) fl[t] = 1;
        }
        __syncthreads();
    }

    // ---- ordered compaction to ascending indices
    {
        const int seg = (L + blockDim.x - 1) / blockDim.x;
        const int t0 = min(L, tid * seg), t1 = min(L, t0 + seg);
        int c = 0;
        for (int t = t0; t < t1; ++t) c += fl[t] != 0;
        int tot;
        int pos = block_excl_scan(c, scr, &tot);
        for (int t = t0; t < t1; ++t)
            if (fl[t]) a.sel_idx[pos++] = t;
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
    p.off_flag = o; o = align_up(o + (size_t)L);
    p.total = o;
    return p;
}

sffn_status run_token_select(const void *y_attn, int L, int d, float mass_thresh, int recent_n, int min_keep,
                             int32_t *sel_idx, int32_t *n_sel, void *ws, const SelectPlan &p, cudaStream_t s) {
    char *w = static_cast<char *>(ws);
    float *norms = reinterpret_cast<float *>(w + p.off_norms);
    const int sms = device_sm_count();
    int grid = (L + kNormWarps - 1) / kNormWarps;
    if (grid > 4 * sms) grid = 4 * sms;
    cudaError_t e = launch_k(k_token_norms, dim3(grid), dim3(32 * kNormWarps), 0, s, y_attn, L, d, norms);
    if (e != cudaSuccess) return SFFN_ERR_CUDA;
    SelectArgs a = {};
    a.s = norms;
    a.L = L;
    a.mass_thresh = mass_thresh;
    a.recent_n = recent_n;
    a.min_keep = min_keep;
    a.flag = reinterpret_cast<uint8_t *>(w + p.off_flag);
    a.sel_idx = sel_idx;
    a.n_sel = n_sel;
    a.staged = L <= kStageKeys;
    const size_t smem = a.staged ? (size_t)L * (sizeof(float) + 1) : 0;
    if (a.staged && set_max_smem((const void *)k_mass_select, (int)(kStageKeys * (sizeof(float) + 1))) != cudaSuccess)
        return SFFN_ERR_CUDA;
    e = launch_k(k_mass_select, dim3(1), dim3(kSelectThreads), smem, s, a);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
