// decode_finish.cuh -- the end of a fused decode call, shared by the decode
// kernels: a bounded grid barrier over the call's CTAs, then the fixed-order
// sum of the per-CTA fp32 partials into the output and the per-token ascending
// lists of active neurons at their global positions.
#pragma once

#include "common.cuh"

namespace sffn {

struct FinishArgs {
    unsigned *gbar;       // [2]: arrivals (never reset), arrivals before this call
    const float *part;    // [gridDim.x, nb, d] fp32 partials, one per CTA
    int nb, d, F;
    int C, R;             // chunks (one per CTA) and rows per chunk
    const int *cnt;       // [nb, C] active rows per chunk, or null (no lists)
    const int *lidx;      // [nb, F] chunk-local ascending lists at row0 of each chunk
    void *out;
    int out_f32;
    int32_t *active_idx, *n_active;
    int32_t *err;
    int nr_cap = 0;  // > 0: at most this many reducers
};

// Called by all threads (>= 256) of every CTA of the call once the CTA's
// partial (and its chunk's counts and lists) are written.  Only the first NR
// CTAs (enough for one 32-column block and four chunk lists each) finish the
// call; the others count their arrival and return at once, so that the next
// call's CTAs can take their SMs while the output is formed.  The reducers are
// resident (one CTA per SM, grid <= #SMs); the wait is bounded all the same.
// gbar[0] counts arrivals and is never reset; this call's barrier opens once it
// has grown by gridDim.x past the base (unsigned differences, so wrap-around is
// harmless).
// Release add / acquire load of a grid-barrier counter at GPU scope.
SFFN_DEV void red_release_add(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
SFFN_DEV unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

SFFN_DEV void finish_call(const FinishArgs &a, unsigned bar_base, bool failed) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t total = (size_t)a.nb * a.d;
    int NR = (int)min((size_t)gridDim.x, max((total + 31) / 32, (size_t)(gridDim.x + 3) / 4));
    if (a.nr_cap > 0 && a.nr_cap < NR) NR = a.nr_cap;
    __shared__ int s_bar_ok;
    __shared__ float red[8][32];
    // The arrival is one release add at GPU scope after a CTA barrier: every
    // write of the CTA (partials, counts, lists) happens before it.  A reducer
    // polls with acquire loads and passes the result on through a CTA barrier.
    __syncthreads();
    if ((int)blockIdx.x >= NR) {
        if (tid == 0) red_release_add(a.gbar, 1u);
        return;
    }
    if (tid == 0) {
        red_release_add(a.gbar, 1u);
        int ok = 1;
        if (ld_acquire(a.gbar) - bar_base < gridDim.x) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire(a.gbar) - bar_base < gridDim.x)
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    ok = 0;
                    record_error(a.err, SFFN_ERR_TIMEOUT);
                    break;
                }
        }
        s_bar_ok = ok;
    }
    __syncthreads();
    // every CTA read the base before it arrived: the next call's base can be
    // published now (the next call reads it after this grid has completed)
    if (blockIdx.x == 0 && tid == 0) *reinterpret_cast<volatile unsigned *>(a.gbar + 1) = bar_base + gridDim.x;
    if (!s_bar_ok || failed) return;

    const int C = gridDim.x;
    // ---- output: this CTA's 32-column blocks i = 0, 1, 2, ... at columns
    // (blockIdx.x + NR i) * 32.  Warps 0..3 take the even i, warps 4..7 (after
    // the lists) the odd i; within a group the partials are summed in a fixed
    // order (warp w of the group adds partials w, w + 4, ... with all its loads
    // in flight at once; then the group's 4 warps in order).
    auto reduce = [&](int grp) {
        const int wl = warp & 3;
        for (int i = grp; (size_t)(blockIdx.x + (size_t)NR * i) * 32 < total; i += 2) {
            const size_t col = (size_t)(blockIdx.x + (size_t)NR * i) * 32 + lane;
            float sum = 0.f;
            if (col < total) {
                float v[40];
#pragma unroll
                for (int q = 0; q < 40; ++q) {
                    const int pp = wl + 4 * q;
                    v[q] = pp < C ? __ldcg(a.part + (size_t)pp * total + col) : 0.f;
                }
#pragma unroll
                for (int q = 0; q < 40; ++q) sum += v[q];
                for (int pp = wl + 160; pp < C; pp += 4) sum += __ldcg(a.part + (size_t)pp * total + col);
            }
            red[warp][lane] = sum;
            named_barrier_sync(1 + grp, 128);
            if (wl == 0 && col < total) {
                const int w0 = 4 * grp;
                const float t = ((red[w0][lane] + red[w0 + 1][lane]) + red[w0 + 2][lane]) + red[w0 + 3][lane];
                if (a.out_f32) static_cast<float *>(a.out)[col] = t;
                else static_cast<uint16_t *>(a.out)[col] = f32_to_bf16_bits(t);
            }
            named_barrier_sync(1 + grp, 128);
        }
    };
    if (warp < 4) {
        reduce(0);
    } else if (warp < 8) {
        if (a.cnt) {
            // ---- the ascending index lists of chunks r, r + NR, ... at their
            // global positions; warps 4..7 share the (chunk, token) pairs
            const int nmine_c = ((int)C - (int)blockIdx.x + NR - 1) / NR;
            for (int q = warp - 4; q < nmine_c * a.nb; q += 4) {
                const int c = (int)blockIdx.x + (q / a.nb) * NR, b = q % a.nb;
                const int crow0 = c * a.R;
                const int *cnt = a.cnt + (size_t)b * a.C;
                // counts of the earlier chunks (C <= 256: 8 per lane, in flight
                // together) and the chunk's entries (R <= 256: 8 per lane)
                // A count outside [0, R] or a list that would end past d_ff means the
                // control block was not a valid start (e.g. not zero-filled before
                // first use, so the barrier opened early): record it, write nothing.
                int cv[8], ev[8];
                const int mine = __ldcg(cnt + c);
                int bad = mine < 0 || mine > a.R;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int cc = lane + 32 * i, e = lane + 32 * i;
                    cv[i] = cc < c ? __ldcg(cnt + cc) : 0;
                    bad |= cv[i] < 0 || cv[i] > a.R;
                    ev[i] = e < a.R && crow0 + e < a.F ? __ldcg(a.lidx + (size_t)b * a.F + crow0 + e) : 0;
                }
                int sacc = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) sacc += cv[i];
                const int off = __reduce_add_sync(0xffffffffu, sacc);
                if (__any_sync(0xffffffffu, bad) || off < 0 || off + mine > a.F) {
                    if (lane == 0) record_error(a.err, SFFN_ERR_DEVICE);
                    continue;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = lane + 32 * i;
                    if (e < mine) a.active_idx[(size_t)b * a.F + off + e] = ev[i];
                }
                if (c == C - 1 && lane == 0) a.n_active[b] = off + mine;
            }
        }
        reduce(1);
    }
}

}  // namespace sffn
