// decode.cu -- activation-sparse gated-FFN decode GEMV kernels (sm_103a).
//
// One decode call runs, in stream order with programmatic dependent launch:
//   gate     gate GEMV over all d_ff neurons + bias + act + score; for exact /
//            threshold gating the per-neuron decision is taken here and each CTA
//            compacts its chunk of neurons into an ascending index list
//            (warp ballot + block prefix sum; no atomics, no inter-CTA waits).
//   select   keep-ratio only: per-token radix select of the k-th largest score
//            over the float bits (no sort), then ordered compaction.
//   updown   persistent grid; every CTA scans the chunk counts, takes an equal
//            share of the active neurons and streams only their W_up rows
//            (dot with x) and W_downT rows (axpy into an fp32 partial held in
//            registers, 8 output columns per thread, 128-bit loads).
//   reduce   fixed-order sum of the per-CTA partials (deterministic), rounding to
//            the output dtype; also writes the per-token ascending active lists.
//
// The gated FFN and the skipping rules follow denseflux ("skipping most of a
// dense FFN", sec. 1 and 5.1-5.3: only active rows of W_up / columns of W_down
// are read, the gate always in full) and the WiSparse write-up (sec. 1.2
// threshold, 2.3 weight-aware score, 3.2 keep-ratio top-k, 3.3 index table
// instead of a bool mask).
#include "common.cuh"
#include "internal.h"

namespace sffn {

// ---------------------------------------------------------------------------
// weight formats: a 16-byte unit of a stored row
// ---------------------------------------------------------------------------

struct WF32 {
    using X = float;                 // activation dtype that goes with these weights
    static constexpr int E = 4;      // elements per 16-byte unit
    static SFFN_DEV void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    static SFFN_DEV float load_x(const void *x, size_t i) { return static_cast<const float *>(x)[i]; }
};

struct WBF16 {
    using X = __nv_bfloat16;
    static constexpr int E = 8;
    static SFFN_DEV void unpack(const uint4 &v, float *f) {
        f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
        f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
        f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
        f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
    }
    static SFFN_DEV float load_x(const void *x, size_t i) {
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(x)[i]);
    }
};

// ---------------------------------------------------------------------------
// down-projection column norms: norms[j] = ||W_downT[j, :]||_2
// ---------------------------------------------------------------------------

template <class W>
__global__ void __launch_bounds__(256) k_down_norms(const void *wdT, int d, int F, float *norms) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (j >= F) return;
    const int units = d / W::E;  // 16-byte units per stored row
    const char *row = static_cast<const char *>(wdT) + (size_t)j * (size_t)units * 16;
    float acc = 0.f;
    for (int u = lane; u < units; u += 32) {
        float f[W::E];
        W::unpack(ldg_stream(row + (size_t)u * 16), f);
#pragma unroll
        for (int e = 0; e < W::E; ++e) acc = fmaf(f[e], f[e], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) norms[j] = sqrtf(acc);
}

// ---------------------------------------------------------------------------
// gate kernel
// ---------------------------------------------------------------------------

struct GateArgs {
    const void *wg, *wu;
    const float *bias, *norms;
    const void *x;        // [nb, d]
    int d, F, nb, R, C;
    int act, mode, score_kind;
    float tau;
    int decide;           // 1: exact / threshold decision + lists here
    float *aeff;          // [nb, F] act value, zeroed where the token is inactive (if decide)
    float *uval;          // [nb, F] u_j (UP only)
    float *score;         // [nb, F] or null
    int *cnt, *lidx;      // chunk counts / chunk-local lists (if decide)
};

constexpr int kGateThreads = 256;
constexpr int kMaxChunk = kGateThreads;  // R <= blockDim so one scan pass compacts a chunk

template <class W, int NB, bool UP>
__global__ void __launch_bounds__(kGateThreads) k_gate(GateArgs a) {
    extern __shared__ float xs[];  // [NB][d] fp32 (tokens >= nb are zero)
    __shared__ uint8_t sflag[kMaxChunk];
    __shared__ int scan_tmp[34];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int d = a.d, F = a.F;
    // x is a call input, complete before this call's first kernel started.
    for (int i = tid; i < NB * d; i += blockDim.x) {
        const int b = i / d;
        xs[i] = b < a.nb ? W::load_x(a.x, (size_t)b * d + (i - b * d)) : 0.f;
    }
    const int row0 = blockIdx.x * a.R;
    const int nrows = min(a.R, F - row0);
    __syncthreads();
    griddep_wait();
    griddep_launch_dependents();

    const int units = d / W::E;  // 16-byte units per row
    const size_t row_bytes = (size_t)units * 16;
    constexpr int BLK = UP ? 8 : 16;  // units in flight per lane per row stream

    for (int r = warp; r < nrows; r += nwarps) {
        const int j = row0 + r;
        const char *pg = static_cast<const char *>(a.wg) + (size_t)j * row_bytes;
        const char *pu = UP ? static_cast<const char *>(a.wu) + (size_t)j * row_bytes : nullptr;
        float accg[NB], accu[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) accg[b] = accu[b] = 0.f;
        for (int u0 = 0; u0 < units; u0 += 32 * BLK) {
            uint4 vg[BLK], vu[UP ? BLK : 1];
#pragma unroll
            for (int i = 0; i < BLK; ++i) {
                const int u = u0 + i * 32 + lane;
                if (u < units) {
                    vg[i] = ldg_stream(pg + (size_t)u * 16);
                    if (UP) vu[i] = ldg_stream(pu + (size_t)u * 16);
                }
            }
#pragma unroll
            for (int i = 0; i < BLK; ++i) {
                const int u = u0 + i * 32 + lane;
                if (u < units) {
                    float fg[W::E];
                    W::unpack(vg[i], fg);
                    float fu[W::E];
                    if (UP) W::unpack(vu[UP ? i : 0], fu);
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float4 *xp = reinterpret_cast<const float4 *>(xs + b * d + u * W::E);
#pragma unroll
                        for (int q = 0; q < W::E / 4; ++q) {
                            const float4 xv = xp[q];
                            accg[b] = fmaf(fg[4 * q + 0], xv.x, accg[b]);
                            accg[b] = fmaf(fg[4 * q + 1], xv.y, accg[b]);
                            accg[b] = fmaf(fg[4 * q + 2], xv.z, accg[b]);
                            accg[b] = fmaf(fg[4 * q + 3], xv.w, accg[b]);
                            if (UP) {
                                accu[b] = fmaf(fu[4 * q + 0], xv.x, accu[b]);
                                accu[b] = fmaf(fu[4 * q + 1], xv.y, accu[b]);
                                accu[b] = fmaf(fu[4 * q + 2], xv.z, accu[b]);
                                accu[b] = fmaf(fu[4 * q + 3], xv.w, accu[b]);
                            }
                        }
                    }
                }
            }
        }
        // every lane gets the full sums; lane b then finishes token b
        float g = 0.f, uu = 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float sg = warp_sum(accg[b]);
            const float su = UP ? warp_sum(accu[b]) : 0.f;
            if (lane == b) { g = sg; uu = su; }
        }
        bool active = false;
        if (lane < a.nb) {
            if (a.bias) g += a.bias[j];
            const float av = act_fn(a.act, g);
            float sc = 0.f;
            if (a.score) {
                const float n = a.norms[j];
                sc = (a.score_kind == SFFN_SCORE_GATE_UP ? fabsf(av * uu) : fabsf(av)) * n;
                a.score[(size_t)lane * F + j] = sc;
            }
            if (a.decide) {
                if (a.mode == SFFN_MODE_EXACT) {
                    active = av != 0.f;
                } else {
                    const float n = a.norms[j];
                    const float s = (a.score_kind == SFFN_SCORE_GATE_UP ? fabsf(av * uu) : fabsf(av)) * n;
                    active = s >= a.tau;
                }
                a.aeff[(size_t)lane * F + j] = active ? av : 0.f;
            } else if (a.aeff) {
                a.aeff[(size_t)lane * F + j] = av;
            }
            if (UP && a.uval) a.uval[(size_t)lane * F + j] = uu;
        }
        const unsigned m = __ballot_sync(0xffffffffu, active);
        if (lane == 0) sflag[r] = (uint8_t)(m & 0xffu);
    }
    if (!a.decide) return;
    __syncthreads();

    // ordered compaction of this chunk, one list per token (+ the union)
    const int nlists = a.nb + (a.nb > 1 ? 1 : 0);
    const uint32_t m = tid < nrows ? sflag[tid] : 0u;
    for (int l = 0; l < nlists; ++l) {
        const int p = l < a.nb ? (int)((m >> l) & 1u) : (int)(m != 0u);
        int total;
        const int pos = block_excl_scan(p, scan_tmp, &total);
        if (p) a.lidx[(size_t)l * F + row0 + pos] = row0 + tid;
        if (tid == 0) a.cnt[(size_t)l * a.C + blockIdx.x] = total;
    }
}

// ---------------------------------------------------------------------------
// keep-ratio selection: k-th largest score by radix select on the float bits
// ---------------------------------------------------------------------------

constexpr int kSelThreads = 1024;

struct KeepArgs {
    const float *score;  // [nb, F]
    float *aeff;         // [nb, F] raw act values -> zeroed outside the selection
    int F, k, nb, C;
    int *cnt, *lidx;
    uint32_t *mask;      // [nb, ceil(F/32)] selection bitmask (nb > 1)
};

// Find, over 2^bits bins scanned from the top, the bin where the running count
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

__global__ void __launch_bounds__(kSelThreads) k_keep_ratio(KeepArgs a) {
    __shared__ unsigned hist[2048];
    __shared__ int tmp[34];
    __shared__ uint32_t smask[2048];  // F <= 65536
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x;
    const int F = a.F;
    const uint32_t *key = reinterpret_cast<const uint32_t *>(a.score + (size_t)b * F);

    // three digit passes: bits 31..21, 20..10, 9..0
    uint32_t prefix = 0, pmask = 0;
    unsigned need = (unsigned)a.k;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass], nbins = 1 << widths[pass];
        for (int i = tid; i < nbins; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int j = tid; j < F; j += blockDim.x) {
            const uint32_t kv = key[j];
            if ((kv & pmask) == prefix) atomicAdd(&hist[(kv >> sh) & (nbins - 1)], 1u);
        }
        __syncthreads();
        unsigned above;
        const int bin = find_cross_bin(hist, nbins, need, &above, tmp);
        prefix |= (uint32_t)bin << sh;
        pmask |= (uint32_t)(nbins - 1) << sh;
        need -= above;
    }
    const uint32_t T = prefix;        // bits of the k-th largest score
    const unsigned take_eq = need;    // how many scores equal to T are kept (lowest index first)

    // ordered compaction over contiguous segments
    const int seg = (F + blockDim.x - 1) / blockDim.x;
    const int j0 = min(F, tid * seg), j1 = min(F, j0 + seg);
    int eq = 0;
    for (int j = j0; j < j1; ++j) eq += key[j] == T;
    int tot;
    const int eq_base = block_excl_scan(eq, tmp, &tot);
    int nsel = 0, eq_seen = 0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t kv = key[j];
        const bool s = kv > T || (kv == T && (unsigned)(eq_base + eq_seen) < take_eq);
        eq_seen += kv == T;
        nsel += s;
    }
    const int sel_base = block_excl_scan(nsel, tmp, &tot);
    const int nw = (F + 31) >> 5;
    for (int i = tid; i < nw; i += blockDim.x) smask[i] = 0;
    __syncthreads();
    int pos = sel_base;
    eq_seen = 0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t kv = key[j];
        const bool s = kv > T || (kv == T && (unsigned)(eq_base + eq_seen) < take_eq);
        eq_seen += kv == T;
        if (s) {
            a.lidx[(size_t)b * F + pos++] = j;
            atomicOr(&smask[j >> 5], 1u << (j & 31));
        } else {
            a.aeff[(size_t)b * F + j] = 0.f;
        }
    }
    __syncthreads();
    for (int c = tid; c < a.C; c += blockDim.x) a.cnt[(size_t)b * a.C + c] = c == 0 ? tot : 0;
    if (a.mask)
        for (int i = tid; i < nw; i += blockDim.x) a.mask[(size_t)b * nw + i] = smask[i];
}

// union of the per-token keep-ratio selections (nb > 1), ascending
__global__ void __launch_bounds__(kSelThreads) k_union(const uint32_t *mask, int nb, int F, int C, int *cnt,
                                                      int *lidx) {
    __shared__ int tmp[34];
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, nw = (F + 31) >> 5;
    const int per = (nw + blockDim.x - 1) / blockDim.x;
    const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
    int n = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t m = 0;
        for (int b = 0; b < nb; ++b) m |= mask[(size_t)b * nw + w];
        n += __popc(m);
    }
    int tot;
    int pos = block_excl_scan(n, tmp, &tot);
    for (int w = w0; w < w1; ++w) {
        uint32_t m = 0;
        for (int b = 0; b < nb; ++b) m |= mask[(size_t)b * nw + w];
        while (m) {
            const int bit = __ffs(m) - 1;
            m &= m - 1;
            lidx[(size_t)nb * F + pos++] = w * 32 + bit;
        }
    }
    for (int c = tid; c < C; c += blockDim.x) cnt[(size_t)nb * C + c] = c == 0 ? tot : 0;
}

// ---------------------------------------------------------------------------
// sparse up / down kernel
// ---------------------------------------------------------------------------

struct UpDownArgs {
    const void *wu, *wdT;
    const void *x;
    int d, F, nb, R, C, list_u;
    const int *cnt, *lidx;
    const float *aeff, *uval;  // uval non-null: u_j already known (gate-and-up score)
    float *part;               // [G2, nb, d]
};

constexpr int kMaxC = 2048;     // max gate CTAs (chunks)

constexpr int kUpDownMaxThreads = 512;   // d_model <= 4096 at 8 columns per thread

template <class W, int NB, bool HAVE_U>
__global__ void __launch_bounds__(kUpDownMaxThreads) k_updown(UpDownArgs a) {
    constexpr int COLS = 8;                 // output columns per thread
    constexpr int UPT = COLS / W::E;        // 16-byte units per thread per row
    constexpr int RB = NB <= 2 ? 8 : 4;     // rows per group (loads in flight)
    extern __shared__ float smf[];
    float *xs = smf;                                              // [NB][d] fp32
    int *coff = reinterpret_cast<int *>(smf + (size_t)NB * a.d);  // [C + 1] exclusive chunk offsets
    int *srow = coff + kMaxC + 1;                                 // this CTA's neuron indices
    __shared__ float red[kUpDownMaxThreads / 32][RB][NB];
    __shared__ float sh[RB][NB];
    __shared__ int tmp[34];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int d = a.d, F = a.F;
    const int col0 = tid * COLS;
    const bool own = col0 < d;

    for (int i = tid; i < NB * d; i += blockDim.x) {
        const int b = i / d;
        xs[i] = b < a.nb ? W::load_x(a.x, (size_t)b * d + (i - b * d)) : 0.f;
    }
    griddep_wait();
    griddep_launch_dependents();

    // exclusive scan of the walked list's chunk counts
    const int *cnt = a.cnt + (size_t)a.list_u * a.C;
    {
        const int per = (a.C + blockDim.x - 1) / blockDim.x;
        const int c0 = min(a.C, tid * per), c1 = min(a.C, c0 + per);
        int s = 0;
        for (int c = c0; c < c1; ++c) s += cnt[c];
        int total;
        int base = block_excl_scan(s, tmp, &total);
        for (int c = c0; c < c1; ++c) { coff[c] = base; base += cnt[c]; }
        if (tid == 0) coff[a.C] = total;
    }
    __syncthreads();
    const int n_u = coff[a.C];
    const int p0 = (int)((long long)blockIdx.x * n_u / gridDim.x);
    const int p1 = (int)((long long)(blockIdx.x + 1) * n_u / gridDim.x);
    const int nr = p1 - p0;
    const int *lidx = a.lidx + (size_t)a.list_u * F;
    for (int q = tid; q < nr; q += blockDim.x) {
        const int p = p0 + q;
        int lo = 0, hi = a.C - 1;  // last chunk c with coff[c] <= p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (coff[mid] <= p) lo = mid; else hi = mid - 1;
        }
        srow[q] = lidx[(size_t)lo * a.R + (p - coff[lo])];
    }
    __syncthreads();

    float acc[NB][COLS];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < COLS; ++e) acc[b][e] = 0.f;

    const size_t row_bytes = (size_t)d * 16 / W::E;
    for (int g0 = 0; g0 < nr; g0 += RB) {
        const int ng = min(RB, nr - g0);
        uint4 dn[RB][UPT], up[HAVE_U ? 1 : RB][UPT];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r < ng && own) {
                const int j = srow[g0 + r];
                const char *pd = static_cast<const char *>(a.wdT) + (size_t)j * row_bytes + (size_t)col0 * 16 / W::E;
#pragma unroll
                for (int q = 0; q < UPT; ++q) dn[r][q] = ldg_stream(pd + q * 16);
                if (!HAVE_U) {
                    const char *pu = static_cast<const char *>(a.wu) + (size_t)j * row_bytes + (size_t)col0 * 16 / W::E;
#pragma unroll
                    for (int q = 0; q < UPT; ++q) up[HAVE_U ? 0 : r][q] = ldg_stream(pu + q * 16);
                }
            } else {
#pragma unroll
                for (int q = 0; q < UPT; ++q) {
                    dn[r][q] = make_uint4(0, 0, 0, 0);
                    if (!HAVE_U) up[HAVE_U ? 0 : r][q] = make_uint4(0, 0, 0, 0);
                }
            }
        }
        if (!HAVE_U) {
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float fu[COLS];
#pragma unroll
                for (int q = 0; q < UPT; ++q) W::unpack(up[HAVE_U ? 0 : r][q], fu + q * W::E);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float s = 0.f;
                    if (own) {
                        const float4 *xp = reinterpret_cast<const float4 *>(xs + (size_t)b * d + col0);
#pragma unroll
                        for (int q = 0; q < COLS / 4; ++q) {
                            const float4 xv = xp[q];
                            s = fmaf(fu[4 * q + 0], xv.x, s);
                            s = fmaf(fu[4 * q + 1], xv.y, s);
                            s = fmaf(fu[4 * q + 2], xv.z, s);
                            s = fmaf(fu[4 * q + 3], xv.w, s);
                        }
                    }
                    s = warp_sum(s);
                    if (lane == 0) red[warp][r][b] = s;
                }
            }
            __syncthreads();
        }
        for (int i = tid; i < RB * NB; i += blockDim.x) {
            const int r = i / NB, b = i - r * NB;
            float h = 0.f;
            if (r < ng && b < a.nb) {
                const int j = srow[g0 + r];
                float u;
                if (HAVE_U) {
                    u = a.uval[(size_t)b * F + j];
                } else {
                    u = 0.f;
                    for (int w = 0; w < nwarps; ++w) u += red[w][r][b];
                }
                h = a.aeff[(size_t)b * F + j] * u;
            }
            sh[r][b] = h;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float fd[COLS];
#pragma unroll
            for (int q = 0; q < UPT; ++q) W::unpack(dn[r][q], fd + q * W::E);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float h = sh[r][b];
#pragma unroll
                for (int e = 0; e < COLS; ++e) acc[b][e] = fmaf(h, fd[e], acc[b][e]);
            }
        }
        // sh is rewritten by the next group: every thread must be done reading it
        // (without HAVE_U the barrier after the partial dots already orders this)
        if (HAVE_U) __syncthreads();
    }
    if (own) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (b < a.nb) {
                float4 *dst = reinterpret_cast<float4 *>(a.part + ((size_t)blockIdx.x * a.nb + b) * d + col0);
                dst[0] = make_float4(acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
                dst[1] = make_float4(acc[b][4], acc[b][5], acc[b][6], acc[b][7]);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// reduction of the partials + per-token active lists
// ---------------------------------------------------------------------------

struct ReduceArgs {
    const float *part;
    int G2, nb, d;
    void *out;
    int out_f32;
    int n_red;                 // CTAs doing the column reduction; the next nb write lists
    int C, R, F;
    const int *cnt, *lidx;
    int32_t *active_idx, *n_active;
};

__global__ void __launch_bounds__(256) k_reduce(ReduceArgs a) {
    __shared__ float4 red[8][32];
    __shared__ int tmp[34];
    __shared__ int coff[kMaxC + 1];
    griddep_wait();
    // last kernel of the call: no early trigger, so the next call sees all writes
    const int tid = threadIdx.x;
    if ((int)blockIdx.x < a.n_red) {
        const int lane = tid & 31, grp = tid >> 5;
        const size_t total = (size_t)a.nb * a.d;
        const size_t c4 = (size_t)blockIdx.x * 128 + lane * 4;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c4 < total) {
            for (int c = grp; c < a.G2; c += 8) {
                const float4 v = *reinterpret_cast<const float4 *>(a.part + (size_t)c * total + c4);
                s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
            }
        }
        red[grp][lane] = s;
        __syncthreads();
        if (grp == 0 && c4 < total) {
            float4 t = red[0][lane];
            for (int g = 1; g < 8; ++g) {
                const float4 v = red[g][lane];
                t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
            }
            if (a.out_f32) {
                *reinterpret_cast<float4 *>(static_cast<float *>(a.out) + c4) = t;
            } else {
                uint2 o;
                o.x = (uint32_t)f32_to_bf16_bits(t.x) | ((uint32_t)f32_to_bf16_bits(t.y) << 16);
                o.y = (uint32_t)f32_to_bf16_bits(t.z) | ((uint32_t)f32_to_bf16_bits(t.w) << 16);
                *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.out) + c4) = o;
            }
        }
        return;
    }
    // per-token list: scan the chunk counts, then copy the chunks in order
    const int b = blockIdx.x - a.n_red;
    const int *cnt = a.cnt + (size_t)b * a.C;
    const int per = (a.C + blockDim.x - 1) / blockDim.x;
    const int c0 = min(a.C, tid * per), c1 = min(a.C, c0 + per);
    int s = 0;
    for (int c = c0; c < c1; ++c) s += cnt[c];
    int total;
    int base = block_excl_scan(s, tmp, &total);
    for (int c = c0; c < c1; ++c) { coff[c] = base; base += cnt[c]; }
    __syncthreads();
    const int *lidx = a.lidx + (size_t)b * a.F;
    int32_t *dst = a.active_idx + (size_t)b * a.F;
    for (int c = 0; c < a.C; ++c) {
        const int n = (c + 1 < a.C ? coff[c + 1] : total) - coff[c];
        for (int i = tid; i < n; i += blockDim.x) dst[coff[c] + i] = lidx[(size_t)c * a.R + i];
    }
    if (tid == 0) a.n_active[b] = total;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

DecodePlan make_decode_plan(int B, int d, int F) {
    DecodePlan p = {};
    p.nb = B;
    p.d = d;
    p.F = F;
    const int sms = device_sm_count();
    int C = 2 * sms;
    if (C > F) C = F;
    int R = (F + C - 1) / C;
    if (R > kMaxChunk) R = kMaxChunk;
    p.R = R;
    p.C = (F + R - 1) / R;
    p.G2 = sms;
    p.nlists = B + (B > 1 ? 1 : 0);
    p.list_u = B > 1 ? B : 0;
    size_t o = 0;
    p.off_err = o; o = align_up(o + sizeof(int32_t));
    p.off_cnt = o; o = align_up(o + sizeof(int) * (size_t)p.nlists * p.C);
    p.off_lidx = o; o = align_up(o + sizeof(int) * (size_t)p.nlists * F);
    p.off_aeff = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_uval = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_score = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_mask = o; o = align_up(o + sizeof(uint32_t) * (size_t)B * ((F + 31) / 32));
    p.off_part = o; o = align_up(o + sizeof(float) * (size_t)p.G2 * B * d);
    p.total = o;
    return p;
}

template <class W, int NB>
static cudaError_t launch_decode_t(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    char *ws = static_cast<char *>(c.ws);
    const sffn_ffn_weights *w = c.w;
    const bool scores_only = c.scores_only != nullptr;
    const bool keep = c.mode == SFFN_MODE_KEEP_RATIO;
    const bool up = c.score == SFFN_SCORE_GATE_UP && (c.mode != SFFN_MODE_EXACT || scores_only);
    int *cnt = reinterpret_cast<int *>(ws + p.off_cnt);
    int *lidx = reinterpret_cast<int *>(ws + p.off_lidx);
    float *aeff = reinterpret_cast<float *>(ws + p.off_aeff);
    float *uval = reinterpret_cast<float *>(ws + p.off_uval);
    float *score = reinterpret_cast<float *>(ws + p.off_score);
    uint32_t *mask = reinterpret_cast<uint32_t *>(ws + p.off_mask);
    float *part = reinterpret_cast<float *>(ws + p.off_part);

    GateArgs ga = {};
    ga.wg = w->w_gate;
    ga.wu = w->w_up;
    ga.bias = w->b_gate;
    ga.norms = w->down_norms;
    ga.x = c.x;
    ga.d = p.d;
    ga.F = p.F;
    ga.nb = p.nb;
    ga.R = p.R;
    ga.C = p.C;
    ga.act = w->act;
    ga.mode = c.mode;
    ga.score_kind = c.score;
    ga.tau = c.param;
    ga.decide = (!scores_only && !keep) ? 1 : 0;
    ga.aeff = scores_only ? nullptr : aeff;
    ga.uval = up && !scores_only ? uval : nullptr;
    ga.score = scores_only ? c.scores_only : (keep ? score : nullptr);
    ga.cnt = cnt;
    ga.lidx = lidx;
    const size_t smem_gate = sizeof(float) * NB * p.d;
    cudaError_t e;
    if (up) {
        e = set_max_smem((const void *)k_gate<W, NB, true>, (int)smem_gate);
        if (e == cudaSuccess) e = launch_k(k_gate<W, NB, true>, dim3(p.C), dim3(kGateThreads), smem_gate, s, ga);
    } else {
        e = set_max_smem((const void *)k_gate<W, NB, false>, (int)smem_gate);
        if (e == cudaSuccess) e = launch_k(k_gate<W, NB, false>, dim3(p.C), dim3(kGateThreads), smem_gate, s, ga);
    }
    if (e != cudaSuccess || scores_only) return e;

    if (keep) {
        KeepArgs ka = {};
        ka.score = score;
        ka.aeff = aeff;
        ka.F = p.F;
        double kk = floor((double)p.F * (double)c.param);
        int k = kk < 1.0 ? 1 : (int)kk;
        if (k > p.F) k = p.F;
        ka.k = k;
        ka.nb = p.nb;
        ka.C = p.C;
        ka.cnt = cnt;
        ka.lidx = lidx;
        ka.mask = p.nb > 1 ? mask : nullptr;
        e = launch_k(k_keep_ratio, dim3(p.nb), dim3(kSelThreads), 0, s, ka);
        if (e != cudaSuccess) return e;
        if (p.nb > 1) {
            e = launch_k(k_union, dim3(1), dim3(kSelThreads), 0, s, (const uint32_t *)mask, p.nb, p.F, p.C, cnt, lidx);
            if (e != cudaSuccess) return e;
        }
    }

    UpDownArgs ua = {};
    ua.wu = w->w_up;
    ua.wdT = w->w_downT;
    ua.x = c.x;
    ua.d = p.d;
    ua.F = p.F;
    ua.nb = p.nb;
    ua.R = p.R;
    ua.C = p.C;
    ua.list_u = p.list_u;
    ua.cnt = cnt;
    ua.lidx = lidx;
    ua.aeff = aeff;
    ua.uval = up ? uval : nullptr;
    ua.part = part;
    const int threads = ((p.d / 8) + 31) / 32 * 32;
    const int max_rows = (p.F + p.G2 - 1) / p.G2 + 1;
    const size_t smem_ud = sizeof(float) * NB * p.d + sizeof(int) * (kMaxC + 1 + max_rows);
    if (up) {
        e = set_max_smem((const void *)k_updown<W, NB, true>, (int)smem_ud);
        if (e == cudaSuccess) e = launch_k(k_updown<W, NB, true>, dim3(p.G2), dim3(threads), smem_ud, s, ua);
    } else {
        e = set_max_smem((const void *)k_updown<W, NB, false>, (int)smem_ud);
        if (e == cudaSuccess) e = launch_k(k_updown<W, NB, false>, dim3(p.G2), dim3(threads), smem_ud, s, ua);
    }
    if (e != cudaSuccess) return e;

    ReduceArgs ra = {};
    ra.part = part;
    ra.G2 = p.G2;
    ra.nb = p.nb;
    ra.d = p.d;
    ra.out = c.out;
    ra.out_f32 = w->wdtype == SFFN_F32;
    ra.n_red = (int)(((size_t)p.nb * p.d + 127) / 128);
    ra.C = p.C;
    ra.R = p.R;
    ra.F = p.F;
    ra.cnt = cnt;
    ra.lidx = lidx;
    ra.active_idx = c.active_idx;
    ra.n_active = c.n_active;
    // keep-ratio lists live in chunk 0 of each token (chunk stride irrelevant there)
    return launch_k(k_reduce, dim3(ra.n_red + p.nb), dim3(256), 0, s, ra);
}

template <class W>
static cudaError_t launch_decode_w(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    if (p.nb == 1) return launch_decode_t<W, 1>(c, p, s);
    if (p.nb == 2) return launch_decode_t<W, 2>(c, p, s);
    if (p.nb <= 4) return launch_decode_t<W, 4>(c, p, s);
    return launch_decode_t<W, 8>(c, p, s);
}

sffn_status run_decode(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    cudaError_t e;
    switch (c.w->wdtype) {
    case SFFN_F32: e = launch_decode_w<WF32>(c, p, s); break;
    case SFFN_BF16: e = launch_decode_w<WBF16>(c, p, s); break;
    default: return SFFN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

sffn_status run_down_norms(const sffn_ffn_weights *w, float *norms, cudaStream_t s) {
    cudaError_t e;
    const dim3 grid((w->d_ff + 7) / 8), block(256);
    switch (w->wdtype) {
    case SFFN_F32: e = launch_k(k_down_norms<WF32>, grid, block, 0, s, w->w_downT, w->d_model, w->d_ff, norms); break;
    case SFFN_BF16: e = launch_k(k_down_norms<WBF16>, grid, block, 0, s, w->w_downT, w->d_model, w->d_ff, norms); break;
    default: return SFFN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
