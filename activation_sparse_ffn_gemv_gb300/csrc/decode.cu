// decode.cu -- activation-sparse gated-FFN decode GEMV kernels (sm_103a).
//
// One decode call runs, in stream order with programmatic dependent launch:
//   exact / threshold gating: one kernel (k_gate) streams the whole gate (and,
//            for active neurons only, W_up and W_downT rows), decides, builds the
//            ascending per-token lists, accumulates per-CTA partials and, with
//            every CTA resident, finishes the output behind a bounded grid
//            barrier (fixed-order sum: deterministic).  With more chunks than
//            SMs, k_reduce finishes instead.
//   keep-ratio: k_gate writes the scores; k_keep_ratio selects the k largest
//            per token by radix select over the float bits (no sort); k_updown /
//            k_down stream the selected W_up / W_downT rows into per-CTA
//            partials; k_reduce sums them in a fixed order and writes the lists.
//
// The gated FFN and the skipping rules follow denseflux ("skipping most of a
// dense FFN", sec. 1 and 5.1-5.3: only active rows of W_up / columns of W_down
// are read, the gate always in full) and the WiSparse write-up (sec. 1.2
// threshold, 2.3 weight-aware score, 3.2 keep-ratio top-k, 3.3 index table
// instead of a bool mask).
#include "common.cuh"
#include "decode_finish.cuh"
#include "internal.h"
#include "topk.cuh"
#include "wformat.cuh"

#include <algorithm>

namespace sffn {

// ---------------------------------------------------------------------------
// down-projection column norms: norms[j] = ||W_downT[j, :]||_2
// ---------------------------------------------------------------------------

template <class W>
__global__ void __launch_bounds__(256) k_down_norms(const void *wdT, const void *sdT, int d, int F, float *norms) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int j = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (j >= F) return;
    const int units = d / W::E;  // 16-byte units per stored row
    const char *row = static_cast<const char *>(wdT) + (size_t)j * (size_t)units * 16;
    const unsigned char *srow = W::Q ? static_cast<const unsigned char *>(sdT) + (size_t)j * (d / 64) * 2 : nullptr;
    float acc = 0.f;
    for (int u = lane; u < units; u += 32) {
        float f[W::E];
        W::dequant(ldg_stream(row + (size_t)u * 16), W::Q ? W::scale_at(srow, u) : 1.f, f);
#pragma unroll
        for (int e = 0; e < W::E; ++e) acc = fmaf(f[e], f[e], acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) norms[j] = sqrtf(acc);
}

// ---------------------------------------------------------------------------
// gate kernel
// ---------------------------------------------------------------------------
//
// One CTA per SM owns R consecutive neurons (a "chunk").  Warp w of the CTA
// streams rows w, w + 8, w + 16, ... of the chunk through its own ring of D
// shared-memory stages (1-D bulk copies issued by its lane 0, one mbarrier per
// stage) and forms the gate dot products (and, for the gate-and-up score, the
// up dot products) against x held in registers, then bias, act, score and the
// decision.  For the exact and threshold rules the item the warp puts into its
// ring after an active row is that neuron's W_up row, so u_j and h_j = a_j u_j
// are known when the gate stream ends; the neuron's W_downT row is prefetched
// into L2 at the decision.  After the stream each CTA compacts its chunk into
// ascending per-token lists, bulk-loads its active W_downT rows into the idle
// ring and accumulates its fp32 partial of the output.  When all CTAs are
// resident (grid <= #SMs) they then meet at a bounded grid barrier, sum
// 32-column blocks of the partials in a fixed order and write their chunk's
// lists; otherwise k_reduce does that.  Every wait is time-bounded; on a
// timeout the CTA records SFFN_ERR_TIMEOUT, lets its own copies in flight land
// and skips the rest of its work.

struct GateArgs {
    const void *wg, *wu;
    const float *bias, *norms;
    const void *x;        // [nb, d]
    int d, F, nb, R, C;
    int act, mode, score_kind;
    float tau;
    int decide;           // 1: exact / threshold decision, lists and h here
    int stages;           // rows in flight per warp (its ring stages)
    float *aeff;          // !decide: [nb, F] raw act values (or null)
    float *uval;          // !decide, UP: [nb, F] u_j (or null)
    float *score;         // [nb, F] or null
    int *cnt, *lidx;      // decide: chunk counts / chunk-local ascending lists
    int32_t *err;
    const void *wdT;      // decide: down projection, read for this chunk's active rows
    float *part;          // decide: [C, nb, d] this CTA's fp32 partial of the output
    const void *sg, *su, *sd;  // int4: fp16 group scales [F, d/64] of gate, up, down
    // fused final reduction (all CTAs co-resident): grid barrier words in the
    // workspace, the output and the per-token index lists
    unsigned *gbar;            // [2]: arrivals (never reset), arrivals before this call
    void *out;
    int out_f32;
    int32_t *active_idx, *n_active;
    // the first pf_early CTAs send rows 0 .. pf_rows-1 of the later chunks to L2
    // before their dependency wait (0: none)
    int pf_early, pf_rows;
};

constexpr int kGateWarps = 8;           // each warp streams its own rows
constexpr int kGatePfRows = 48;         // rows of each later chunk sent to L2 by the early CTAs
constexpr int kGateThreads = 32 * kGateWarps;
constexpr int kMaxChunk = 256;   // R <= kMaxChunk <= blockDim: one scan pass compacts a chunk
constexpr int kMaxStages = 16;   // ring stages per warp
constexpr int kMaxChunks = 256;  // C <= kMaxChunks <= blockDim: one scan pass over the chunk counts
constexpr int kUpItem = 1 << 16; // ring item tag: the W_up row of the neuron in the low bits

// Bytes of the gate kernel's mbarrier block (one per stage, one for the active
// rows' copies after the stream), 128-byte aligned.
SFFN_HOST_DEV uint32_t gate_bar_bytes(int D) { return ((uint32_t)((kGateWarps * D + 1) * 8) + 127u) & ~127u; }

// Dot products of one stored row (and, with TWO, a second row) with the nb
// tokens' activations: each lane takes units lane, lane + 32, ... (d_model <=
// 4096), four independent accumulators per token and row.  x comes from
// registers (xr, one token) or shared memory (xs).
template <class W, int NB, bool TWO, bool XREG>
SFFN_DEV void row_dots(const unsigned char *ra, const unsigned char *rb, uint32_t units, uint32_t row_bytes,
                       const float *xr, const uint4 *xs, uint32_t xunits, float (&acca)[NB][4],
                       float (&accb)[NB][4]) {
    constexpr int UPL = 128 / W::E;         // units per lane at d_model <= 4096
    constexpr int CU = W::E >= 32 ? 1 : 4;  // units loaded together (ILP)
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int c = 0; c < 4; ++c) acca[b][c] = accb[b][c] = 0.f;
#pragma unroll
    for (int i0 = 0; i0 < UPL; i0 += CU) {
        uint4 va[CU], vb[CU];
        float sa[CU], sb[CU];
#pragma unroll
        for (int c = 0; c < CU; ++c) {
            const uint32_t u = (i0 + c) * 32 + lane;
            const bool in = u < units;
            va[c] = in ? *reinterpret_cast<const uint4 *>(ra + u * 16) : make_uint4(0, 0, 0, 0);
            sa[c] = W::Q && in ? W::scale_at(ra + row_bytes, u) : 1.f;
            if (TWO) {
                vb[c] = in ? *reinterpret_cast<const uint4 *>(rb + u * 16) : make_uint4(0, 0, 0, 0);
                sb[c] = W::Q && in ? W::scale_at(rb + row_bytes, u) : 1.f;
            }
        }
#pragma unroll
        for (int c = 0; c < CU; ++c) {
            const uint32_t u = (i0 + c) * 32 + lane;
            if constexpr (W::Q) {
                // group-scaled codes: the unit's 32 exact small-integer codes are
                // dotted with x, then multiplied by the group scale once
                float fa[W::E], fb[W::E];
                W::codes(va[c], fa);
                if (TWO) W::codes(vb[c], fb);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float xf[W::E];
                    if (XREG) {
#pragma unroll
                        for (int e = 0; e < W::E; ++e) xf[e] = xr[(i0 + c) * W::E + e];
                    } else if (u < units) {
                        W::load_xu(xs + (size_t)b * xunits, u, xf);
                    } else {
#pragma unroll
                        for (int e = 0; e < W::E; ++e) xf[e] = 0.f;
                    }
                    float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int e = 0; e < W::E; ++e) {
                        pa[e & 3] = fmaf(fa[e], xf[e], pa[e & 3]);
                        if (TWO) pb[e & 3] = fmaf(fb[e], xf[e], pb[e & 3]);
                    }
                    const int ai = (i0 + c) & 3;
                    acca[b][ai] = fmaf(sa[c], (pa[0] + pa[1]) + (pa[2] + pa[3]), acca[b][ai]);
                    if (TWO) accb[b][ai] = fmaf(sb[c], (pb[0] + pb[1]) + (pb[2] + pb[3]), accb[b][ai]);
                }
                continue;
            }
            float fa[W::E], fb[W::E];
            W::dequant(va[c], sa[c], fa);
            if (TWO) W::dequant(vb[c], sb[c], fb);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                float xf[W::E];
                if (XREG) {
#pragma unroll
                    for (int e = 0; e < W::E; ++e) xf[e] = xr[(i0 + c) * W::E + e];
                } else if (u < units) {
                    W::load_xu(xs + (size_t)b * xunits, u, xf);
                } else {
#pragma unroll
                    for (int e = 0; e < W::E; ++e) xf[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < W::E; ++e) {
                    const int ai = CU == 1 ? (e & 3) : c;
                    acca[b][ai] = fmaf(fa[e], xf[e], acca[b][ai]);
                    if (TWO) accb[b][ai] = fmaf(fb[e], xf[e], accb[b][ai]);
                }
            }
        }
        if ((i0 + CU) * 32 >= (int)units) break;
    }
}

template <class W, int NB, bool UP>
__global__ void __launch_bounds__(kGateThreads, 1) k_gate(GateArgs a) {
    extern __shared__ __align__(128) unsigned char smraw[];
    const int d = a.d, F = a.F;
    const uint32_t units = (uint32_t)(d / W::E);  // 16-byte units per row
    const uint32_t row_bytes = units * 16u;
    const uint32_t sbytes = W::Q ? (uint32_t)(d / 64) * 2u : 0u;  // group scales of one row
    const uint32_t rspace = row_bytes + sbytes;    // a row (codes, then scales) in shared memory
    const uint32_t stage_bytes = UP ? 2u * rspace : rspace;
    const uint32_t xunits = (uint32_t)(d * (int)sizeof(typename W::X) / 16);
    const int D = a.stages;                        // stages (items in flight) per warp
    // dynamic shared memory: [warps][D] + 1 mbarriers | [warps][D] stages | x
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw);
    uint64_t *dbar = full + (size_t)kGateWarps * D;  // active-row copies after the stream
    const uint32_t bar_bytes = gate_bar_bytes(D);
    unsigned char *ring = smraw + bar_bytes;
    unsigned char *xraw = ring + (size_t)kGateWarps * D * stage_bytes;
    const uint4 *xs = reinterpret_cast<const uint4 *>(xraw);   // x in its own dtype [NB][d]
    __shared__ int sitem[kGateWarps][kMaxStages];  // item in each stage: row, | kUpItem for its W_up row
    __shared__ uint8_t sflag[kMaxChunk];
    __shared__ float sh[kMaxChunk][NB];
    __shared__ float sbias[kMaxChunk], snorm[kMaxChunk];
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row0 = blockIdx.x * a.R;
    const int nrows = min(a.R, F - row0);
    // warp w handles rows w, w + 8, w + 16, ... of the chunk
    const int nmine = nrows > warp ? (nrows - warp + kGateWarps - 1) / kGateWarps : 0;
    const bool up_items = a.decide && !UP;  // W_up rows of active neurons join the stream
    uint64_t *wfull = full + (size_t)warp * D;
    unsigned char *wring = ring + (size_t)warp * D * stage_bytes;
    int *witem = sitem[warp];
    const char *gbase = static_cast<const char *>(a.wg) + (size_t)row0 * row_bytes;
    const char *ubase = static_cast<const char *>(a.wu) + (size_t)row0 * row_bytes;
    const char *gsbase = W::Q ? static_cast<const char *>(a.sg) + (size_t)row0 * sbytes : nullptr;
    const char *usbase = W::Q ? static_cast<const char *>(a.su) + (size_t)row0 * sbytes : nullptr;
    uint64_t pol = 0;
    // Put item `it` into stage s (lane 0): gate row codes [+ scales] [+ up row
    // codes [+ scales]], or one W_up row for an up item.
    auto issue = [&](int s, int it) {
        unsigned char *stage = wring + (size_t)s * stage_bytes;
        uint64_t *bar = &wfull[s];
        const size_t r = (size_t)(it & (kUpItem - 1));
        witem[s] = it;
        if (it & kUpItem) {
            mbar_arrive_expect_tx(bar, rspace);
            bulk_load(stage, ubase + r * row_bytes, row_bytes, bar, pol);
            if (W::Q) bulk_load(stage + row_bytes, usbase + r * sbytes, sbytes, bar, pol);
            return;
        }
        mbar_arrive_expect_tx(bar, stage_bytes);
        bulk_load(stage, gbase + r * row_bytes, row_bytes, bar, pol);
        if (W::Q) bulk_load(stage + row_bytes, gsbase + r * sbytes, sbytes, bar, pol);
        if (UP) {
            bulk_load(stage + rspace, ubase + r * row_bytes, row_bytes, bar, pol);
            if (W::Q) bulk_load(stage + rspace + row_bytes, usbase + r * sbytes, sbytes, bar, pol);
        }
    };
    // Each warp keeps its own D items in flight and re-issues as soon as it has
    // consumed one: no producer warp, so a slow warp never holds back another
    // warp's stream.  Item i always sits in stage i % D.  Weights are constant
    // inputs: they stream before the dependency wait.
    int issued = min(D, nmine);  // items issued by this warp (warp-uniform)
    int gnext = issued;          // gate rows issued: the warp's rows 0 .. gnext-1
    if (lane == 0) {
        for (int i = 0; i < D; ++i) mbar_init(&wfull[i], 1);
        mbar_fence_init();
        pol = l2_evict_first_policy();
        for (int i = 0; i < issued; ++i) issue(i, warp + i * kGateWarps);
    }
    if (tid == 0) {
        s_abort = 0;
        mbar_init(dbar, 1);
        mbar_fence_init();
    }
    // When calls follow each other, the first CTAs of this call find free SMs
    // (the previous call's CTAs that do not reduce have left) while the
    // previous call's reducers still hold the others.  Those early CTAs send the
    // first rows of the later chunks to L2, so that HBM streams through that
    // gap and the later CTAs' first ring items are L2 hits.  Chunk c >= E is
    // covered by early CTA c % E; the rows go out in row order across chunks.
    if (a.pf_early > 0 && (int)blockIdx.x < a.pf_early && warp == kGateWarps - 1) {
        const int E = a.pf_early;
        const int nch = (a.C - 1 - (int)blockIdx.x) / E;  // chunks blockIdx.x + E m, m = 1 .. nch
        const int P = min(a.pf_rows, a.R);
        const char *wg = static_cast<const char *>(a.wg);
        for (int i = lane; i < nch * P; i += 32) {
            const int r = i / nch, c = (int)blockIdx.x + (1 + i % nch) * E;
            const int j = c * a.R + r;
            if (j < F) {
                bulk_prefetch_l2(wg + (size_t)j * row_bytes, row_bytes);
                if (W::Q) bulk_prefetch_l2(static_cast<const char *>(a.sg) + (size_t)j * sbytes, sbytes);
            }
        }
    }
    // x may be the previous layer's output: read it only after the dependency wait
    griddep_wait();
    // the reduction may be scheduled now (its small CTAs fit beside this one)
    griddep_launch_dependents();
    // grid-barrier base: arrivals counted before this call (moves only after
    // every CTA of this call has arrived)
    const unsigned bar_base = a.gbar ? *reinterpret_cast<volatile unsigned *>(a.gbar + 1) : 0u;
    {
        constexpr int XE = 16 / (int)sizeof(typename W::X);
        const int per_row = d / XE, total = NB * per_row;
        uint4 *dst = reinterpret_cast<uint4 *>(xraw);
        for (int u = tid; u < total; u += blockDim.x)
            dst[u] = u / per_row < a.nb ? ldg_v4(static_cast<const char *>(a.x) + (size_t)u * 16)
                                        : make_uint4(0, 0, 0, 0);
        for (int i = tid; i < nrows; i += blockDim.x) {
            sbias[i] = a.bias ? a.bias[row0 + i] : 0.f;
            snorm[i] = a.norms ? a.norms[row0 + i] : 0.f;
        }
    }
    __syncthreads();
    {
        // This lane always handles units lane, lane + 32, ... of a row: for one
        // token its slice of x is unpacked into registers once and reused for
        // every row.  Units per lane <= UPL (d_model <= 4096).
        constexpr int UPL = 128 / W::E;
        constexpr bool XREG = NB == 1;
        float xr[XREG ? UPL * W::E : 1];
        if (XREG) {
#pragma unroll
            for (int i = 0; i < UPL; ++i) {
                const uint32_t u = i * 32 + lane;
                float f[W::E];
                if (u < units) {
                    W::load_xu(xs, u, f);
                } else {
#pragma unroll
                    for (int e = 0; e < W::E; ++e) f[e] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < W::E; ++e) xr[XREG ? i * W::E + e : 0] = f[e];
            }
        }
        for (int k = 0; k < issued; ++k) {
            const int si = k % D;
            const bool ok = mbar_wait(&wfull[si], (uint32_t)(k / D) & 1u);
            if (!__all_sync(0xffffffffu, ok && !s_abort)) {
                // a wait timed out here or in another warp: record it, let this
                // warp's own copies in flight land (bounded), then stop
                if (lane == 0) {
                    if (!ok) {
                        s_abort = 1;
                        record_error(a.err, SFFN_ERR_TIMEOUT);
                    }
                    for (int kk = k; kk < issued; ++kk) mbar_wait(&wfull[kk % D], (uint32_t)(kk / D) & 1u);
                }
                __syncwarp();
                break;
            }
            const int it = witem[si];
            const int r = it & (kUpItem - 1);
            const unsigned char *st = wring + (size_t)si * stage_bytes;
            int next = -1;  // the item that goes into the ring after this one
            if (it & kUpItem) {
                // W_up row of an active neuron: u_j per token, h_j = a_j u_j
                float acu[NB][4], unused[NB][4];
                row_dots<W, NB, false, XREG>(st, nullptr, units, row_bytes, xr, xs, xunits, acu, unused);
                __syncwarp();
                if (gnext < nmine) next = warp + (gnext++) * kGateWarps;
                if (lane == 0 && next >= 0) {
                    fence_proxy_async_smem();
                    issue(issued % D, next);
                }
                float uu = 0.f;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float t = warp_sum((acu[b][0] + acu[b][1]) + (acu[b][2] + acu[b][3]));
                    if (lane == b) uu = t;
                }
                if (lane < a.nb) sh[r][lane] = ((sflag[r] >> lane) & 1u) ? sh[r][lane] * uu : 0.f;
                if (next >= 0) ++issued;
                continue;
            }
            float accg[NB][4], accu[NB][4];
            row_dots<W, NB, UP, XREG>(st, st + rspace, units, row_bytes, xr, xs, xunits, accg, accu);
            __syncwarp();
            if (!up_items) {
                // stage consumed: refill it now with this warp's next gate row
                if (gnext < nmine) next = warp + (gnext++) * kGateWarps;
                if (lane == 0 && next >= 0) {
                    fence_proxy_async_smem();
                    issue(issued % D, next);
                }
                if (next >= 0) ++issued;
            }
            float g = 0.f, uu = 0.f;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float sg = warp_sum((accg[b][0] + accg[b][1]) + (accg[b][2] + accg[b][3]));
                const float su = UP ? warp_sum((accu[b][0] + accu[b][1]) + (accu[b][2] + accu[b][3])) : 0.f;
                if (lane == b) { g = sg; uu = su; }
            }
            const int j = row0 + r;
            bool active = false;
            float av = 0.f;
            if (lane < a.nb) {
                g += sbias[r];
                av = act_fn(a.act, g);
                float sc = 0.f;
                if (a.score || (a.decide && a.mode != SFFN_MODE_EXACT)) {
                    sc = (a.score_kind == SFFN_SCORE_GATE_UP ? fabsf(av * uu) : fabsf(av)) * snorm[r];
                    if (a.score) a.score[(size_t)lane * F + j] = sc;
                }
                if (a.decide) {
                    active = a.mode == SFFN_MODE_EXACT ? av != 0.f : sc >= a.tau;
                } else {
                    if (a.aeff) a.aeff[(size_t)lane * F + j] = av;
                    if (UP && a.uval) a.uval[(size_t)lane * F + j] = uu;
                }
            }
            if (!a.decide) continue;
            const unsigned m = __ballot_sync(0xffffffffu, active) & 0xffu;
            // UP: h_j = a_j u_j now; otherwise the masked a_j, times u_j when the
            // W_up row (the next item) arrives
            if (lane < NB) sh[r][lane] = active ? (UP ? av * uu : av) : 0.f;
            if (lane == 0) sflag[r] = (uint8_t)m;
            if (up_items) {
                if (m != 0u) next = r | kUpItem;
                else if (gnext < nmine) next = warp + (gnext++) * kGateWarps;
                if (lane == 0 && next >= 0) {
                    fence_proxy_async_smem();
                    issue(issued % D, next);
                }
                if (next >= 0) ++issued;
            }
            if (m != 0u && lane == 0) {
                bulk_prefetch_l2(static_cast<const char *>(a.wdT) + (size_t)j * row_bytes, row_bytes);
                if (W::Q) bulk_prefetch_l2(static_cast<const char *>(a.sd) + (size_t)j * sbytes, sbytes);
            }
            __syncwarp();  // sh / sflag of this row before a later up item of the warp reads them
        }
    }
    __syncthreads();
    // after a timed-out copy the CTA still meets the grid barrier (so that the
    // barrier words stay consistent) but streams nothing more
    if (!a.decide || (s_abort && !a.gbar)) return;
    bool failed = s_abort;

    // ordered compaction of this chunk: one list per token for the active_idx
    // output, and (in shared memory) the chunk's rows active for any token
    // (row r = tid; R <= 256: one ballot per warp and list, one pass).  A row
    // of the union that falls in the first batch starts the bulk copy of its
    // W_downT row (sent to L2 at the decision) into its ring slot right away.
    const int cap = (int)((size_t)kGateWarps * D * stage_bytes / rspace);
    const char *wd = static_cast<const char *>(a.wdT);
    const char *sd = static_cast<const char *>(a.sd);
    __shared__ int sdown[kMaxChunk];
    __shared__ int s_ndown;
    __shared__ int wcnt[NB + 1][kGateWarps];
    const uint32_t m = tid < nrows ? sflag[tid] : 0u;
    for (int l = 0; l <= a.nb; ++l) {
        const bool bit = l < a.nb ? ((m >> l) & 1u) : m != 0u;
        const unsigned bl = __ballot_sync(0xffffffffu, bit);
        if (lane == 0) wcnt[l][warp] = __popc(bl);
    }
    __syncthreads();
    {
        const unsigned lt = (1u << lane) - 1u;
        for (int l = 0; l <= a.nb; ++l) {
            const bool bit = l < a.nb ? ((m >> l) & 1u) : m != 0u;
            const unsigned bl = __ballot_sync(0xffffffffu, bit);
            int base = 0, tot = 0;
#pragma unroll
            for (int w = 0; w < kGateWarps; ++w) {
                base += w < warp ? wcnt[l][w] : 0;
                tot += wcnt[l][w];
            }
            const int pos = base + __popc(bl & lt);
            if (bit) {
                if (l < a.nb) {
                    a.lidx[(size_t)l * F + row0 + pos] = row0 + tid;
                } else {
                    sdown[pos] = tid;
                    if (pos < cap && !failed) {
                        const size_t j = (size_t)(row0 + tid);
                        unsigned char *dslot = ring + (size_t)pos * rspace;
                        const uint64_t dpol = l2_evict_first_policy();
                        fence_proxy_async_smem();  // the ring's reads passed the barrier above
                        asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(dbar)),
                                     "r"(rspace)
                                     : "memory");
                        bulk_load(dslot, wd + j * row_bytes, row_bytes, dbar, dpol);
                        if (W::Q) bulk_load(dslot + row_bytes, sd + j * sbytes, sbytes, dbar, dpol);
                    }
                }
            }
            if (tid == 0) {
                if (l < a.nb) a.cnt[(size_t)l * a.C + blockIdx.x] = tot;
                else s_ndown = tot;
            }
        }
    }
    __syncthreads();

    // Active neurons of this chunk (h_j already known), in batches that fit the
    // idle ring: their W_downT rows come from L2 (prefetched at the decision) by
    // bulk copy in one round trip; then every thread owns 16-byte column units
    // and accumulates h_j * W_down[:, j] over the rows in ascending order
    // (deterministic) into this CTA's partial.
    const int ndown = failed ? 0 : s_ndown;
    for (int b0 = 0, batch = 0;; b0 += cap, ++batch) {
        const int bn = min(cap, ndown - b0);
        if (bn > 0) {
            if (tid == 0 && batch == 0) {
                mbar_arrive(dbar);  // the rows raised the count and started their copies
            } else if (tid == 0) {
                fence_proxy_async_smem();  // earlier generic reads of the ring precede the copies
                const uint64_t pol = l2_evict_first_policy();
                mbar_arrive_expect_tx(dbar, (uint32_t)bn * rspace);
                for (int i = 0; i < bn; ++i) {
                    const size_t j = (size_t)(row0 + sdown[b0 + i]);
                    unsigned char *dslot = ring + (size_t)i * rspace;
                    bulk_load(dslot, wd + j * row_bytes, row_bytes, dbar, pol);
                    if (W::Q) bulk_load(dslot + row_bytes, sd + j * sbytes, sbytes, dbar, pol);
                }
            }
            const bool ok = mbar_wait(dbar, (uint32_t)batch & 1u);
            if (!__syncthreads_and(ok)) {
                if (tid == 0) record_error(a.err, SFFN_ERR_TIMEOUT);
                failed = true;
                break;
            }
        }
        for (uint32_t u = tid; u < units; u += blockDim.x) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b >= a.nb) break;
                float acc[W::E];
#pragma unroll
                for (int e = 0; e < W::E; ++e) acc[e] = 0.f;
                for (int i = 0; i < bn; ++i) {
                    const float h = sh[sdown[b0 + i]][b];
                    const unsigned char *dr = ring + (size_t)i * rspace;
                    float f[W::E];
                    W::dequant(*reinterpret_cast<const uint4 *>(dr + u * 16), W::Q ? W::scale_at(dr + row_bytes, u) : 1.f, f);
#pragma unroll
                    for (int e = 0; e < W::E; ++e) acc[e] = fmaf(h, f[e], acc[e]);
                }
                float4 *dst = reinterpret_cast<float4 *>(a.part + ((size_t)blockIdx.x * a.nb + b) * d + u * W::E);
#pragma unroll
                for (int q = 0; q < W::E / 4; ++q) {
                    float4 v = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
                    if (batch > 0) {
                        const float4 o = dst[q];
                        v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
                    }
                    dst[q] = v;
                }
            }
        }
        if (b0 + cap >= ndown) break;
        __syncthreads();  // the next batch overwrites the ring
    }
    if (!a.gbar) return;
    FinishArgs fa;
    fa.gbar = a.gbar; fa.part = a.part; fa.nb = a.nb; fa.d = d; fa.F = F; fa.C = a.C; fa.R = a.R;
    fa.cnt = a.cnt; fa.lidx = a.lidx; fa.out = a.out; fa.out_f32 = a.out_f32; fa.active_idx = a.active_idx;
    fa.n_active = a.n_active; fa.err = a.err;
    finish_call(fa, bar_base, failed);
}

// ---------------------------------------------------------------------------
// keep-ratio selection: k-th largest score by radix select on the float bits
// ---------------------------------------------------------------------------

constexpr int kSelThreads = 1024;

struct KeepArgs {
    const float *score;  // [nb, F]
    float *aeff;         // [nb, F] raw act values -> zeroed outside the selection
    const float *uval;   // [nb, F] u_j when known (gate-and-up score), else null
    float *lh;           // with uval: h = a * u aligned with the token's list (nb == 1)
    int F, k, nb, C;
    int *cnt, *lidx;
    uint32_t *mask;      // [nb, ceil(F/32)] selection bitmask (nb > 1)
    const int32_t *core; // the layer's core set (always kept; the top-k runs on the rest), or null
    int n_core;
    int32_t *err;        // the workspace's error word (a core index out of range)
};

// Scores of one token are staged in shared memory up to this many neurons.
constexpr int kKeepStage = 40960;

// One CTA per token.  The token's scores are staged in shared memory (when F
// fits) for the top-k (topk.cuh).  With a core set the core columns are always
// kept and the select takes the k - |core| largest scores of the other columns
// (none when the core holds k or more).  The ordered pass writes the token's
// ascending list, its mask words, and zeroes a_j outside the selection.
__global__ void __launch_bounds__(kSelThreads) k_keep_ratio(KeepArgs a) {
    extern __shared__ __align__(16) uint32_t skey[];  // [F] staged score bits (F <= kKeepStage)
    __shared__ unsigned hist[2048];
    __shared__ int tmp[34];
    __shared__ uint32_t fmask[2048];  // the core as a bitmask (F <= 65536)
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const int F = a.F, nwords = (F + 31) >> 5;
    const uint32_t *key = reinterpret_cast<const uint32_t *>(a.score + (size_t)b * F);
    if (F <= kKeepStage) {
        stage_keys(skey, key, F);
        key = skey;
    }
    const uint32_t *forced = nullptr;
    unsigned kk = (unsigned)a.k;
    if (a.core) {
        for (int i = tid; i < nwords; i += blockDim.x) fmask[i] = 0u;
        __syncthreads();
        for (int q = tid; q < a.n_core; q += blockDim.x) {
            const int j = a.core[q];
            if (j >= 0 && j < F) atomicOr(&fmask[j >> 5], 1u << (j & 31));
            else if (b == 0) record_error(a.err, SFFN_ERR_DEVICE);
        }
        __syncthreads();
        int c = 0;
        for (int i = tid; i < nwords; i += blockDim.x) c += __popc(fmask[i]);
        int c_eff;
        block_excl_scan(c, tmp, &c_eff);
        kk = kk > (unsigned)c_eff ? kk - (unsigned)c_eff : 0u;
        forced = fmask;
    }
    const TopkCut cut = radix_topk(key, F, kk, forced, hist, tmp);

    const bool want_h = a.lh && a.nb == 1;  // h_j = a_j * u_j for the selected neurons
    // a_j outside the selection is read only through the union of B > 1 tokens
    const bool zero_rest = a.nb > 1;
    float *aeff = a.aeff + (size_t)b * F;
    int32_t *lidx = a.lidx + (size_t)b * F;
    if (key == skey && cut.take_eq == cut.n_eq) {
        // Every candidate equal to the cut is taken (no tie straddles it), so the
        // selection is key >= T or forced and needs no count of the keys before a
        // warp's chunk: one pass ranks each warp's selections into its own,
        // already-read stretch of the staged keys; then the warps' offsets, and
        // the lists and h_j are written with all their loads in flight.
        __shared__ int wtot[32];
        const int warp = tid >> 5, nw = blockDim.x >> 5;
        const int wchunk = (nwords + nw - 1) / nw;
        const int w0 = min(nwords, warp * wchunk), w1 = min(nwords, w0 + wchunk);
        uint32_t *buf = skey + 32 * w0;
        const unsigned lt = (1u << lane) - 1u;
        int nsel = 0;
        for (int w = w0; w < w1; ++w) {
            const int j = 32 * w + lane;
            const bool ok = j < F;
            const uint32_t kv = ok ? skey[j] : 0u;
            const bool sel = ok && (bit_at(forced, j) || kv >= cut.T);
            const unsigned bal = __ballot_sync(0xffffffffu, sel);
            __syncwarp();  // every lane has read this word's key before any is overwritten
            if (sel) buf[nsel + __popc(bal & lt)] = (uint32_t)j;
            else if (zero_rest && ok) aeff[j] = 0.f;
            nsel += __popc(bal);
            if (lane == 0 && a.mask) a.mask[(size_t)b * nwords + w] = bal;
        }
        if (lane == 0) wtot[warp] = nsel;
        __syncthreads();
        int off = 0, total = 0;
        for (int v = 0; v < nw; ++v) {
            off += v < warp ? wtot[v] : 0;
            total += wtot[v];
        }
        constexpr int UC = 4;
        for (int i0 = 0; i0 < nsel; i0 += 32 * UC) {
            int jj[UC];
            float av[UC], uv[UC];
#pragma unroll
            for (int q = 0; q < UC; ++q) {
                const int i = i0 + 32 * q + lane;
                jj[q] = i < nsel ? (int)buf[i] : -1;
            }
#pragma unroll
            for (int q = 0; q < UC; ++q) {
                av[q] = want_h && jj[q] >= 0 ? aeff[jj[q]] : 0.f;
                uv[q] = want_h && jj[q] >= 0 ? a.uval[jj[q]] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < UC; ++q) {
                const int i = i0 + 32 * q + lane;
                if (jj[q] < 0) continue;
                lidx[off + i] = jj[q];
                if (want_h) a.lh[off + i] = av[q] * uv[q];
            }
        }
        for (int c = tid; c < a.C; c += blockDim.x) a.cnt[(size_t)b * a.C + c] = c == 0 ? total : 0;
        return;
    }
    TopkChunk ch = topk_chunk(key, F, forced, cut, tmp);
    constexpr int U = 4;  // mask words per step: their selections first, then the a_j, u_j loads together
    for (int w = ch.w0; w < ch.w1; w += U) {
        TopkWord t[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            t[q] = TopkWord{false, 0, 0u};
            if (w + q < ch.w1) t[q] = topk_word(key, F, forced, cut, w + q, ch);
        }
        float av[U], uv[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int j = 32 * (w + q) + lane;
            av[q] = want_h && t[q].sel ? aeff[j] : 0.f;
            uv[q] = want_h && t[q].sel ? a.uval[j] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            if (w + q >= ch.w1) break;
            const int j = 32 * (w + q) + lane;
            if (t[q].sel) {
                if (want_h) a.lh[t[q].pos] = av[q] * uv[q];
                lidx[t[q].pos] = j;
            } else if (zero_rest && j < F) {
                aeff[j] = 0.f;
            }
            if (lane == 0 && a.mask) a.mask[(size_t)b * nwords + w + q] = t[q].bal;
        }
    }
    for (int c = tid; c < a.C; c += blockDim.x) a.cnt[(size_t)b * a.C + c] = c == 0 ? ch.total : 0;
}

// union of the per-token keep-ratio selections (nb > 1), ascending
__global__ void __launch_bounds__(kSelThreads) k_union(const uint32_t *mask, int nb, int F, int C, int *cnt,
                                                      int *lidx, const float *aeff, const float *uval, float *lh) {
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
            const int j = w * 32 + bit;
            if (lh)  // aeff is already zero where a token did not select j
                for (int b = 0; b < nb; ++b) lh[(size_t)b * F + pos] = aeff[(size_t)b * F + j] * uval[(size_t)b * F + j];
            lidx[(size_t)nb * F + pos++] = j;
        }
    }
    for (int c = tid; c < C; c += blockDim.x) cnt[(size_t)nb * C + c] = c == 0 ? tot : 0;
}

// ---------------------------------------------------------------------------
// sparse up / down kernel
// ---------------------------------------------------------------------------

struct UpDownArgs {
    const void *wu, *wdT;
    const void *su, *sdT;      // int4: fp16 group scales of W_up / W_downT rows
    const void *x;
    int d, F, nb, R, C, list_u;
    const int *cnt, *lidx;
    const float *aeff, *uval;  // uval non-null: u_j already known (gate-and-up score)
    float *part;               // [G2, nb, d]
    int32_t *active_idx;       // nb == 1: the walked list is the token's own list; write it here
    int32_t *n_active;
    unsigned *gbar;            // non-null: finish the call here (grid barrier, sum of the partials)
    void *out;
    int out_f32;
    int32_t *err;
};

// The end of a keep-ratio call inside its down kernel: every CTA is resident
// (grid <= #SMs) and the token's list is already written, so the CTAs meet at
// the grid barrier and sum the partials (decode_finish.cuh) without a list.
template <class A>
SFFN_DEV void finish_partials(const A &a, int d, unsigned bar_base) {
    FinishArgs fa = {};
    fa.gbar = a.gbar;
    fa.part = a.part;
    fa.nb = a.nb;
    fa.d = d;
    fa.F = a.F;
    fa.C = a.C;
    fa.R = a.R;
    fa.out = a.out;
    fa.out_f32 = a.out_f32;
    fa.err = a.err;
    finish_call(fa, bar_base, false);
}

constexpr int kMaxC = 2048;     // max gate CTAs (chunks)
constexpr int kListChunks = 8;  // chunks per list-writing CTA of the reduction

constexpr int kUpDownMaxThreads = 512;   // d_model <= 4096 at 8 columns per thread

template <class W, int NB, bool HAVE_U>
__global__ void __launch_bounds__(kUpDownMaxThreads) k_updown(UpDownArgs a) {
    constexpr int COLS = 8;                 // output columns per thread (load_row8)
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

    stage_x<W>(xs, a.x, a.nb, NB, d);
    griddep_wait();
    griddep_launch_dependents();
    const unsigned bar_base = a.gbar ? *reinterpret_cast<volatile unsigned *>(a.gbar + 1) : 0u;

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
        const int j = lidx[(size_t)lo * a.R + (p - coff[lo])];
        srow[q] = j;
        if (a.active_idx) a.active_idx[p] = j;
    }
    if (a.n_active && blockIdx.x == 0 && tid == 0) a.n_active[0] = n_u;
    __syncthreads();

    float acc[NB][COLS];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < COLS; ++e) acc[b][e] = 0.f;

    const size_t row_bytes = (size_t)d * 16 / W::E;
    for (int g0 = 0; g0 < nr; g0 += RB) {
        const int ng = min(RB, nr - g0);
        Row8 dn[RB], up[HAVE_U ? 1 : RB];
        float ds[RB], us[HAVE_U ? 1 : RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            dn[r] = Row8{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            ds[r] = 0.f;
            if (!HAVE_U) {
                up[HAVE_U ? 0 : r] = dn[r];
                us[HAVE_U ? 0 : r] = 0.f;
            }
            if (r < ng && own) {
                const int j = srow[g0 + r];
                dn[r] = load_row8<W>(static_cast<const char *>(a.wdT) + (size_t)j * row_bytes, col0);
                ds[r] = row_scale8<W>(a.sdT, (size_t)j, d, col0);
                if (!HAVE_U) {
                    up[HAVE_U ? 0 : r] = load_row8<W>(static_cast<const char *>(a.wu) + (size_t)j * row_bytes, col0);
                    us[HAVE_U ? 0 : r] = row_scale8<W>(a.su, (size_t)j, d, col0);
                }
            }
        }
        if (!HAVE_U) {
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                float fu[COLS];
                unpack_row8<W>(up[HAVE_U ? 0 : r], us[HAVE_U ? 0 : r], fu);
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
            unpack_row8<W>(dn[r], ds[r], fd);
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
    if (a.gbar) finish_partials(a, d, bar_base);
}

// ---------------------------------------------------------------------------
// sparse down kernel: h_j already known
// ---------------------------------------------------------------------------
//
// Persistent grid.  Each CTA takes an equal share of the walked list's
// entries (j, h_j[b]), then every thread owns 8 output columns and issues the
// 16-byte W_downT loads of all its rows at once (one memory round trip for the
// usual handful of rows per CTA), accumulating h_j * W_down[:, j] in fp32.

struct DownArgs {
    const void *wdT;
    const void *sdT;           // int4: fp16 group scales of the W_downT rows
    int d, F, nb, R, C, list_u;
    int by_chunk;              // 1: CTA c walks gate chunk c (grid == C); 0: equal shares of the list
    int max_rows;              // capacity of the row list in shared memory
    const int *cnt, *lidx;
    const float *lh;           // [nb, F] aligned with list list_u
    float *part;               // [G2, nb, d]
    int32_t *active_idx;       // nb == 1: write the token's list here
    int32_t *n_active;
    unsigned *gbar;            // non-null: finish the call here (grid barrier, sum of the partials)
    void *out;
    int out_f32;
    int32_t *err;
};



constexpr int kDownMaxThreads = 512;

template <class W, int NB>
__global__ void __launch_bounds__(kDownMaxThreads) k_down(DownArgs a) {
    constexpr int COLS = 8;  // output columns per thread (load_row8)
    constexpr int RB = NB <= 2 ? 16 : 8;
    extern __shared__ int smi[];
    int *coff = smi;                                   // [C + 1]
    int *srow = smi + kMaxC + 1;                       // [max_rows]
    __shared__ int tmp[34];
    const int tid = threadIdx.x;
    const int d = a.d, F = a.F;
    const int col0 = tid * COLS;
    const bool own = col0 < d;
    float *shv = reinterpret_cast<float *>(srow + a.max_rows);  // [max_rows][NB]

    griddep_wait();
    griddep_launch_dependents();
    const unsigned bar_base = a.gbar ? *reinterpret_cast<volatile unsigned *>(a.gbar + 1) : 0u;
    const int *cnt = a.cnt + (size_t)a.list_u * a.C;
    const int *lidx = a.lidx + (size_t)a.list_u * F;
    int nr;
    if (a.by_chunk) {
        // this CTA's rows are exactly gate chunk blockIdx.x: no scan before the loads
        const int c = blockIdx.x;
        nr = cnt[c];
        for (int q = tid; q < nr; q += blockDim.x) {
            const size_t pos = (size_t)c * a.R + q;
            srow[q] = lidx[pos];
            for (int b = 0; b < NB; ++b) shv[q * NB + b] = b < a.nb ? a.lh[(size_t)b * F + pos] : 0.f;
        }
        __syncthreads();
    } else {
        const int per = (a.C + blockDim.x - 1) / blockDim.x;
        const int c0 = min(a.C, tid * per), c1 = min(a.C, c0 + per);
        int s = 0;
        for (int c = c0; c < c1; ++c) s += cnt[c];
        int total;
        int base = block_excl_scan(s, tmp, &total);
        for (int c = c0; c < c1; ++c) { coff[c] = base; base += cnt[c]; }
        if (tid == 0) coff[a.C] = total;
        __syncthreads();
        const int n_u = coff[a.C];
        const int p0 = (int)((long long)blockIdx.x * n_u / gridDim.x);
        const int p1 = (int)((long long)(blockIdx.x + 1) * n_u / gridDim.x);
        nr = p1 - p0;
        for (int q = tid; q < nr; q += blockDim.x) {
            const int p = p0 + q;
            int lo = 0, hi = a.C - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (coff[mid] <= p) lo = mid; else hi = mid - 1;
            }
            const size_t pos = (size_t)lo * a.R + (p - coff[lo]);
            const int j = lidx[pos];
            srow[q] = j;
            for (int b = 0; b < NB; ++b) shv[q * NB + b] = b < a.nb ? a.lh[(size_t)b * F + pos] : 0.f;
            if (a.active_idx) a.active_idx[p] = j;
        }
        if (a.n_active && blockIdx.x == 0 && tid == 0) a.n_active[0] = n_u;
        __syncthreads();
    }

    float acc[NB][COLS];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < COLS; ++e) acc[b][e] = 0.f;
    const size_t row_bytes = (size_t)d * 16 / W::E;
    // all threads run the same control flow (the scan below has barriers);
    // threads beyond the last column only skip their loads and stores
    for (int g0 = 0; g0 < nr; g0 += RB) {
        Row8 dn[RB];
        float ds[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            dn[r] = Row8{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            ds[r] = 0.f;
            if (own && g0 + r < nr) {
                const int j = srow[g0 + r];
                dn[r] = load_row8<W>(static_cast<const char *>(a.wdT) + (size_t)j * row_bytes, col0);
                ds[r] = row_scale8<W>(a.sdT, (size_t)j, d, col0);
            }
        }
        if (a.by_chunk && g0 == 0) {
            // while the first loads are in flight: this chunk's position in the
            // token's ascending list = exclusive prefix of the earlier chunks' counts
            int sacc = 0;
            for (int c = tid; c < (int)blockIdx.x; c += blockDim.x) sacc += cnt[c];
            int total;
            block_excl_scan(sacc, tmp, &total);
            if (a.active_idx)
                for (int q = tid; q < nr; q += blockDim.x) a.active_idx[total + q] = srow[q];
            if (a.n_active && blockIdx.x == gridDim.x - 1 && tid == 0) a.n_active[0] = total + nr;
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (g0 + r < nr) {
                float fd[COLS];
                unpack_row8<W>(dn[r], ds[r], fd);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float h = shv[(g0 + r) * NB + b];
#pragma unroll
                    for (int e = 0; e < COLS; ++e) acc[b][e] = fmaf(h, fd[e], acc[b][e]);
                }
            }
        }
    }
    if (a.by_chunk && nr == 0) {  // no rows: still publish this chunk's list position
        int sacc = 0;
        for (int c = tid; c < (int)blockIdx.x; c += blockDim.x) sacc += cnt[c];
        int total;
        block_excl_scan(sacc, tmp, &total);
        if (a.n_active && blockIdx.x == gridDim.x - 1 && tid == 0) a.n_active[0] = total;
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
    if (a.gbar) finish_partials(a, d, bar_base);
}

// ---------------------------------------------------------------------------
// reduction of the partials + per-token active lists
// ---------------------------------------------------------------------------

struct ReduceArgs {
    const float *part;
    int G2, nb, d;
    void *out;
    int out_f32;
    int n_red;                 // CTAs doing the column reduction; the next ones write per-token lists
    int C, R, F;
    const int *cnt, *lidx;
    int32_t *active_idx, *n_active;
};

__global__ void __launch_bounds__(256) k_reduce(ReduceArgs a) {
    __shared__ float red[8][32];
    __shared__ int tmp[34];
    griddep_wait();
    // The next call's first kernel may start now: before its own dependency
    // wait it only streams weights, which no kernel of this library writes.
    griddep_launch_dependents();
    const int tid = threadIdx.x;
    if ((int)blockIdx.x < a.n_red) {
        // 32 consecutive outputs per CTA; 8 groups each sum every 8th partial
        // (fixed assignment and order: deterministic)
        const int lane = tid & 31, grp = tid >> 5;
        const size_t total = (size_t)a.nb * a.d;
        const size_t c = (size_t)blockIdx.x * 32 + lane;
        float s = 0.f;
        if (c < total) {
            // every load in flight at once (G2 <= 8 * 32); summed in a fixed order
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int p = grp + 8 * i;
                v[i] = p < a.G2 ? a.part[(size_t)p * total + c] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) s += v[i];
            for (int p = grp + 256; p < a.G2; p += 8) s += a.part[(size_t)p * total + c];
        }
        red[grp][lane] = s;
        __syncthreads();
        if (grp == 0 && c < total) {
            float t = red[0][lane];
#pragma unroll
            for (int g = 1; g < 8; ++g) t += red[g][lane];
            if (a.out_f32) static_cast<float *>(a.out)[c] = t;
            else static_cast<uint16_t *>(a.out)[c] = f32_to_bf16_bits(t);
        }
        return;
    }
    // Per-token ascending lists: each list CTA owns kListChunks consecutive
    // chunks of one token; its offset is the sum of the earlier chunks' counts
    // (a warp-parallel sum), then a warp per chunk copies the chunk's entries.
    const int li = blockIdx.x - a.n_red;
    const int groups = (a.C + kListChunks - 1) / kListChunks;
    const int b = li / groups, grp = li - b * groups;
    const int c0 = grp * kListChunks, c1 = min(a.C, c0 + kListChunks);
    const int *cnt = a.cnt + (size_t)b * a.C;
    int s = 0;
    for (int c = tid; c < c0; c += blockDim.x) s += cnt[c];
    int base;
    block_excl_scan(s, tmp, &base);   // base = total over the CTA = offset of chunk c0
    const int lane = tid & 31, wp = tid >> 5;
    __shared__ int ccnt[kListChunks], coffs[kListChunks];
    if (tid == 0) {
        int o = base;
        for (int c = c0; c < c1; ++c) {
            ccnt[c - c0] = cnt[c];
            coffs[c - c0] = o;
            o += cnt[c];
        }
        if (c1 == a.C) a.n_active[b] = o;
    }
    __syncthreads();
    const int *lidx = a.lidx + (size_t)b * a.F;
    int32_t *dst = a.active_idx + (size_t)b * a.F;
    // (a count or offset outside the token's list is never written)
    for (int c = c0 + wp; c < c1; c += blockDim.x >> 5) {
        const int n = ccnt[c - c0], o = coffs[c - c0];
        if (n >= 0 && n <= 128 && o >= 0 && o + n <= a.F)
            for (int i = lane; i < n; i += 32) dst[o + i] = lidx[(size_t)c * a.R + i];
    }
    for (int c = c0; c < c1; ++c) {  // long lists (keep-ratio: the whole list sits in chunk 0)
        const int n = ccnt[c - c0], o = coffs[c - c0];
        if (n > 128 && o >= 0 && o + n <= a.F)
            for (int i = tid; i < n; i += blockDim.x) dst[o + i] = lidx[(size_t)c * a.R + i];
    }
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
    int C = sms < kMaxChunks ? sms : kMaxChunks;  // one gate CTA per SM
    if (C > F) C = F;
    int R = (F + C - 1) / C;
    if (R > kMaxChunk) R = kMaxChunk;
    p.R = R;
    p.C = (F + R - 1) / R;
    p.G2 = sms;
    p.nlists = B + (B > 1 ? 1 : 0);
    p.list_u = B > 1 ? B : 0;
    size_t o = 0;
    p.off_err = o;  // the control block: error word, grid-barrier counters
    o = align_up(o + kControlBytes);
    p.off_cnt = o; o = align_up(o + sizeof(int) * (size_t)p.nlists * p.C);
    p.off_lidx = o; o = align_up(o + sizeof(int) * (size_t)p.nlists * F);
    p.off_lh = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_aeff = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_uval = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_score = o; o = align_up(o + sizeof(float) * (size_t)B * F);
    p.off_mask = o; o = align_up(o + sizeof(uint32_t) * (size_t)B * ((F + 31) / 32));
    p.off_part = o; o = align_up(o + sizeof(float) * (size_t)(p.G2 > p.C ? p.G2 : p.C) * B * d);
    p.total = o;
    return p;
}

// Dynamic shared memory of the gate kernel with D rows in flight per warp.
static size_t gate_smem(size_t x_bytes, uint32_t stage_bytes, int D) {
    return gate_bar_bytes(D) + (size_t)kGateWarps * D * stage_bytes + x_bytes;
}

template <class W, int NB, bool UP>
static cudaError_t launch_gate(const GateArgs &ga_in, const DecodePlan &p, cudaStream_t s) {
    GateArgs ga = ga_in;
    const uint32_t row_bytes = (uint32_t)(p.d / W::E) * 16u;
    const uint32_t sbytes = W::Q ? (uint32_t)(p.d / 64) * 2u : 0u;
    const uint32_t stage_bytes = (UP ? 2u : 1u) * (row_bytes + sbytes);
    const size_t x_bytes = (size_t)NB * p.d * sizeof(typename W::X);
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, (const void *)k_gate<W, NB, UP>);
    if (e != cudaSuccess) return e;
    const long avail = (long)device_smem_optin() - (long)fa.sharedSizeBytes - 1024 - (long)x_bytes - 16;
    long D = avail / ((long)kGateWarps * (stage_bytes + sizeof(uint64_t)));
    if (D > 16) D = 16;  // small rows: a warp's whole share of the chunk can be in flight
    const int rows_per_warp = (p.R + kGateWarps - 1) / kGateWarps;
    if (D > rows_per_warp) D = rows_per_warp;
    if (D < 1) return cudaErrorInvalidConfiguration;
    ga.stages = (int)D;
    if (ga.gbar && ga.pf_rows > 0) {
        // CTAs that start before the previous call's reducers leave: the idle
        // SMs plus the previous call's non-reducing CTAs (the reducer count of
        // decode_finish.cuh for the same grid)
        const long C = p.C, total = (long)p.nb * p.d;
        const long NR = std::min(C, std::max((total + 31) / 32, (C + 3) / 4));
        const int E = device_sm_count() - (int)NR;
        ga.pf_early = E > 0 && E < p.C ? E : 0;
    }
    const size_t smem = gate_smem(x_bytes, stage_bytes, ga.stages);
    e = set_max_smem((const void *)k_gate<W, NB, UP>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_gate<W, NB, UP>, dim3(p.C), dim3(kGateThreads), smem, s, ga);
}

template <class W, int NB>
static cudaError_t launch_decode_t(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    char *ws = static_cast<char *>(c.ws);
    const sffn_ffn_weights *w = c.w;
    const bool scores_only = c.scores_only != nullptr;
    const bool keep = c.mode == SFFN_MODE_KEEP_RATIO;
    const bool up = c.score == SFFN_SCORE_GATE_UP && (c.mode != SFFN_MODE_EXACT || scores_only);
    int32_t *err = reinterpret_cast<int32_t *>(ws + p.off_err);
    int *cnt = reinterpret_cast<int *>(ws + p.off_cnt);
    int *lidx = reinterpret_cast<int *>(ws + p.off_lidx);
    float *lh = reinterpret_cast<float *>(ws + p.off_lh);
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
    ga.aeff = (keep && !scores_only) ? aeff : nullptr;
    ga.uval = (keep && up && !scores_only) ? uval : nullptr;
    ga.score = scores_only ? c.scores_only : (keep ? score : nullptr);
    ga.cnt = cnt;
    ga.lidx = lidx;
    ga.err = err;
    // exact / threshold with every gate CTA resident: the gate kernel finishes
    // the call itself (grid barrier + distributed reduction + index lists)
    const bool fused = !scores_only && !keep && p.C <= device_sm_count();
    ga.gbar = fused ? reinterpret_cast<unsigned *>(ws + p.off_err + kCtlBar) : nullptr;
    ga.pf_rows = fused ? kGatePfRows : 0;
    ga.out = c.out;
    ga.out_f32 = w->wdtype == SFFN_F32;
    ga.active_idx = c.active_idx;
    ga.n_active = c.n_active;
    ga.wdT = w->w_downT;
    ga.part = part;
    ga.sg = w->s_gate;
    ga.su = w->s_up;
    ga.sd = w->s_downT;
    cudaError_t e;
    if (W::Q && up && !ga.decide && scores_q1_eligible(w, p))  // int4, one token, gate-and-up scores
        e = run_scores_q1(w, c.x, p, ga.score, ga.aeff, ga.uval, s);
    else
        e = up ? launch_gate<W, NB, true>(ga, p, s) : launch_gate<W, NB, false>(ga, p, s);
    if (e != cudaSuccess || scores_only || fused) return e;

    int nparts = p.G2;
    bool list_ctas = p.nb > 1;
    bool fin_down = false;
    if (!keep) {  // exact / threshold: the gate kernel already wrote per-chunk partials
        nparts = p.C;
        list_ctas = true;
    }
    {
        bool have_h = up;  // keep-ratio: h_j known before the down pass
        if (keep) {
            KeepArgs ka = {};
            ka.score = score;
            ka.aeff = aeff;
            ka.uval = up ? uval : nullptr;
            ka.lh = up ? lh : nullptr;
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
            ka.core = c.core;
            ka.n_core = c.n_core;
            ka.err = err;
            const size_t ksm = p.F <= kKeepStage ? sizeof(uint32_t) * (size_t)p.F : 0;
            if (ksm && (e = set_max_smem((const void *)k_keep_ratio, (int)(sizeof(uint32_t) * kKeepStage))) !=
                           cudaSuccess)
                return e;
            e = launch_k(k_keep_ratio, dim3(p.nb), dim3(kSelThreads), ksm, s, ka);
            if (e != cudaSuccess) return e;
            if (p.nb > 1) {
                e = launch_k(k_union, dim3(1), dim3(kSelThreads), 0, s, (const uint32_t *)mask, p.nb, p.F, p.C, cnt, lidx,
                             (const float *)aeff, (const float *)uval, up ? lh : (float *)nullptr);
                if (e != cudaSuccess) return e;
            }
        }

        const int threads = ((p.d / 8) + 31) / 32 * 32;
        const int max_rows = (p.F + p.G2 - 1) / p.G2 + 1;
        // keep-ratio with one token: the token's list is written by the select and
        // the down kernel, so the down kernel can finish the call itself (its CTAs
        // are all resident and at least 256 threads wide)
        fin_down = keep && p.nb == 1 && threads >= 256 && nparts <= device_sm_count();
        unsigned *gbar = fin_down ? reinterpret_cast<unsigned *>(ws + p.off_err + kCtlBar) : nullptr;
        if (!keep) {
            // nothing between the gate kernel and the reduction
        } else if (have_h) {
            DownArgs da = {};
            da.wdT = w->w_downT;
            da.sdT = w->s_downT;
            da.d = p.d;
            da.F = p.F;
            da.nb = p.nb;
            da.R = p.R;
            da.C = p.C;
            da.list_u = p.list_u;
            da.cnt = cnt;
            da.lidx = lidx;
            da.lh = lh;
            da.part = part;
            da.active_idx = p.nb == 1 ? c.active_idx : nullptr;
            da.n_active = p.nb == 1 ? c.n_active : nullptr;
            da.by_chunk = 0;  // keep-ratio lists are one block, not per gate chunk
            da.max_rows = max_rows;
            da.gbar = gbar;
            da.out = c.out;
            da.out_f32 = w->wdtype == SFFN_F32;
            da.err = err;
            const size_t smem = sizeof(int) * (kMaxC + 1 + da.max_rows) + sizeof(float) * (size_t)da.max_rows * NB;
            e = set_max_smem((const void *)k_down<W, NB>, (int)smem);
            if (e == cudaSuccess) e = launch_k(k_down<W, NB>, dim3(nparts), dim3(threads), smem, s, da);
        } else {
            UpDownArgs ua = {};
            ua.wu = w->w_up;
            ua.wdT = w->w_downT;
            ua.su = w->s_up;
            ua.sdT = w->s_downT;
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
            ua.uval = nullptr;
            ua.part = part;
            ua.active_idx = p.nb == 1 ? c.active_idx : nullptr;
            ua.n_active = p.nb == 1 ? c.n_active : nullptr;
            ua.gbar = gbar;
            ua.out = c.out;
            ua.out_f32 = w->wdtype == SFFN_F32;
            ua.err = err;
            const size_t smem = sizeof(float) * NB * p.d + sizeof(int) * (kMaxC + 1 + max_rows);
            e = set_max_smem((const void *)k_updown<W, NB, false>, (int)smem);
            if (e == cudaSuccess) e = launch_k(k_updown<W, NB, false>, dim3(p.G2), dim3(threads), smem, s, ua);
        }
        if (e != cudaSuccess) return e;
    }
    if (fin_down) return cudaSuccess;

    ReduceArgs ra = {};
    ra.part = part;
    ra.G2 = nparts;
    ra.nb = p.nb;
    ra.d = p.d;
    ra.out = c.out;
    ra.out_f32 = w->wdtype == SFFN_F32;
    ra.n_red = (int)(((size_t)p.nb * p.d + 31) / 32);
    ra.C = p.C;
    ra.R = p.R;
    ra.F = p.F;
    ra.cnt = cnt;
    ra.lidx = lidx;
    ra.active_idx = c.active_idx;
    ra.n_active = c.n_active;
    // keep-ratio lists live in chunk 0 of each token (chunk stride irrelevant there)
    const int list_grid = list_ctas ? p.nb * ((p.C + kListChunks - 1) / kListChunks) : 0;
    return launch_k(k_reduce, dim3(ra.n_red + list_grid), dim3(256), 0, s, ra);
}

template <class W>
static cudaError_t launch_decode_w(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    if (p.nb == 1) return launch_decode_t<W, 1>(c, p, s);
    if (p.nb == 2) return launch_decode_t<W, 2>(c, p, s);
    if (p.nb <= 4) return launch_decode_t<W, 4>(c, p, s);
    return launch_decode_t<W, 8>(c, p, s);
}

// The finish of a one-token decode whose C gate chunks have each written a
// partial output part[c, d] and an ascending list of its active neurons
// (cnt [C], lidx [C, R]): the fixed-order sum of the partials into `out`, and
// the token's list and count.
sffn_status run_reduce_chunks(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    char *ws = static_cast<char *>(c.ws);
    ReduceArgs ra = {};
    ra.part = reinterpret_cast<float *>(ws + p.off_part);
    ra.G2 = p.C;
    ra.nb = 1;
    ra.d = p.d;
    ra.out = c.out;
    ra.out_f32 = c.w->wdtype == SFFN_F32;
    ra.n_red = (p.d + 31) / 32;
    ra.C = p.C;
    ra.R = p.R;
    ra.F = p.F;
    ra.cnt = reinterpret_cast<int *>(ws + p.off_cnt);
    ra.lidx = reinterpret_cast<int *>(ws + p.off_lidx);
    ra.active_idx = c.active_idx;
    ra.n_active = c.n_active;
    const int list_grid = (p.C + kListChunks - 1) / kListChunks;
    const cudaError_t e = launch_k(k_reduce, dim3(ra.n_red + list_grid), dim3(256), 0, s, ra);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

sffn_status run_decode(const DecodeCall &c, const DecodePlan &p, cudaStream_t s) {
    if (decode_q1_eligible(c, p, false)) return run_decode_q1(c, p, s, false);
    if (decode_tc_eligible(c, p)) return run_decode_tc(c, p, s, false);
    cudaError_t e;
    switch (c.w->wdtype) {
    case SFFN_F32: e = launch_decode_w<WF32>(c, p, s); break;
    case SFFN_BF16: e = launch_decode_w<WBF16>(c, p, s); break;
    case SFFN_INT4_G64: e = launch_decode_w<WINT4>(c, p, s); break;
    default: return SFFN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

sffn_status run_down_norms(const sffn_ffn_weights *w, float *norms, cudaStream_t s) {
    cudaError_t e;
    const dim3 grid((w->d_ff + 7) / 8), block(256);
    switch (w->wdtype) {
    case SFFN_F32:
        e = launch_k(k_down_norms<WF32>, grid, block, 0, s, w->w_downT, (const void *)nullptr, w->d_model, w->d_ff, norms);
        break;
    case SFFN_BF16:
        e = launch_k(k_down_norms<WBF16>, grid, block, 0, s, w->w_downT, (const void *)nullptr, w->d_model, w->d_ff, norms);
        break;
    case SFFN_INT4_G64:
        e = launch_k(k_down_norms<WINT4>, grid, block, 0, s, w->w_downT, w->s_downT, w->d_model, w->d_ff, norms);
        break;
    default: return SFFN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
