// decode_tc.cu -- decode with the dot products on the tensor cores
// (mma.sync, bf16 operands, fp32 accumulation), for int4-g64 weights at any
// token count, bf16 weights with 2..8 tokens, and the dense layer (every neuron,
// nothing skipped) that the sparse calls are measured against.
//
// Same computation as the gate kernel in decode.cu (denseflux, "skipping most
// of a dense FFN", sec. 5.1-5.3: the gate is read in full, then only the active
// rows of W_up and of W_downT; WiSparse write-up sec. 1.2 / 2.3: the threshold
// on |a_j| * ||W_down[:, j]||_2), organised for a tensor-core contraction.
//
// One CTA per SM owns a chunk of R <= 128 neurons.  "Stages" of up to 8 rows of
// one matrix move into a ring of shared-memory slots by bulk copies (a chunk's
// consecutive gate rows in one copy; the gathered rows of the active neurons
// with consecutive rows merged), each stage completing on its own mbarrier.
// All 8 warps consume every stage; the last warp to release a slot (a
// shared-memory count) issues the stage that goes into it next, so no warp
// waits to refill the ring.  The weights are constant inputs: the first stages
// are in flight before the kernel waits for the previous one in the stream.
//
//   gate   Per stage, m16n8k16 MMAs with the tokens as M (8 real, 8 zero),
//          the stage's 8 rows as N and the columns as K; the 8 consumer warps
//          split the columns, each with its eighth of the activations held in
//          registers.  A dot product is a sum over k, so the MMA's k order is
//          free: a lane reads 16 B of bf16 (8 columns) or 4 B of int4 codes (8
//          columns) of its row, and the activations are laid out once in the
//          same order.  int4 codes become exact bf16 integers (OR the nibble
//          into the mantissa of 128, subtract 136); the fp16 group scale
//          multiplies each 64-column group's exact partial.
//   decide The warps' partials are summed in a fixed order; bias, act, score
//          and the decision per (neuron, token); the chunk's ascending
//          per-token lists and the union of its active rows.
//   up     The same contraction over the union rows of W_up: u_j, then
//          h_j = a_j u_j per token (0 where the token did not select j).
//   down   out_partial[col][token] += W_downT[j][col] * h_j[token] as m16n8k8
//          MMAs with the columns as M (split across the warps), the stage's
//          rows as K and the tokens as N; h is split into a bf16 high part and
//          the bf16 rounding of its remainder (two MMAs: ~16 significant bits).
//          For int4 the row's group scale is folded into h.
//   finish The per-CTA fp32 partials are summed in a fixed order behind a
//          bounded grid barrier (decode_finish.cuh).  Deterministic.
#include "common.cuh"
#include "decode_finish.cuh"
#include "internal.h"

#include <algorithm>

namespace sffn {

namespace {

constexpr int kTcCons = 8;                   // warps: all consume every stage
constexpr int kTcThreads = 32 * kTcCons;
constexpr int kTcPfRows = 48;               // rows of each later chunk sent to L2 by the early CTAs
constexpr int kTcMaxRows = 128;              // rows per chunk
constexpr int kTcStageRows = 8;              // rows per stage: the MMA's N
constexpr int kTcMaxSlots = 16;
constexpr int kTcN = 8;                      // tokens

struct TcArgs {
    const char *wg, *wu, *wd;  // [F, row_bytes] stored rows (int4: packed codes)
    const char *sg, *su, *sd;  // int4: fp16 group scales [F, d/64]
    const float *bias, *norms;
    const uint16_t *x;         // bf16 [nb, d]
    int d, F, nb, R, C;
    int act, mode;
    float tau;
    int slots;                 // ring slots
    int *cnt, *lidx;           // sparse: chunk counts and chunk-local lists
    int32_t *err;
    float *part;               // [C, nb, d]
    unsigned *gbar;
    void *out;
    int32_t *active_idx, *n_active;
    int nr_cap;                // reducers of the finish (fewest with the same load rounds)
    int pf_early, pf_rows;     // the first pf_early CTAs send rows 0 .. pf_rows-1 of the later chunks to L2
};

// D += A * B, m16n8k16 / m16n8k8, bf16 inputs, fp32 accumulators.
SFFN_DEV void mma16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
SFFN_DEV void mma8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// Two int4 codes -> a bf16 pair, exactly.  w holds, after XOR 0x8 per nibble
// (the code + 8 as an unsigned nibble), one code in bits 0..3 and one in bits
// 16..19; OR-ing them into the mantissa of bf16 128.0 gives 128 + code + 8,
// and one fma (times 1, minus 136) leaves the code.
SFFN_DEV uint32_t codes2_bf16(uint32_t w) {
    const uint32_t v = (w & 0x000F000Fu) | 0x43004300u;
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0x3F803F80u), "r"(0xC308C308u));
    return r;
}

SFFN_DEV float half_bits_to_f32(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)h)); }
SFFN_DEV float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// (hi, lo) bf16 pairs of two fp32 values: hi = bf16(v), lo = bf16(v - hi).
SFFN_DEV void split_pair(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    const uint32_t h0 = f32_to_bf16_bits(v0), h1 = f32_to_bf16_bits(v1);
    hi = h0 | (h1 << 16);
    lo = (uint32_t)f32_to_bf16_bits(v0 - bf16_bits_to_f32(h0)) | ((uint32_t)f32_to_bf16_bits(v1 - bf16_bits_to_f32(h1)) << 16);
}

}  // namespace

// Shared memory of the kernel with the given number of ring slots.
// A stage: 8 rows of weights, each padded by 16 bytes (so that the rows a warp
// reads together fall in different shared-memory banks), then their scales.
constexpr uint32_t kTcRowPad = 16;
SFFN_HOST_DEV size_t tc_stage_bytes(int d, bool q) {
    return (size_t)kTcStageRows * ((q ? (size_t)d / 2 : (size_t)d * 2) + kTcRowPad + (q ? (size_t)d / 32 : 0));
}
SFFN_HOST_DEV size_t tc_smem_bytes(int d, bool q, int slots) {
    return (size_t)128                                   // slots mbarriers (<= 16)
           + (size_t)slots * tc_stage_bytes(d, q)        // ring
           + (size_t)kTcCons * kTcMaxRows * kTcN * 4     // warp partials
           + (size_t)2 * kTcMaxRows * kTcN * 4           // a, h
           + (size_t)kTcMaxRows * 4;                     // union rows
}

namespace {

// NU = d / 256: 32-column units per consumer warp.
template <bool Q, int NU, bool DENSE>
__global__ void __launch_bounds__(kTcThreads, 1) k_gate_tc(TcArgs a) {
    constexpr int d = NU * 256;
    constexpr uint32_t row_bytes = Q ? d / 2 : d * 2;
    constexpr uint32_t sbytes = Q ? d / 32 : 0;          // int4 group scales of one row
    constexpr uint32_t rstride = row_bytes + kTcRowPad;  // a row's place in a stage
    constexpr uint32_t scl_off = kTcStageRows * rstride;
    constexpr uint32_t stage_bytes = kTcStageRows * (rstride + sbytes);
    extern __shared__ __align__(128) unsigned char smraw[];
    const int F = a.F, nb = a.nb, NS = a.slots;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw);
    unsigned char *ring = smraw + 128;
    float *gp = reinterpret_cast<float *>(ring + (size_t)NS * stage_bytes);  // [warp][row][token]
    float *sa = gp + kTcCons * kTcMaxRows * kTcN;                          // a per (row, token), 0 if inactive
    float *hs = sa + kTcMaxRows * kTcN;                                    // h per (union position, token)
    int *urow = reinterpret_cast<int *>(hs + kTcMaxRows * kTcN);          // union rows, ascending
    __shared__ uint32_t sflag[kTcMaxRows];
    __shared__ float sbias[kTcMaxRows], snorm[kTcMaxRows];
    __shared__ int wcnt[kTcN + 1][4];
    __shared__ int slot_rel[kTcMaxSlots];   // warps done with the slot's current stage
    __shared__ int slot_iss[kTcMaxSlots];   // stages issued into the slot
    __shared__ int s_nu, s_known;
    __shared__ volatile int s_abort;

    const int row0 = blockIdx.x * a.R;
    const int nrows = min(a.R, F - row0);
    const char *gbase = a.wg + (size_t)row0 * row_bytes, *ubase = a.wu + (size_t)row0 * row_bytes;
    const char *dbase = a.wd + (size_t)row0 * row_bytes;
    const char *gsb = Q ? a.sg + (size_t)row0 * sbytes : nullptr, *usb = Q ? a.su + (size_t)row0 * sbytes : nullptr;
    const char *dsb = Q ? a.sd + (size_t)row0 * sbytes : nullptr;
    const int ngs = (nrows + kTcStageRows - 1) / kTcStageRows;  // gate stages

    if (tid < kTcMaxRows) sflag[tid] = 0u;
    // the gate bias of the chunk's rows: an input, like the weights
    if (tid < nrows) sbias[tid] = a.bias ? __ldg(a.bias + row0 + tid) : 0.f;
    if (tid < kTcMaxSlots) slot_rel[tid] = slot_iss[tid] = 0;
    if (tid == 0) {
        s_abort = 0;
        // stages known before the decision: the gate's (the dense layer: all)
        s_known = DENSE ? 3 * ngs : ngs;
        for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
        mbar_fence_init();
    }
    __syncthreads();

    // Stage j: gate stages 0 .. ngs-1 (chunk rows 8j ..), then the up and then
    // the down stages over the union positions (the dense layer: every row),
    // in slot j % NS once the slot's previous stage is released by every warp.
    // A whole warp issues a stage: lane 0 arms the barrier, lane i < cnt copies
    // row i to its padded place, lanes 8 .. 15 copy the scales of each run of
    // consecutive rows.  (A bulk copy holds its issuing thread for a while;
    // spread over lanes the copies of a stage go out together.)
    const uint64_t pol = l2_evict_first_policy();
    auto issue_stage = [&](int j) {
        const char *m, *sm;
        int p0, cnt;
        bool gathered = false;
        if (j < ngs) {
            m = gbase; sm = gsb; p0 = j * kTcStageRows; cnt = min(kTcStageRows, nrows - p0);
        } else {
            const int nu = DENSE ? nrows : s_nu;
            const int nus = (nu + kTcStageRows - 1) / kTcStageRows;
            const int jj = j - ngs;
            const bool up = jj < nus;
            m = up ? ubase : dbase;
            sm = up ? usb : dsb;
            p0 = (up ? jj : jj - nus) * kTcStageRows;
            cnt = min(kTcStageRows, nu - p0);
            gathered = !DENSE;
        }
        const int slot = j % NS;
        unsigned char *st = ring + (size_t)slot * stage_bytes;
        uint64_t *bar = &full[slot];
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, (uint32_t)cnt * (row_bytes + sbytes));
            slot_iss[slot] += 1;
        }
        __syncwarp();
        auto rowof = [&](int i) { return gathered ? urow[p0 + i] : p0 + i; };
        if (lane < cnt) {
            fence_proxy_async_smem();
            bulk_load(st + (size_t)lane * rstride, m + (size_t)rowof(lane) * row_bytes, row_bytes, bar, pol);
        }
        if (Q && lane >= 8 && lane < 8 + cnt) {
            const int i = lane - 8, r = rowof(i);
            if (i == 0 || rowof(i - 1) != r - 1) {
                int n = 1;
                while (i + n < cnt && rowof(i + n) == r + n) ++n;
                fence_proxy_async_smem();
                bulk_load(st + scl_off + (size_t)i * sbytes, sm + (size_t)r * sbytes, (uint32_t)n * sbytes, bar, pol);
            }
        }
    };
    // The weights are constant inputs: the first stages move before the wait
    for (int j = warp; j < NS && j < s_known; j += kTcCons) issue_stage(j);
    // The first CTAs of a call find free SMs while the previous call's reducers
    // still hold the others; they send the first gate rows of the later chunks
    // (chunk c >= E to CTA c mod E, row order across chunks) to L2, so that HBM
    // streams through the previous call's finish.
    if (a.pf_early > 0 && (int)blockIdx.x < a.pf_early && warp == kTcCons - 1) {
        const int E = a.pf_early;
        const int nch = (a.C - 1 - (int)blockIdx.x) / E;
        const int P = min(a.pf_rows, a.R);
        for (int i = lane; i < nch * P; i += 32) {
            const int r = i / nch, c = (int)blockIdx.x + (1 + i % nch) * E;
            const int jr = c * a.R + r;
            if (r < a.R && jr < F) {
                bulk_prefetch_l2(a.wg + (size_t)jr * row_bytes, row_bytes);
                if (Q) bulk_prefetch_l2(a.sg + (size_t)jr * sbytes, sbytes);
            }
        }
    }
    // x may be the previous layer's output: read it only after the dependency wait
    griddep_wait();
    griddep_launch_dependents();
    const unsigned bar_base = *reinterpret_cast<volatile unsigned *>(a.gbar + 1);
    // the rows' ||W_down[:, j]|| (threshold rule; they may come from the previous
    // kernel), in shared memory long before the decision reads them
    if (tid < nrows) snorm[tid] = !DENSE && a.mode != SFFN_MODE_EXACT && a.norms ? a.norms[row0 + tid] : 0.f;

    int ck = 0;  // stages consumed by this warp
    auto consume_wait = [&](int k) -> bool {
        const bool ok = mbar_wait(&full[k % NS], (uint32_t)(k / NS) & 1u);
        if (!ok && lane == 0) {
            s_abort = 1;
            record_error(a.err, SFFN_ERR_TIMEOUT);
        }
        return __all_sync(0xffffffffu, ok) && !s_abort;
    };
    // This warp is done with stage k; the last warp to be done refills the slot
    // with stage k + NS when that stage is known.
    auto release = [&](int k) {
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            const int slot = k % NS;
            last = atomicAdd(&slot_rel[slot], 1) == kTcCons - 1;
            if (last) {
                slot_rel[slot] = 0;
                __threadfence_block();
            }
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last && k + NS < s_known && !s_abort) issue_stage(k + NS);
    };

    // activation fragments of this warp's columns: unit u covers columns
    // kw0 + 32 u .. + 32; lane (g, t) holds token g's 8 columns at + 8 t, in the
    // order its weight fragments use (bf16: as stored; int4: (k, k + 4) pairs)
    uint32_t xr[NU][4];
    const int kw0 = warp * (d / kTcCons);
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (g < nb) v = ldg_v4(a.x + (size_t)g * d + kw0 + u * 32 + 8 * t);
        if constexpr (Q) {
            xr[u][0] = __byte_perm(v.x, v.z, 0x5410);
            xr[u][1] = __byte_perm(v.x, v.z, 0x7632);
            xr[u][2] = __byte_perm(v.y, v.w, 0x5410);
            xr[u][3] = __byte_perm(v.y, v.w, 0x7632);
        } else {
            xr[u][0] = v.x; xr[u][1] = v.y; xr[u][2] = v.z; xr[u][3] = v.w;
        }
    }

    // One gate / up stage: this warp's partial dot products of the stage's rows
    // with the tokens over its columns, to gp[warp][p0 + row][token].
    auto dot_stage = [&](const unsigned char *st, int cnt, int p0) {
        float c[4] = {0.f, 0.f, 0.f, 0.f};
        const unsigned char *rowp = st + (size_t)g * rstride;  // lane group g reads stage row g
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int kb = kw0 + u * 32;
            if constexpr (Q) {
                float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t cw = *reinterpret_cast<const uint32_t *>(rowp + kb / 2 + 4 * t) ^ 0x88888888u;
                mma16(tmp, xr[u][0], 0u, xr[u][1], 0u, codes2_bf16(cw), codes2_bf16(cw >> 4));
                mma16(tmp, xr[u][2], 0u, xr[u][3], 0u, codes2_bf16(cw >> 8), codes2_bf16(cw >> 12));
                // the unit's 64-column group scale per row (N = 2t, 2t + 1)
                const int grp = kb / 64;
                const uint16_t *sr = reinterpret_cast<const uint16_t *>(st + scl_off);
                const float s0 = half_bits_to_f32(sr[(2 * t) * (sbytes / 2) + grp]);
                const float s1 = half_bits_to_f32(sr[(2 * t + 1) * (sbytes / 2) + grp]);
                c[0] = fmaf(s0, tmp[0], c[0]);
                c[1] = fmaf(s1, tmp[1], c[1]);
            } else {
                const uint4 wv = *reinterpret_cast<const uint4 *>(rowp + (size_t)(kb + 8 * t) * 2);
                mma16(c, xr[u][0], 0u, xr[u][1], 0u, wv.x, wv.y);
                mma16(c, xr[u][2], 0u, xr[u][3], 0u, wv.z, wv.w);
            }
        }
        // c0 = (token g, row 2t), c1 = (token g, row 2t + 1)
        if (g < nb) {
            float *o = gp + ((size_t)warp * kTcMaxRows + p0) * kTcN + g;
            if (2 * t < cnt) o[(2 * t) * kTcN] = c[0];
            if (2 * t + 1 < cnt) o[(2 * t + 1) * kTcN] = c[1];
        }
    };

    // ---- gate pass ----
    for (int i = 0; i < ngs; ++i, ++ck) {
        if (!consume_wait(ck)) break;
        dot_stage(ring + (size_t)(ck % NS) * stage_bytes, min(kTcStageRows, nrows - i * kTcStageRows), i * kTcStageRows);
        release(ck);
    }
    __syncthreads();

    // ---- bias, act, score, decision per (neuron, token) ----
    if (!s_abort) {
        for (int i = tid; i < nrows * nb; i += blockDim.x) {
            const int r = i / nb, b = i - r * nb;
            float gv = 0.f;
#pragma unroll
            for (int w = 0; w < kTcCons; ++w) gv += gp[((size_t)w * kTcMaxRows + r) * kTcN + b];
            gv += sbias[r];
            const float av = act_fn(a.act, gv);
            if (DENSE) {
                sa[r * kTcN + b] = av;
            } else {
                const bool active = a.mode == SFFN_MODE_EXACT ? av != 0.f : fabsf(av) * snorm[r] >= a.tau;
                sa[r * kTcN + b] = active ? av : 0.f;
                if (active) atomicOr(&sflag[r], 1u << b);
            }
        }
    }
    int nu = nrows;
    if constexpr (!DENSE) {
        __syncthreads();
        // ---- ordered compaction: per-token lists (for active_idx) and the
        // union of the chunk's active rows (row r = tid < nrows <= 128: warps 0..3)
        const uint32_t f = tid < nrows ? sflag[tid] : 0u;
        if (warp < 4) {
            for (int l = 0; l <= nb; ++l) {
                const bool bit = l < nb ? ((f >> l) & 1u) : f != 0u;
                const unsigned bl = __ballot_sync(0xffffffffu, bit);
                if (lane == 0) wcnt[l][warp] = __popc(bl);
            }
        }
        __syncthreads();
        if (warp < 4) {
            const unsigned lt = (1u << lane) - 1u;
            for (int l = 0; l <= nb; ++l) {
                const bool bit = l < nb ? ((f >> l) & 1u) : f != 0u;
                const unsigned bl = __ballot_sync(0xffffffffu, bit);
                int base = 0, tot = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    base += w < warp ? wcnt[l][w] : 0;
                    tot += wcnt[l][w];
                }
                const int pos = base + __popc(bl & lt);
                if (bit) {
                    if (l < nb) a.lidx[(size_t)l * F + row0 + pos] = row0 + tid;
                    else urow[pos] = tid;
                }
                if (tid == 0) {
                    if (l < nb) a.cnt[(size_t)l * a.C + blockIdx.x] = tot;
                    else s_nu = tot;
                }
            }
        }
        __syncthreads();
        nu = s_nu;
        // Every gate stage is released and none of the stages after them was
        // issued (they were unknown): the up and down stages whose slots are free
        // now (stages ngs .. ngs + NS - 1) are issued here, the rest by the warps
        // that free their slots.
        if (tid == 0) s_known = ngs + 2 * ((nu + kTcStageRows - 1) / kTcStageRows);
        __syncthreads();
        if (!s_abort)
            for (int j = ngs + warp; j < ngs + NS && j < s_known; j += kTcCons) issue_stage(j);
    } else {
        if (tid < nrows) urow[tid] = tid;
    }
    const int nus = (nu + kTcStageRows - 1) / kTcStageRows;

    // ---- up pass over the union rows; h = a u per token ----
    for (int i = 0; i < nus && !s_abort; ++i, ++ck) {
        if (!consume_wait(ck)) break;
        dot_stage(ring + (size_t)(ck % NS) * stage_bytes, min(kTcStageRows, nu - i * kTcStageRows), i * kTcStageRows);
        release(ck);
    }
    __syncthreads();
    for (int i = tid; i < nu * nb; i += blockDim.x) {
        const int p = i / nb, b = i - p * nb;
        float u = 0.f;
#pragma unroll
        for (int w = 0; w < kTcCons; ++w) u += gp[((size_t)w * kTcMaxRows + p) * kTcN + b];
        hs[p * kTcN + b] = sa[urow[p] * kTcN + b] * u;
    }
    __syncthreads();

    // ---- down projection: this warp's columns [kw0, kw0 + d/8) in blocks of 64,
    // four m16 tiles per block (lane g holds columns 8g .. 8g + 7 of a block:
    // tile p takes 8g + 2p as M row g and 8g + 2p + 1 as M row g + 8) ----
    constexpr int NBLK = NU / 2;
    {
        float acc[NBLK][4][4];
#pragma unroll
        for (int k = 0; k < NBLK; ++k)
#pragma unroll
            for (int p = 0; p < 4; ++p) acc[k][p][0] = acc[k][p][1] = acc[k][p][2] = acc[k][p][3] = 0.f;
        for (int i = 0; i < nus && !s_abort; ++i, ++ck) {
            if (!consume_wait(ck)) break;
            const unsigned char *st = ring + (size_t)(ck % NS) * stage_bytes;
            const int cnt = min(kTcStageRows, nu - i * kTcStageRows);
            const int p0 = i * kTcStageRows;
            const bool v0 = 2 * t < cnt, v1 = 2 * t + 1 < cnt;  // K rows of this lane present
            const float h0 = (v0 && g < nb) ? hs[(p0 + 2 * t) * kTcN + g] : 0.f;
            const float h1 = (v1 && g < nb) ? hs[(p0 + 2 * t + 1) * kTcN + g] : 0.f;
            const unsigned char *r0p = st + (size_t)(2 * t) * rstride, *r1p = st + (size_t)(2 * t + 1) * rstride;
            uint32_t bh = 0, bl = 0;
            if constexpr (!Q) split_pair(h0, h1, bh, bl);
#pragma unroll
            for (int k = 0; k < NBLK; ++k) {
                const int cb = kw0 + k * 64;
                if constexpr (Q) {
                    const uint16_t *sr = reinterpret_cast<const uint16_t *>(st + scl_off);
                    const int grp = cb / 64;
                    const float s0 = v0 ? half_bits_to_f32(sr[(2 * t) * (sbytes / 2) + grp]) : 0.f;
                    const float s1 = v1 ? half_bits_to_f32(sr[(2 * t + 1) * (sbytes / 2) + grp]) : 0.f;
                    split_pair(h0 * s0, h1 * s1, bh, bl);
                    const uint32_t w0 = v0 ? *reinterpret_cast<const uint32_t *>(r0p + (cb + 8 * g) / 2) ^ 0x88888888u : 0x88888888u;
                    const uint32_t w1 = v1 ? *reinterpret_cast<const uint32_t *>(r1p + (cb + 8 * g) / 2) ^ 0x88888888u : 0x88888888u;
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const int sh = 8 * p;
                        const uint32_t a0 = codes2_bf16(((w0 >> sh) & 0xFu) | (((w1 >> sh) & 0xFu) << 16));
                        const uint32_t a1 = codes2_bf16(((w0 >> (sh + 4)) & 0xFu) | (((w1 >> (sh + 4)) & 0xFu) << 16));
                        mma8(acc[k][p], a0, a1, bh);
                        mma8(acc[k][p], a0, a1, bl);
                    }
                } else {
                    const uint4 z = make_uint4(0, 0, 0, 0);
                    const uint4 q0 = v0 ? *reinterpret_cast<const uint4 *>(r0p + (size_t)(cb + 8 * g) * 2) : z;
                    const uint4 q1 = v1 ? *reinterpret_cast<const uint4 *>(r1p + (size_t)(cb + 8 * g) * 2) : z;
                    const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w}, w1[4] = {q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const uint32_t a0 = __byte_perm(w0[p], w1[p], 0x5410);
                        const uint32_t a1 = __byte_perm(w0[p], w1[p], 0x7632);
                        mma8(acc[k][p], a0, a1, bh);
                        mma8(acc[k][p], a0, a1, bl);
                    }
                }
            }
            release(ck);
        }
        // c0 = (column 8g + 2p, token 2t), c1 = (same column, token 2t + 1),
        // c2, c3 = (column 8g + 2p + 1, tokens 2t, 2t + 1)
        float *pc = a.part + (size_t)blockIdx.x * nb * d;
#pragma unroll
        for (int k = 0; k < NBLK; ++k)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int col = kw0 + k * 64 + 8 * g + 2 * p;
                if (2 * t < nb) *reinterpret_cast<float2 *>(pc + (size_t)(2 * t) * d + col) = make_float2(acc[k][p][0], acc[k][p][2]);
                if (2 * t + 1 < nb)
                    *reinterpret_cast<float2 *>(pc + (size_t)(2 * t + 1) * d + col) = make_float2(acc[k][p][1], acc[k][p][3]);
            }
    }
    __syncthreads();
    // after a timeout: the last stage issued into every slot lands (bounded)
    // before the CTA ends
    if (s_abort && tid < NS && slot_iss[tid] > 0) mbar_wait(&full[tid], (uint32_t)(slot_iss[tid] - 1) & 1u);
    FinishArgs fa;
    fa.gbar = a.gbar;
    fa.part = a.part;
    fa.nb = nb;
    fa.d = d;
    fa.F = F;
    fa.C = a.C;
    fa.R = a.R;
    fa.cnt = DENSE ? nullptr : a.cnt;
    fa.lidx = a.lidx;
    fa.out = a.out;
    fa.out_f32 = 0;
    fa.active_idx = a.active_idx;
    fa.n_active = a.n_active;
    fa.err = a.err;
    fa.nr_cap = a.nr_cap;
    finish_call(fa, bar_base, s_abort != 0);
}

template <bool Q, int NU, bool DENSE>
cudaError_t launch_tc(TcArgs ta, const DecodePlan &p, cudaStream_t s) {
    constexpr int d = NU * 256;
    const size_t fixed = tc_smem_bytes(d, Q, 0);
    long slots = ((long)device_smem_optin() - 4096 - (long)fixed) / (long)tc_stage_bytes(d, Q);
    const int need = 3 * ((p.R + kTcStageRows - 1) / kTcStageRows);  // gate, up and down stages of a chunk
    if (slots > kTcMaxSlots) slots = kTcMaxSlots;
    if (slots > need) slots = need;
    if (slots < 2) return cudaErrorInvalidConfiguration;
    ta.slots = (int)slots;
    {
        // When the finish takes at most two rounds of 32-column blocks (two
        // blocks per round), only the fewest reducers that keep that many
        // rounds wait at the barrier; the other CTAs leave, and as many CTAs
        // of the next call start early (with the idle SMs) and prefetch.  With
        // more rounds every CTA reduces (measured: capping them at B = 8 made
        // the call slower).
        const long C = p.C, nblk = ((long)p.nb * p.d + 31) / 32, minr = (C + 3) / 4;
        const long nr0 = std::min(C, std::max(nblk, minr));
        const long rounds = (nblk + 2 * nr0 - 1) / (2 * nr0);
        const bool cap = rounds <= 2;
        const long nr = cap ? std::min(nr0, std::max((nblk + 2 * rounds - 1) / (2 * rounds), minr)) : nr0;
        ta.nr_cap = (int)nr;
        const long E = (long)device_sm_count() - nr;
        ta.pf_early = cap && E > 0 && E < C ? (int)E : 0;
        ta.pf_rows = kTcPfRows;
    }
    const size_t smem = tc_smem_bytes(d, Q, (int)slots);
    cudaError_t e = set_max_smem((const void *)k_gate_tc<Q, NU, DENSE>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_gate_tc<Q, NU, DENSE>, dim3(p.C), dim3(kTcThreads), smem, s, ta);
}

template <bool Q, bool DENSE>
cudaError_t launch_tc_d(const TcArgs &ta, const DecodePlan &p, cudaStream_t s) {
    switch (p.d) {
    case 1024: return launch_tc<Q, 4, DENSE>(ta, p, s);
    case 2048: return launch_tc<Q, 8, DENSE>(ta, p, s);
    case 4096: return launch_tc<Q, 16, DENSE>(ta, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_tc_shape_ok(const sffn_ffn_weights *w, const DecodePlan &p) {
    const int d = w->d_model;
    if (d != 1024 && d != 2048 && d != 4096) return false;
    if (p.R > kTcMaxRows || p.C > device_sm_count()) return false;
    const bool q = w->wdtype == SFFN_INT4_G64;
    return tc_smem_bytes(d, q, 2) + 4096 <= (size_t)device_smem_optin();
}

bool decode_tc_eligible(const DecodeCall &c, const DecodePlan &p) {
    const sffn_ffn_weights *w = c.w;
    if (c.scores_only) return false;
    if (w->wdtype == SFFN_BF16) {
        if (c.B < 2) return false;
    } else if (w->wdtype != SFFN_INT4_G64) {
        return false;
    }
    if (c.mode == SFFN_MODE_KEEP_RATIO) return false;
    if (c.mode == SFFN_MODE_THRESHOLD && c.score != SFFN_SCORE_GATE) return false;
    return decode_tc_shape_ok(w, p);
}

sffn_status run_decode_tc(const DecodeCall &c, const DecodePlan &p, cudaStream_t s, bool dense) {
    char *ws = static_cast<char *>(c.ws);
    const sffn_ffn_weights *w = c.w;
    TcArgs ta = {};
    ta.wg = static_cast<const char *>(w->w_gate);
    ta.wu = static_cast<const char *>(w->w_up);
    ta.wd = static_cast<const char *>(w->w_downT);
    ta.sg = static_cast<const char *>(w->s_gate);
    ta.su = static_cast<const char *>(w->s_up);
    ta.sd = static_cast<const char *>(w->s_downT);
    ta.bias = w->b_gate;
    ta.norms = w->down_norms;
    ta.x = static_cast<const uint16_t *>(c.x);
    ta.d = p.d;
    ta.F = p.F;
    ta.nb = p.nb;
    ta.R = p.R;
    ta.C = p.C;
    ta.act = w->act;
    ta.mode = c.mode;
    ta.tau = c.param;
    ta.cnt = reinterpret_cast<int *>(ws + p.off_cnt);
    ta.lidx = reinterpret_cast<int *>(ws + p.off_lidx);
    ta.err = reinterpret_cast<int32_t *>(ws + p.off_err);
    ta.part = reinterpret_cast<float *>(ws + p.off_part);
    ta.gbar = reinterpret_cast<unsigned *>(ws + p.off_err + kCtlBar);
    ta.out = c.out;
    ta.active_idx = c.active_idx;
    ta.n_active = c.n_active;
    const bool q = w->wdtype == SFFN_INT4_G64;
    cudaError_t e;
    if (dense) e = q ? launch_tc_d<true, true>(ta, p, s) : launch_tc_d<false, true>(ta, p, s);
    else e = q ? launch_tc_d<true, false>(ta, p, s) : launch_tc_d<false, false>(ta, p, s);
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
