// decode_q1.cu -- one-token decode with int4-g64 weights on the CUDA cores
// (sm_103a).
//
// The same computation as the other decode kernels (denseflux, "skipping most
// of a dense FFN", sec. 5.1-5.3: the gate read in full, then only the active
// rows of W_up and W_downT; WiSparse write-up sec. 1.2 / 2.3: the threshold on
// |a_j| * ||W_down[:, j]||_2), organised for one token: every weight is used
// once, so the dot products are fp32 FMAs and the work per code is its
// conversion, which is kept short (packed f32x2 arithmetic, two codes per
// instruction) and overlapped with the weight stream.
//
// One CTA per SM owns a chunk of R <= 256 neurons (the decode plan's chunks).
//   stage  At the start, before the wait for the previous kernel, bulk copies
//          bring the chunk's gate rows (one copy per row into a padded row
//          stride; one mbarrier per tile of 16 rows) and their scales into
//          shared memory: the whole chunk in flight at once.
//   gate   The dot products run on the tensor cores (mma.sync m16n8k16, bf16
//          operands, fp32 accumulation), the 16 rows of a tile as M and the
//          columns as K; only one of the 8 N columns carries x, the rest repeat
//          it.  A dot product is a sum over k, so the order of k within an MMA
//          is free: ldmatrix gives a lane 8 consecutive codes of a row, and one
//          mask + XOR per pair of codes (nibbles k and k + 4 of the word) makes
//          the bf16 pair 128 + code + 8, one bf16x2 FMA (times 1, minus 136)
//          leaves the codes exactly; x is laid out once in registers in the
//          same order.  The four MMAs of a 64-column group start from zero and
//          their exact sum is multiplied by the row's fp16 group scale.  The
//          warps split the columns (whole groups); their per-row partials are
//          added in a fixed order.  Bias, act, score and the decision.
//   list   Thread j decides row j; ballots rank the active rows into the
//          chunk's ascending list, and an active row of the first batch starts
//          its own copies at once.
//   batch  Each active row's W_up and W_downT rows with their scales go by bulk
//          copies into one slot of a double-buffered batch (the next batch in
//          flight while one is used).  u_j = W_up[j] . x as in the gate,
//          h_j = a_j u_j; then each thread adds (scale h_j) * code into its 8
//          output columns, rows in ascending order (deterministic), converting
//          codes on the CUDA cores: a byte permute places a nibble under the
//          exponent of 2^23 and a packed f32x2 add of -(2^23 + 8) leaves two
//          codes exactly.
//   finish The per-CTA fp32 partials summed in a fixed order behind a bounded
//          grid barrier, and the lists (decode_finish.cuh).
// The dense layer (every neuron, nothing decided) is the same kernel with every
// row of the chunk active.
#include <algorithm>

#include "common.cuh"
#include "decode_finish.cuh"
#include "internal.h"

namespace sffn {

namespace {

constexpr int kQ1Threads = 256;
constexpr int kQ1Warps = kQ1Threads / 32;
constexpr int kQ1MaxRows = 256;
constexpr int kQ1Tile = 16;                          // rows per MMA tile (and per gate piece)
constexpr int kQ1MaxTiles = kQ1MaxRows / kQ1Tile;
constexpr int kQ1BarBytes = 256;                     // kQ1MaxTiles + 2 mbarriers, padded
constexpr float kQ1Magic = 8388616.0f;               // 2^23 + 8
constexpr size_t kQ1StaticReserve = 7680;            // static shared memory of the kernel, with margin
constexpr size_t kQ1SmemPerSm = 233472;              // shared memory of an SM
constexpr size_t kQ1CtaReserve = 1024;               // shared memory the system keeps per CTA

struct Q1Args {
    const uint8_t *wg, *wu, *wd;  // packed codes [F, d/2], column 2i in the low nibble of byte i
    const __half *sg, *su, *sd;   // fp16 group scales [F, d/64]
    const float *bias, *norms;
    const uint16_t *x;            // bf16 [d]
    int F, R, C, act, mode;
    float tau;
    uint32_t region;              // bytes of the staging region
    int *cnt, *lidx;              // [C], [F]: the chunks' ascending lists at their rows
    float *part;                  // [C, d]
    unsigned *gbar;
    void *out;
    int32_t *active_idx, *n_active, *err;
};

// Shapes for CS = d / 256 column slices of 256 columns: code and scale bytes of
// a row, the padded shared-memory row stride of the gate rows, a batch slot
// (up row + scales, down row + scales) and its padded stride.  A stride of
// 16 mod 128 bytes puts the 8 rows of an ldmatrix on distinct banks.
SFFN_HOST_DEV constexpr uint32_t q1_row_bytes(int cs) { return 128u * cs; }
SFFN_HOST_DEV constexpr uint32_t q1_scale_bytes(int cs) { return 8u * cs; }
SFFN_HOST_DEV constexpr uint32_t q1_gate_stride(int cs) { return q1_row_bytes(cs) + 16u; }
SFFN_HOST_DEV constexpr uint32_t q1_slot_stride(int cs) {
    return ((2u * (q1_row_bytes(cs) + q1_scale_bytes(cs)) + 127u) & ~127u) + 16u;
}
// Warp layout of the contractions: NWC warps across the 4 CS groups of 64
// columns (GPW groups each), NWR warps across the row tiles.
SFFN_HOST_DEV constexpr int q1_nwc(int cs) { return 4 * cs < kQ1Warps ? 4 * cs : kQ1Warps; }
// Up to d_model 2048 two CTAs fit an SM (registers and shared memory), so the
// next call's CTAs stage their gate rows while this call finishes.
SFFN_HOST_DEV constexpr int q1_ctas_per_sm(int cs) { return cs <= 8 ? 2 : 1; }

size_t q1_fixed_bytes(int cs) { return (size_t)kQ1BarBytes + sizeof(float) * (size_t)q1_nwc(cs) * kQ1MaxRows; }

// Bytes the staging region needs: the chunk's gate rows and scales, two batch
// slots, and the down partials of the extra thread groups at the end.
size_t q1_region_need(int cs, int R) {
    const size_t gate = (size_t)R * (q1_gate_stride(cs) + q1_scale_bytes(cs));
    const size_t slots = 2u * (size_t)q1_slot_stride(cs);
    const size_t dg = cs < 8 ? (size_t)(8 / cs) : 1u;  // down thread groups (kQ1Threads / (d / 8), at least 1)
    const size_t red = 4u * 256u * (size_t)cs * (dg - 1);
    return std::max(gate, std::max(slots, red));
}

// The region used: what is needed, grown (within the shared memory a CTA may
// have with q1_ctas_per_sm CTAs per SM) towards R slots, so that a dense
// chunk's rows fit two batches.
uint32_t q1_region_bytes(int cs, int R) {
    const size_t need = q1_region_need(cs, R);
    const size_t per_cta = std::min((size_t)device_smem_optin(), kQ1SmemPerSm / q1_ctas_per_sm(cs) - kQ1CtaReserve);
    const size_t avail = per_cta > kQ1StaticReserve + q1_fixed_bytes(cs) ? per_cta - kQ1StaticReserve - q1_fixed_bytes(cs)
                                                                        : 0;
    const size_t want = std::min((size_t)R * q1_slot_stride(cs), avail);
    return (uint32_t)((std::max(need, want) + 15u) & ~(size_t)15u);
}

size_t q1_smem_bytes(int cs, int R) { return q1_fixed_bytes(cs) + q1_region_bytes(cs, R); }

// D += A * B, m16n8k16, bf16 operands, fp32 accumulators.
SFFN_DEV void q1_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 b16 matrices from shared memory; lane l gives the address of row
// l % 8 of matrix l / 8 and receives word l % 4 of row l / 4 of each.
SFFN_DEV void q1_ldsm4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Nibbles k and k + 4 of a word of codes (two's complement) as an exact bf16
// pair: the nibble XOR 8 OR-ed into the mantissa of 128 gives 128 + code + 8,
// an fma (times 1, minus 136) leaves the code.
template <int K>
SFFN_DEV uint32_t q1_pair(uint32_t w) {
    const uint32_t sh = K ? (w >> (4 * K)) : w;
    uint32_t v;  // (sh & 0x000F000F) ^ 0x43084308 as one three-input logic op
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(v) : "r"(sh), "n"(0x000F000F), "n"(0x43084308));
    uint32_t r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(v), "r"(0x3F803F80u), "r"(0xC308C308u));
    return r;
}

// The 64-column groups of a 16-row tile: per group, rows g and g + 8 of the
// lane's quad (words w[0] / w[1] of the group's first 32 columns, w[2] / w[3]
// of the next 32) as four MMAs against the group's x fragments, the groups'
// chains interleaved; d[i][0] and d[i][2] end as the exact code . x sums of
// rows g and g + 8 over group i.
template <int NGR>
SFFN_DEV void q1_groups(float (&d)[NGR][4], const uint32_t (&w)[NGR][4], const uint32_t (&b)[NGR][8]) {
#pragma unroll
    for (int i = 0; i < NGR; ++i) d[i][0] = d[i][1] = d[i][2] = d[i][3] = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int i = 0; i < NGR; ++i)
            q1_mma(d[i], q1_pair<0>(w[i][2 * h]), q1_pair<0>(w[i][2 * h + 1]), q1_pair<1>(w[i][2 * h]),
                   q1_pair<1>(w[i][2 * h + 1]), b[i][4 * h], b[i][4 * h + 1]);
#pragma unroll
        for (int i = 0; i < NGR; ++i)
            q1_mma(d[i], q1_pair<2>(w[i][2 * h]), q1_pair<2>(w[i][2 * h + 1]), q1_pair<3>(w[i][2 * h]),
                   q1_pair<3>(w[i][2 * h + 1]), b[i][4 * h + 2], b[i][4 * h + 3]);
    }
}

// The codes of byte k of two byte vectors (lo: even columns, hi: odd columns)
// as exact floats: 2^23 + (code + 8) by a byte permute, then minus 2^23 + 8.
SFFN_DEV float2 code_pair(uint32_t lo, uint32_t hi, int k) {
    const float a = __uint_as_float(__byte_perm(lo, 0x4B000000u, (uint32_t)(k | 0x7650)));
    const float b = __uint_as_float(__byte_perm(hi, 0x4B000000u, (uint32_t)(k | 0x7650)));
    return __fadd2_rn(make_float2(a, b), make_float2(-kQ1Magic, -kQ1Magic));
}

// Raise the transaction count an mbarrier phase waits for (no arrival).
SFFN_DEV void q1_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Split a word of 8 codes (two's-complement nibbles, column k at bits 4k) into
// the byte vectors of code + 8 for columns 0, 2, 4, 6 and 1, 3, 5, 7.
SFFN_DEV void split_word(uint32_t w, uint32_t &lo, uint32_t &hi) {
    lo = (w & 0x0F0F0F0Fu) ^ 0x08080808u;
    hi = ((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u;
}

// x fragments of the GPW groups from group g0 on, in the order the codes are
// unpacked: per 32-column block bb and quad lane q, columns 32 bb + 8 q +
// {0,4 | 1,5} and {2,6 | 3,7}.
template <int GPW>
SFFN_DEV void q1_x_frags(uint32_t (&bx)[GPW][8], const uint16_t *x, int g0, int q) {
#pragma unroll
    for (int i = 0; i < GPW; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int bb = 2 * (g0 + i) + h;
            const uint4 v = ldg_v4(x + 32 * bb + 8 * q);
            bx[i][4 * h + 0] = __byte_perm(v.x, v.z, 0x5410);
            bx[i][4 * h + 1] = __byte_perm(v.x, v.z, 0x7632);
            bx[i][4 * h + 2] = __byte_perm(v.y, v.w, 0x5410);
            bx[i][4 * h + 3] = __byte_perm(v.y, v.w, 0x7632);
        }
    }
}

// Row sums over the GPW groups from g0 of one 16-row tile: rows at base + i *
// stride (i clamped below n), group scales at sbase + i * sstride.  The sums
// of rows tile * 16 + (0..15) go to out[0..15] (lanes with q == 0 store).
template <int GPW>
SFFN_DEV void q1_tile_dots(const unsigned char *base, uint32_t stride, const unsigned char *sbase, uint32_t sstride,
                           int tile, int n, int g0, const uint32_t (&bx)[GPW][8], float *out) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lblk = lane >> 4;  // ldmatrix row / 16-byte block
    const int ri = min(kQ1Tile * tile + lrow, n - 1);
    const uint32_t rowaddr = smem_u32(base + (size_t)ri * stride) + 16u * lblk;
    const int r0i = min(kQ1Tile * tile + g, n - 1), r1i = min(kQ1Tile * tile + g + 8, n - 1);
    const unsigned char *s0 = sbase + (size_t)r0i * sstride, *s1 = sbase + (size_t)r1i * sstride;
    uint32_t w[GPW][4];
#pragma unroll
    for (int i = 0; i < GPW; ++i) q1_ldsm4(rowaddr + 32u * (g0 + i), w[i][0], w[i][1], w[i][2], w[i][3]);
    float dd[GPW][4];
    q1_groups<GPW>(dd, w, bx);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int i = 0; i < GPW; ++i) {
        acc0 = fmaf(dd[i][0], __half2float(*reinterpret_cast<const __half *>(s0 + 2 * (g0 + i))), acc0);
        acc1 = fmaf(dd[i][2], __half2float(*reinterpret_cast<const __half *>(s1 + 2 * (g0 + i))), acc1);
    }
    if (q == 0) {
        out[g] = acc0;
        out[g + 8] = acc1;
    }
}

template <int CS, bool DENSE>
__global__ void __launch_bounds__(kQ1Threads, q1_ctas_per_sm(CS)) k_gate_q1(Q1Args a) {
    constexpr int D = 256 * CS;                   // d_model
    constexpr uint32_t RB = q1_row_bytes(CS);
    constexpr uint32_t SB = q1_scale_bytes(CS);
    constexpr uint32_t PS = q1_gate_stride(CS);
    constexpr uint32_t SLOT = q1_slot_stride(CS);
    constexpr int NWC = q1_nwc(CS);               // warps across the columns
    constexpr int GPW = 4 * CS / NWC;             // 64-column groups per warp
    static_assert(NWC == kQ1Warps, "every warp takes every row tile");
    constexpr int WPT = D / 8 > kQ1Threads ? D / 8 / kQ1Threads : 1;  // down: code words per thread
    constexpr int TPR = D / 8 / WPT;              // down: threads per row
    constexpr int DG = kQ1Threads / TPR;          // down: thread groups
    static_assert(DG == (CS < 8 ? 8 / CS : 1), "down thread groups");
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *pbar = reinterpret_cast<uint64_t *>(sm);           // [kQ1MaxTiles] gate tiles
    uint64_t *bbar = pbar + kQ1MaxTiles;                          // [2] batch buffers
    float *red = reinterpret_cast<float *>(sm + kQ1BarBytes);     // [NWC][kQ1MaxRows]
    unsigned char *region = sm + kQ1BarBytes + sizeof(float) * NWC * kQ1MaxRows;
    __shared__ float sbias[kQ1MaxRows], snorm[kQ1MaxRows];
    __shared__ int alist[kQ1MaxRows];
    __shared__ float hval[kQ1MaxRows];
    __shared__ int wcnt[kQ1Warps];
    __shared__ int s_fail;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wc = warp;
    const int q = lane & 3;                        // quad lane of the MMA fragments
    const int F = a.F, R = a.R;
    const int row0 = blockIdx.x * R, nrows = min(R, F - row0);
    const int ntiles = (nrows + kQ1Tile - 1) / kQ1Tile;
    const int cap = (int)(a.region / 2 / SLOT);   // rows per batch buffer
    const uint64_t pol = l2_evict_first_policy();
    const unsigned char *gscale = region + (size_t)R * PS;
    // the gate bias of the chunk's rows (an input, like the weights)
    if (tid < nrows) sbias[tid] = a.bias ? __ldg(a.bias + row0 + tid) : 0.f;

    // ---- stage the chunk's gate rows (weights are inputs of the call, not
    // results of the previous kernel: no dependency wait needed)
    if (tid == 0) {
        for (int t = 0; t < ntiles; ++t) mbar_init(&pbar[t], 1);
        mbar_init(&bbar[0], 1);
        mbar_init(&bbar[1], 1);
        mbar_fence_init();
        s_fail = 0;
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0)
            for (int t = 0; t < ntiles; ++t)
                mbar_arrive_expect_tx(&pbar[t], (uint32_t)min(kQ1Tile, nrows - kQ1Tile * t) * RB +
                                                    (t == 0 ? (uint32_t)nrows * SB : 0u));
        __syncwarp();
        if (lane == 0) bulk_load(region + (size_t)R * PS, a.sg + (size_t)row0 * (SB / 2), (uint32_t)nrows * SB,
                                 &pbar[0], pol);
        for (int r = lane; r < nrows; r += 32)
            bulk_load(region + (size_t)r * PS, a.wg + (size_t)(row0 + r) * RB, RB, &pbar[r / kQ1Tile], pol);
    } else if (DENSE && warp == 1 && lane == 0) {
        // every row is active: its W_up and W_downT rows go to L2 now
        bulk_prefetch_l2(a.wu + (size_t)row0 * RB, (uint32_t)nrows * RB);
        bulk_prefetch_l2(a.wd + (size_t)row0 * RB, (uint32_t)nrows * RB);
        bulk_prefetch_l2(a.su + (size_t)row0 * (SB / 2), (uint32_t)nrows * SB);
        bulk_prefetch_l2(a.sd + (size_t)row0 * (SB / 2), (uint32_t)nrows * SB);
    }

    griddep_wait();
    griddep_launch_dependents();
    const unsigned bar_base = *reinterpret_cast<volatile unsigned *>(a.gbar + 1);
    // the rows' ||W_down[:, j]|| (threshold rule; they may come from the previous kernel)
    if (tid < nrows) snorm[tid] = !DENSE && a.mode == SFFN_MODE_THRESHOLD ? a.norms[row0 + tid] : 0.f;

    uint32_t bx[GPW][8];
    q1_x_frags<GPW>(bx, a.x, wc * GPW, q);
    bool ok = true;
    auto tile_dots = [&](const unsigned char *base, uint32_t stride, const unsigned char *sbase, uint32_t sstride,
                         int tile, int n) {
        q1_tile_dots<GPW>(base, stride, sbase, sstride, tile, n, wc * GPW, bx, red + wc * kQ1MaxRows + kQ1Tile * tile);
    };

    // ---- gate
    ok &= mbar_wait(&pbar[0], 0);  // the scales ride on tile 0
    for (int t = 0; t < ntiles; ++t) {
        ok &= mbar_wait(&pbar[t], 0);
        tile_dots(region, PS, gscale, SB, t, nrows);
    }
    if (!ok) s_fail = 1;
    __syncthreads();

    // ---- decision, the chunk's ascending list and the first batch's copies in
    // one pass: thread tid decides row tid, ranks it by ballots, and an active
    // row among the first `cap` starts its own W_up / W_downT copies at once
    bool on = false;
    float av = 0.f;
    if (tid < nrows) {
        float gs = 0.f;
#pragma unroll
        for (int c = 0; c < NWC; ++c) gs += red[c * kQ1MaxRows + tid];
        av = act_fn(a.act, gs + sbias[tid]);
        if (DENSE) on = true;
        else if (a.mode == SFFN_MODE_EXACT) on = av != 0.f;
        else on = fabsf(av) * snorm[tid] >= a.tau;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, on);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int nact = 0, before = 0;
#pragma unroll
    for (int w = 0; w < kQ1Warps; ++w) {
        before += w < warp ? wcnt[w] : 0;
        nact += wcnt[w];
    }
    const int nbat = (nact + cap - 1) / cap;
    // one active row's W_up and W_downT rows with their scales into slot i % cap
    // of buffer (i / cap) & 1
    auto issue_row = [&](int i, int64_t row, uint64_t *bar) {
        const size_t j = (size_t)row;
        unsigned char *sl = region + (size_t)((i / cap) & 1) * cap * SLOT + (size_t)(i % cap) * SLOT;
        bulk_load(sl, a.wu + j * RB, RB, bar, pol);
        bulk_load(sl + RB, a.su + j * (SB / 2), SB, bar, pol);
        bulk_load(sl + RB + SB, a.wd + j * RB, RB, bar, pol);
        bulk_load(sl + 2 * RB + SB, a.sd + j * (SB / 2), SB, bar, pol);
    };
    if (on) {
        const int m = before + __popc(bal & ((1u << lane) - 1u));
        alist[m] = row0 + tid;
        hval[m] = av;
        if (!DENSE) a.lidx[(size_t)row0 + m] = row0 + tid;
        if (m < cap) {
            fence_proxy_async_smem();  // every warp's reads of the gate rows passed the barrier
            q1_expect_tx(&bbar[0], 2u * (RB + SB));
            issue_row(m, row0 + tid, &bbar[0]);
        }
    }
    if (tid == 0 && !DENSE) a.cnt[blockIdx.x] = nact;
    __syncthreads();  // the list is complete; batch 0's transaction count is raised
    if (tid == 0 && nact > 0) mbar_arrive(&bbar[0]);

    // batch bt >= 1 into buffer bt & 1 (warp 0; the buffer's earlier readers
    // have passed a barrier)
    auto issue_batch = [&](int bt) {
        const int i0 = bt * cap, nb = min(cap, nact - i0);
        uint64_t *bar = &bbar[bt & 1];
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nb * 2u * (RB + SB));
        __syncwarp();
        for (int i = lane; i < nb; i += 32) issue_row(i0 + i, alist[i0 + i], bar);
    };
    if (warp == 0 && nbat > 1) issue_batch(1);

    // down: thread group dg = tid / TPR owns batch rows dg, dg + DG, ...; thread
    // tg of a group owns the 8 WPT columns from col0 (one scale group)
    const int dg = tid / TPR, tg = tid - dg * TPR, col0 = 8 * WPT * tg;
    float2 acc[4 * WPT];
#pragma unroll
    for (int k = 0; k < 4 * WPT; ++k) acc[k] = make_float2(0.f, 0.f);

    for (int bt = 0; bt < nbat; ++bt) {
        const int i0 = bt * cap, nb = min(cap, nact - i0);
        const unsigned char *buf = region + (size_t)(bt & 1) * cap * SLOT;
        ok &= mbar_wait(&bbar[bt & 1], (uint32_t)((bt >> 1) & 1));
        // up dots
        for (int t = 0; t * kQ1Tile < nb; ++t) tile_dots(buf, SLOT, buf + RB, SLOT, t, nb);
        __syncthreads();
        if (tid < nb) {
            float u = 0.f;
#pragma unroll
            for (int c = 0; c < NWC; ++c) u += red[c * kQ1MaxRows + tid];
            hval[i0 + tid] *= u;
        }
        __syncthreads();
        // down rows of the batch, ascending within each thread group
        for (int i = dg; i < nb; i += DG) {
            const unsigned char *s = buf + (size_t)i * SLOT + RB + SB;
            uint32_t w[WPT];
            if (WPT == 2) {
                const uint2 v = *reinterpret_cast<const uint2 *>(s + 8 * tg);
                w[0] = v.x;
                w[WPT - 1] = v.y;
            } else {
                w[0] = *reinterpret_cast<const uint32_t *>(s + 4 * tg);
            }
            const float sh = __half2float(*reinterpret_cast<const __half *>(s + RB + (col0 >> 6) * 2)) * hval[i0 + i];
            const float2 s2 = make_float2(sh, sh);
#pragma unroll
            for (int e = 0; e < WPT; ++e) {
                uint32_t lo, hi;
                split_word(w[e], lo, hi);
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[4 * e + k] = __ffma2_rn(code_pair(lo, hi, k), s2, acc[4 * e + k]);
            }
        }
        __syncthreads();  // buffer bt & 1 and the partial sums are free again
        if (warp == 0 && bt + 2 < nbat) issue_batch(bt + 2);
    }
    if (!ok) s_fail = 1;

    // groups 1.. hand their sums to group 0, which adds them in group order
    if (DG > 1) {
        float2 *gred = reinterpret_cast<float2 *>(region);
        if (dg > 0)
#pragma unroll
            for (int k = 0; k < 4 * WPT; ++k) gred[(size_t)(dg - 1) * (D / 2) + col0 / 2 + k] = acc[k];
        __syncthreads();
        if (dg == 0)
            for (int t = 1; t < DG; ++t)
#pragma unroll
                for (int k = 0; k < 4 * WPT; ++k) {
                    const float2 v = gred[(size_t)(t - 1) * (D / 2) + col0 / 2 + k];
                    acc[k].x += v.x;
                    acc[k].y += v.y;
                }
    }
    if (dg == 0) {
        float4 *dst = reinterpret_cast<float4 *>(a.part + (size_t)blockIdx.x * D + col0);
#pragma unroll
        for (int k = 0; k < 2 * WPT; ++k) dst[k] = make_float4(acc[2 * k].x, acc[2 * k].y, acc[2 * k + 1].x, acc[2 * k + 1].y);
    }
    __syncthreads();
    const bool failed = s_fail != 0;
    if (failed && tid == 0) {
        // a wait gave up: record it, and let every copy this CTA issued land
        // (bounded) before the CTA's shared memory goes away
        record_error(a.err, SFFN_ERR_TIMEOUT);
        for (int t = 0; t < ntiles; ++t) mbar_wait(&pbar[t], 0);
        for (int bt = (nbat > 2 ? nbat - 2 : 0); bt < nbat; ++bt) mbar_wait(&bbar[bt & 1], (uint32_t)((bt >> 1) & 1));
    }

    FinishArgs fa;
    fa.gbar = a.gbar;
    fa.part = a.part;
    fa.nb = 1;
    fa.d = D;
    fa.F = F;
    fa.C = a.C;
    fa.R = R;
    fa.cnt = DENSE ? nullptr : a.cnt;
    fa.lidx = a.lidx;
    fa.out = a.out;
    fa.out_f32 = 0;
    fa.active_idx = a.active_idx;
    fa.n_active = a.n_active;
    fa.err = a.err;
    finish_call(fa, bar_base, failed);
}


// ---------------------------------------------------------------------------
// The dense layer (every neuron) as one stream.  Every row is used, so nothing
// waits for a decision: tiles of 16 rows of W_gate, W_up and W_downT (with
// their scales) flow through a ring of shared-memory stages by bulk copies,
// the first stages before the wait for the previous kernel.  Warps 0-7 take the
// gate and warps 8-15 the up dot products of a tile (the MMA contraction of the
// gate kernel, each warp a share of the 64-column groups); 16 threads form
// h_j = act(g_j + b_j) u_j; then every thread adds (scale h_j) * code of the
// tile's down rows into its 8 output columns (rows in ascending order within a
// thread group, the groups added in order at the end).
constexpr int kQ1DThreads = 512;
constexpr int kQ1DMaxStages = 8;

// Bytes of one stage: 16 gate and 16 up rows at the padded stride, 16 down
// rows, the three matrices' scales.
SFFN_HOST_DEV constexpr uint32_t q1d_stage_bytes(int cs) {
    return 2u * kQ1Tile * q1_gate_stride(cs) + kQ1Tile * q1_row_bytes(cs) + 3u * kQ1Tile * q1_scale_bytes(cs);
}

template <int CS>
__global__ void __launch_bounds__(kQ1DThreads, 1) k_dense_q1(Q1Args a, int nstages) {
    constexpr int D = 256 * CS;
    constexpr uint32_t RB = q1_row_bytes(CS);
    constexpr uint32_t SB = q1_scale_bytes(CS);
    constexpr uint32_t PS = q1_gate_stride(CS);
    constexpr uint32_t ST = q1d_stage_bytes(CS);
    constexpr uint32_t OFF_U = kQ1Tile * PS, OFF_D = 2 * kQ1Tile * PS, OFF_GS = OFF_D + kQ1Tile * RB;
    constexpr uint32_t OFF_US = OFF_GS + kQ1Tile * SB, OFF_DS = OFF_US + kQ1Tile * SB;
    constexpr int GPW = 4 * CS / 8;               // 64-column groups per warp (8 warps per matrix)
    constexpr int TPR = D / 8;                    // down: threads per row (8 columns each)
    constexpr int DG = kQ1DThreads / TPR;         // down: thread groups
    static_assert(DG * TPR == kQ1DThreads, "down thread groups");
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);           // [kQ1DMaxStages]
    unsigned char *stages = sm + 128;
    __shared__ float sbias[kQ1MaxRows];
    __shared__ float red[2][2][8][kQ1Tile];  // [tile parity][gate, up][warp][row]
    __shared__ int s_fail;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mat = warp >> 3, wc = warp & 7;     // 0: gate, 1: up
    const int F = a.F, R = a.R;
    const int row0 = blockIdx.x * R, nrows = min(R, F - row0);
    const int ntiles = (nrows + kQ1Tile - 1) / kQ1Tile;
    const int NS = nstages;
    const uint64_t pol = l2_evict_first_policy();

    // tile tt into its stage (warp 0)
    auto issue_tile = [&](int tt) {
        unsigned char *st = stages + (size_t)(tt % NS) * ST;
        uint64_t *bar = &full[tt % NS];
        const int r0 = kQ1Tile * tt, nr = min(kQ1Tile, nrows - r0);
        const size_t j0 = (size_t)(row0 + r0);
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nr * (3u * RB + 3u * SB));
        __syncwarp();
        if (lane < nr) bulk_load(st + (size_t)lane * PS, a.wg + (j0 + lane) * RB, RB, bar, pol);
        else if (lane >= kQ1Tile && lane - kQ1Tile < nr)
            bulk_load(st + OFF_U + (size_t)(lane - kQ1Tile) * PS, a.wu + (j0 + lane - kQ1Tile) * RB, RB, bar, pol);
        if (lane == 0) bulk_load(st + OFF_D, a.wd + j0 * RB, (uint32_t)nr * RB, bar, pol);
        if (lane == 1) bulk_load(st + OFF_GS, a.sg + j0 * (SB / 2), (uint32_t)nr * SB, bar, pol);
        if (lane == 2) bulk_load(st + OFF_US, a.su + j0 * (SB / 2), (uint32_t)nr * SB, bar, pol);
        if (lane == 3) bulk_load(st + OFF_DS, a.sd + j0 * (SB / 2), (uint32_t)nr * SB, bar, pol);
    };

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
        mbar_fence_init();
        s_fail = 0;
    }
    if (tid < nrows) sbias[tid] = a.bias ? __ldg(a.bias + row0 + tid) : 0.f;
    __syncthreads();
    // weights are inputs of the call: the first stages stream before the wait
    if (warp == 0)
        for (int tt = 0; tt < min(NS, ntiles); ++tt) issue_tile(tt);

    griddep_wait();
    griddep_launch_dependents();
    const unsigned bar_base = *reinterpret_cast<volatile unsigned *>(a.gbar + 1);

    uint32_t bx[GPW][8];
    q1_x_frags<GPW>(bx, a.x, wc * GPW, lane & 3);
    const int dg = tid / TPR, tg = tid - dg * TPR, col0 = 8 * tg;
    float2 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
    bool ok = true;

    for (int t = 0; t < ntiles; ++t) {
        const unsigned char *st = stages + (size_t)(t % NS) * ST;
        ok &= mbar_wait(&full[t % NS], (uint32_t)((t / NS) & 1));
        const int nr = min(kQ1Tile, nrows - kQ1Tile * t);
        // gate (warps 0-7) or up (warps 8-15) sums of the tile's rows
        q1_tile_dots<GPW>(st + (mat ? OFF_U : 0u), PS, st + (mat ? OFF_US : OFF_GS), SB, 0, nr, wc * GPW, bx,
                          red[t & 1][mat][wc]);
        // the sums are in; every thread is done with tile t - 1's stage and with
        // the sums of tile t - 1 (the other half of red, written next by tile t + 1)
        __syncthreads();
        if (warp == 0 && t > 0 && t - 1 + NS < ntiles) issue_tile(t - 1 + NS);
        // every warp forms the tile's h_j (lane j), so no second barrier
        float hj = 0.f;
        if (lane < nr) {
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                gs += red[t & 1][0][c][lane];
                us += red[t & 1][1][c][lane];
            }
            hj = act_fn(a.act, gs + sbias[kQ1Tile * t + lane]) * us;
        }
        // down rows of the tile, ascending within each thread group
#pragma unroll
        for (int k0 = 0; k0 < kQ1Tile; k0 += DG) {
            const int i = k0 + dg;
            const float h = __shfl_sync(0xffffffffu, hj, i & 31);
            if (i < nr) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(st + OFF_D + (size_t)i * RB + 4 * tg);
                const float sh =
                    __half2float(*reinterpret_cast<const __half *>(st + OFF_DS + (size_t)i * SB + (col0 >> 6) * 2)) * h;
                const float2 s2 = make_float2(sh, sh);
                uint32_t lo, hi;
                split_word(w, lo, hi);
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = __ffma2_rn(code_pair(lo, hi, k), s2, acc[k]);
            }
        }
    }
    if (!ok) s_fail = 1;
    __syncthreads();
    // groups 1.. hand their sums to group 0, which adds them in group order
    // (the stage area holds (DG - 1) d floats: q1d_smem_bytes)
    if (DG > 1) {
        float2 *gred = reinterpret_cast<float2 *>(stages);
        if (dg > 0)
#pragma unroll
            for (int k = 0; k < 4; ++k) gred[(size_t)(dg - 1) * (D / 2) + col0 / 2 + k] = acc[k];
        __syncthreads();
        if (dg == 0)
            for (int u = 1; u < DG; ++u)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 v = gred[(size_t)(u - 1) * (D / 2) + col0 / 2 + k];
                    acc[k].x += v.x;
                    acc[k].y += v.y;
                }
    }
    if (dg == 0) {
        float4 *dst = reinterpret_cast<float4 *>(a.part + (size_t)blockIdx.x * D + col0);
        dst[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        dst[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    }
    const bool failed = s_fail != 0;
    if (failed && tid == 0) {
        // a wait gave up: record it and let this CTA's copies land (bounded)
        record_error(a.err, SFFN_ERR_TIMEOUT);
        for (int t = max(0, ntiles - NS); t < ntiles; ++t) mbar_wait(&full[t % NS], (uint32_t)((t / NS) & 1));
    }

    FinishArgs fa;
    fa.gbar = a.gbar;
    fa.part = a.part;
    fa.nb = 1;
    fa.d = D;
    fa.F = F;
    fa.C = a.C;
    fa.R = R;
    fa.cnt = nullptr;
    fa.lidx = a.lidx;
    fa.out = a.out;
    fa.out_f32 = 0;
    fa.active_idx = a.active_idx;
    fa.n_active = a.n_active;
    fa.err = a.err;
    finish_call(fa, bar_base, failed);
}

// ---------------------------------------------------------------------------
// Gate-and-up scores of one token for the keep-ratio rule (WiSparse write-up,
// sec. 2.1: s_j = |a_j u_j| ||W_down[:, j]||): the same stream as the dense
// layer without W_downT.  Tiles of 16 W_gate and W_up rows with their scales
// flow through a ring of bulk-copied stages; warps 0-7 take the gate and 8-15
// the up contraction; 16 threads write s_j, a_j and u_j of the tile's rows.
SFFN_HOST_DEV constexpr uint32_t q1s_stage_bytes(int cs) {
    return 2u * kQ1Tile * q1_gate_stride(cs) + 2u * kQ1Tile * q1_scale_bytes(cs);
}

struct Q1ScoreArgs {
    const uint8_t *wg, *wu;
    const __half *sg, *su;
    const float *bias, *norms;
    const uint16_t *x;
    int F, R, act;
    float *score, *aeff, *uval;   // [F] each; aeff / uval may be null
};

template <int CS>
__global__ void __launch_bounds__(kQ1DThreads, 1) k_scores_q1(Q1ScoreArgs a, int nstages) {
    constexpr uint32_t RB = q1_row_bytes(CS);
    constexpr uint32_t SB = q1_scale_bytes(CS);
    constexpr uint32_t PS = q1_gate_stride(CS);
    constexpr uint32_t ST = q1s_stage_bytes(CS);
    constexpr uint32_t OFF_U = kQ1Tile * PS, OFF_GS = 2 * kQ1Tile * PS, OFF_US = OFF_GS + kQ1Tile * SB;
    constexpr int GPW = 4 * CS / 8;
    extern __shared__ __align__(128) unsigned char sm[];
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    unsigned char *stages = sm + 128;
    __shared__ float sbias[kQ1MaxRows], snorm[kQ1MaxRows];
    __shared__ float red[2][2][8][kQ1Tile];
    __shared__ int s_fail;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mat = warp >> 3, wc = warp & 7;
    const int F = a.F, R = a.R;
    const int row0 = blockIdx.x * R, nrows = min(R, F - row0);
    const int ntiles = (nrows + kQ1Tile - 1) / kQ1Tile;
    const int NS = nstages;
    const uint64_t pol = l2_evict_first_policy();

    auto issue_tile = [&](int tt) {
        unsigned char *st = stages + (size_t)(tt % NS) * ST;
        uint64_t *bar = &full[tt % NS];
        const int r0 = kQ1Tile * tt, nr = min(kQ1Tile, nrows - r0);
        const size_t j0 = (size_t)(row0 + r0);
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nr * (2u * RB + 2u * SB));
        __syncwarp();
        if (lane < nr) bulk_load(st + (size_t)lane * PS, a.wg + (j0 + lane) * RB, RB, bar, pol);
        else if (lane >= kQ1Tile && lane - kQ1Tile < nr)
            bulk_load(st + OFF_U + (size_t)(lane - kQ1Tile) * PS, a.wu + (j0 + lane - kQ1Tile) * RB, RB, bar, pol);
        if (lane == 1) bulk_load(st + OFF_GS, a.sg + j0 * (SB / 2), (uint32_t)nr * SB, bar, pol);
        if (lane == 2) bulk_load(st + OFF_US, a.su + j0 * (SB / 2), (uint32_t)nr * SB, bar, pol);
    };

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
        mbar_fence_init();
        s_fail = 0;
    }
    if (tid < nrows) sbias[tid] = a.bias ? __ldg(a.bias + row0 + tid) : 0.f;
    __syncthreads();
    if (warp == 0)
        for (int tt = 0; tt < min(NS, ntiles); ++tt) issue_tile(tt);

    griddep_wait();
    griddep_launch_dependents();
    // the norms may come from the previous kernel
    if (tid < nrows) snorm[tid] = a.norms ? a.norms[row0 + tid] : 0.f;
    uint32_t bx[GPW][8];
    q1_x_frags<GPW>(bx, a.x, wc * GPW, lane & 3);
    __syncthreads();
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
        const unsigned char *st = stages + (size_t)(t % NS) * ST;
        ok &= mbar_wait(&full[t % NS], (uint32_t)((t / NS) & 1));
        const int nr = min(kQ1Tile, nrows - kQ1Tile * t);
        q1_tile_dots<GPW>(st + (mat ? OFF_U : 0u), PS, st + (mat ? OFF_US : OFF_GS), SB, 0, nr, wc * GPW, bx,
                          red[t & 1][mat][wc]);
        // the sums are in; every thread is done with tile t - 1's stage and sums
        __syncthreads();
        if (warp == 0 && t > 0 && t - 1 + NS < ntiles) issue_tile(t - 1 + NS);
        if (tid < nr) {
            float gs = 0.f, us = 0.f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                gs += red[t & 1][0][c][tid];
                us += red[t & 1][1][c][tid];
            }
            const int r = kQ1Tile * t + tid;
            const float av = act_fn(a.act, gs + sbias[r]);
            const size_t j = (size_t)(row0 + r);
            a.score[j] = fabsf(av * us) * snorm[r];
            if (a.aeff) a.aeff[j] = av;
            if (a.uval) a.uval[j] = us;
        }
    }
    if (!ok) s_fail = 1;
    __syncthreads();
    if (s_fail && tid == 0) {
        // a wait gave up: let this CTA's copies land (bounded); the scores are not valid
        for (int t = max(0, ntiles - NS); t < ntiles; ++t) mbar_wait(&full[t % NS], (uint32_t)((t / NS) & 1));
    }
}

int q1s_stages(int cs, int R) {
    const size_t avail = (size_t)device_smem_optin() - 128 - 6144;  // barriers; static shared memory
    const int ntiles = (R + kQ1Tile - 1) / kQ1Tile;
    int ns = (int)(avail / q1s_stage_bytes(cs));
    ns = std::min(std::min(ns, kQ1DMaxStages), ntiles);
    return ns >= 2 || (ns == 1 && ntiles == 1) ? ns : 0;
}

template <int CS>
cudaError_t launch_q1s(const Q1ScoreArgs &sa, int C, int ns, cudaStream_t s) {
    const size_t smem = 128 + (size_t)ns * q1s_stage_bytes(CS);
    cudaError_t e = set_max_smem((const void *)k_scores_q1<CS>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_scores_q1<CS>, dim3(C), dim3(kQ1DThreads), smem, s, sa, ns);
}

// Stages of the dense stream that fit the shared memory of one CTA (0: it
// does not fit twice).
int q1d_stages(int cs, int R) {
    const size_t avail = (size_t)device_smem_optin() - 128 - 4096;  // barriers; static shared memory
    const int ntiles = (R + kQ1Tile - 1) / kQ1Tile;
    int ns = (int)(avail / q1d_stage_bytes(cs));
    ns = std::min(std::min(ns, kQ1DMaxStages), ntiles);
    return ns >= 2 || (ns == 1 && ntiles == 1) ? ns : 0;
}

// Shared memory of the dense stream: barriers, then the stages, which must
// also hold the down sums of thread groups 1.. at the end ((DG - 1) d floats,
// DG = 4096 / d).
size_t q1d_smem_bytes(int cs, int ns) {
    const size_t d = 256u * (size_t)cs;
    return 128 + std::max((size_t)ns * q1d_stage_bytes(cs), 4u * (4096u - d));
}

template <int CS>
cudaError_t launch_q1d(const Q1Args &qa, int C, int ns, cudaStream_t s) {
    const size_t smem = q1d_smem_bytes(CS, ns);
    cudaError_t e = set_max_smem((const void *)k_dense_q1<CS>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_dense_q1<CS>, dim3(C), dim3(kQ1DThreads), smem, s, qa, ns);
}

template <int CS, bool DENSE>
cudaError_t launch_q1(const Q1Args &qa, int C, cudaStream_t s) {
    const size_t smem = q1_smem_bytes(CS, qa.R);
    cudaError_t e = set_max_smem((const void *)k_gate_q1<CS, DENSE>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_k(k_gate_q1<CS, DENSE>, dim3(C), dim3(kQ1Threads), smem, s, qa);
}

template <int CS>
cudaError_t launch_q1_d(const Q1Args &qa, int C, bool dense, cudaStream_t s) {
    return dense ? launch_q1<CS, true>(qa, C, s) : launch_q1<CS, false>(qa, C, s);
}

int q1_slices(int d) { return d == 512 ? 2 : d == 1024 ? 4 : d == 2048 ? 8 : d == 4096 ? 16 : 0; }

}  // namespace

bool scores_q1_eligible(const sffn_ffn_weights *w, const DecodePlan &p) {
    if (w->wdtype != SFFN_INT4_G64 || p.nb != 1) return false;
    const int cs = q1_slices(w->d_model);
    return cs != 0 && p.R <= kQ1MaxRows && q1s_stages(cs, p.R) > 0;
}

cudaError_t run_scores_q1(const sffn_ffn_weights *w, const void *x, const DecodePlan &p, float *score, float *aeff,
                          float *uval, cudaStream_t s) {
    Q1ScoreArgs sa = {};
    sa.wg = static_cast<const uint8_t *>(w->w_gate);
    sa.wu = static_cast<const uint8_t *>(w->w_up);
    sa.sg = static_cast<const __half *>(w->s_gate);
    sa.su = static_cast<const __half *>(w->s_up);
    sa.bias = w->b_gate;
    sa.norms = w->down_norms;
    sa.x = static_cast<const uint16_t *>(x);
    sa.F = p.F;
    sa.R = p.R;
    sa.act = w->act;
    sa.score = score;
    sa.aeff = aeff;
    sa.uval = uval;
    const int cs = q1_slices(p.d), ns = q1s_stages(cs, p.R);
    switch (cs) {
    case 2: return launch_q1s<2>(sa, p.C, ns, s);
    case 4: return launch_q1s<4>(sa, p.C, ns, s);
    case 8: return launch_q1s<8>(sa, p.C, ns, s);
    case 16: return launch_q1s<16>(sa, p.C, ns, s);
    default: return cudaErrorInvalidValue;
    }
}

bool decode_q1_eligible(const DecodeCall &c, const DecodePlan &p, bool dense) {
    const sffn_ffn_weights *w = c.w;
    if (w->wdtype != SFFN_INT4_G64 || c.B != 1 || c.scores_only) return false;
    const int cs = q1_slices(w->d_model);
    if (cs == 0 || p.R > kQ1MaxRows || p.C > device_sm_count()) return false;
    if (q1_fixed_bytes(cs) + q1_region_need(cs, p.R) + kQ1StaticReserve > (size_t)device_smem_optin()) return false;
    if (dense) return true;
    return c.mode == SFFN_MODE_EXACT || (c.mode == SFFN_MODE_THRESHOLD && c.score == SFFN_SCORE_GATE);
}

sffn_status run_decode_q1(const DecodeCall &c, const DecodePlan &p, cudaStream_t s, bool dense) {
    char *ws = static_cast<char *>(c.ws);
    const sffn_ffn_weights *w = c.w;
    const int cs = q1_slices(p.d);
    Q1Args qa = {};
    qa.wg = static_cast<const uint8_t *>(w->w_gate);
    qa.wu = static_cast<const uint8_t *>(w->w_up);
    qa.wd = static_cast<const uint8_t *>(w->w_downT);
    qa.sg = static_cast<const __half *>(w->s_gate);
    qa.su = static_cast<const __half *>(w->s_up);
    qa.sd = static_cast<const __half *>(w->s_downT);
    qa.bias = w->b_gate;
    qa.norms = w->down_norms;
    qa.x = static_cast<const uint16_t *>(c.x);
    qa.F = p.F;
    qa.R = p.R;
    qa.C = p.C;
    qa.act = w->act;
    qa.mode = c.mode;
    qa.tau = c.param;
    qa.region = q1_region_bytes(cs, p.R);
    qa.cnt = reinterpret_cast<int *>(ws + p.off_cnt);
    qa.lidx = reinterpret_cast<int *>(ws + p.off_lidx);
    qa.part = reinterpret_cast<float *>(ws + p.off_part);
    qa.gbar = reinterpret_cast<unsigned *>(ws + p.off_err + kCtlBar);
    qa.out = c.out;
    qa.active_idx = c.active_idx;
    qa.n_active = c.n_active;
    qa.err = reinterpret_cast<int32_t *>(ws + p.off_err);
    cudaError_t e;
    const int ns = dense ? q1d_stages(cs, p.R) : 0;
    if (ns > 0) {
        switch (cs) {
        case 2: e = launch_q1d<2>(qa, p.C, ns, s); break;
        case 4: e = launch_q1d<4>(qa, p.C, ns, s); break;
        case 8: e = launch_q1d<8>(qa, p.C, ns, s); break;
        case 16: e = launch_q1d<16>(qa, p.C, ns, s); break;
        default: return SFFN_ERR_UNSUPPORTED;
        }
        return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
    }
    switch (cs) {
    case 2: e = launch_q1_d<2>(qa, p.C, dense, s); break;
    case 4: e = launch_q1_d<4>(qa, p.C, dense, s); break;
    case 8: e = launch_q1_d<8>(qa, p.C, dense, s); break;
    case 16: e = launch_q1_d<16>(qa, p.C, dense, s); break;
    default: return SFFN_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
