// prefill.cu -- token-selective prefill (sm_103a): residual + gather, and the two
// tensor-core GEMMs of the FFN on the selected tokens.
//
// RedKnot Algorithm 1 (bhfrc.com/news/43276): S <- Select(A); Z[S] <- FFN(Y[S]);
// Z[~S] <- 0; X_next <- Y + Z.  Here Y = bf16(X + Y_attn) is the post-attention
// residual stream and FFN(y) = W_down (SiLU(W_gate y) (.) (W_up y)).
//
//   residual_gather  out[t] = Y[t] for every token (the final value for the
//                    unselected ones), Ysel[i] = Y[sel[i]] compacted
//   gemm<SwiGLU>     H = SiLU(Ysel W_gate^T) (.) (Ysel W_up^T): one tcgen05.mma
//                    of N = 256 covers 128 gate and the matching 128 up rows
//                    (stacked in shared memory), the epilogue reads both halves
//                    of the fp32 accumulator from TMEM and writes bf16 H
//   gemm<Down>       Z = H W_down with B = W_downT read MN-major straight from
//                    its [d_ff, d_model] layout (no transposed copy); the
//                    epilogue writes out[sel[i]] = bf16(Ysel[i] + Z[i])
//
// Both GEMMs are persistent (one CTA per SM), warp specialised: warp 0 issues
// TMA tile loads into a 4-stage shared-memory ring (128-byte swizzle), warp 1
// owns the TMEM allocation and issues tcgen05.mma (128 x 256 x 16, fp32
// accumulators double-buffered in TMEM), warps 2-5 drain TMEM with tcgen05.ld.
// With int4-g64 weights (the RedKnot write-up measures INT4 Qwen3-32B) warps
// 6-13 fill each stage's weight tile instead of TMA: a thread loads one
// 64-code run of a stored row (32 bytes, six stages ahead) and its fp16 group
// scale, and writes the 64 values code * scale in bf16 (see dequant_row64) as
// one 128-byte row of the tile in the same 128-byte swizzle the MMA
// descriptors expect (K-major for W_gate / W_up, MN-major for W_downT).
// Tiles are rasterised in groups of m-tiles so weight tiles are reused from L2.
// Every mbarrier wait is bounded; the selected-token count and indices are
// read on the device and checked against L.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace sffn {

// ---------------------------------------------------------------------------
// residual + gather
// ---------------------------------------------------------------------------

constexpr int kResWarps = 8;

__global__ void __launch_bounds__(32 * kResWarps) k_residual_gather(const uint16_t *x, const uint16_t *ya, int L,
                                                                     int d, const int32_t *sel, const int32_t *n_sel,
                                                                     uint16_t *out, uint16_t *ysel, int32_t *err) {
    griddep_wait();
    griddep_launch_dependents();
    int nsel = *n_sel;
    if (nsel < 0 || nsel > L) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, SFFN_ERR_DEVICE);
        nsel = nsel < 0 ? 0 : L;
    }
    const int lane = threadIdx.x & 31;
    const int units = d / 8;
    const long long items = (long long)L + nsel;
    const long long gw = (long long)blockIdx.x * kResWarps + (threadIdx.x >> 5);
    const long long nw = (long long)gridDim.x * kResWarps;
    for (long long it = gw; it < items; it += nw) {
        int t;
        uint16_t *dst;
        if (it < L) {
            t = (int)it;
            dst = out + (size_t)t * d;
        } else {
            const int i = (int)(it - L);
            t = sel[i];
            if (t < 0 || t >= L) {
                if (lane == 0) record_error(err, SFFN_ERR_DEVICE);
                continue;
            }
            dst = ysel + (size_t)i * d;
        }
        const char *xr = reinterpret_cast<const char *>(x + (size_t)t * d);
        const char *yr = reinterpret_cast<const char *>(ya + (size_t)t * d);
        constexpr int U = 4;
        for (int u0 = 0; u0 < units; u0 += 32 * U) {
            uint4 xv[U], yv[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int u = u0 + k * 32 + lane;
                if (u < units) {
                    xv[k] = ldg_stream(xr + (size_t)u * 16);
                    yv[k] = ldg_stream(yr + (size_t)u * 16);
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int u = u0 + k * 32 + lane;
                if (u < units) {
                    uint4 r;  // Y = bf16(X + Y_attn), one rounding of the exact sum
                    r.x = bf16x2_add_rn(xv[k].x, yv[k].x);
                    r.y = bf16x2_add_rn(xv[k].y, yv[k].y);
                    r.z = bf16x2_add_rn(xv[k].z, yv[k].z);
                    r.w = bf16x2_add_rn(xv[k].w, yv[k].w);
                    reinterpret_cast<uint4 *>(dst)[u] = r;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// persistent tcgen05 GEMM
// ---------------------------------------------------------------------------

constexpr int GBM = 128;                         // rows (selected tokens) per tile
constexpr int GBK = 64;                          // K per stage (one 128-byte swizzle row)
constexpr int GMMA_N = 256;                      // N of one tcgen05.mma
constexpr int GSTAGES = 4;
constexpr int G_A_BYTES = GBM * GBK * 2;         // 16 KB
constexpr int G_B_BYTES = GMMA_N * GBK * 2;      // 32 KB
constexpr int G_STAGE_BYTES = G_A_BYTES + G_B_BYTES;
constexpr int kGemmThreads = 192;                // producer, MMA, 4 epilogue warps
constexpr int kDequantThreads = 256;             // int4 weights: one 64-code run of the tile per thread
constexpr int kTmemCols = 2 * GMMA_N;            // two accumulators of 128 x 256 fp32
constexpr size_t kGemmSmem = (size_t)GSTAGES * G_STAGE_BYTES + 1024 /*alignment*/ + 256 /*barriers*/;

enum { EPI_SWIGLU = 0, EPI_DOWN = 1 };

struct GemmArgs {
    const int32_t *n_sel;      // selected-token count (device)
    // int4-g64 weights: packed codes [F, d/2] (low nibble = even column) and fp16
    // group scales [F, d/64]; SwiGLU: W_gate (0) and W_up (1); Down: W_downT (0)
    const uint8_t *qw0, *qw1;
    const __half *qs0, *qs1;
    int qd;                    // d_model
    const int32_t *sel_idx;    // EPI_DOWN: selected token ids, ascending
    const uint16_t *ysel;      // EPI_DOWN: compact residual rows [L, d]
    uint16_t *out;             // EPI_SWIGLU: H [L, d_ff]; EPI_DOWN: out [L, d]
    int L;
    int n_out;                 // output columns (d_ff for H, d_model for out)
    int tile_n;                // output columns per tile (128 / 256)
    int kblocks;               // K / 64
    int group_m;               // m-tiles per rasterisation group
    int32_t *err;
};

SFFN_DEV void tile_coords(int t, int m_tiles, int n_tiles, int group_m, int &mt, int &nt) {
    const int per_group = group_m * n_tiles;
    const int g = t / per_group;
    const int first_m = g * group_m;
    const int gm = min(group_m, m_tiles - first_m);
    const int local = t - g * per_group;
    mt = first_m + local % gm;
    nt = local / gm;
}

// 64 int4 codes (32 bytes) times the group scale in bf16, as one 128-byte
// tile row with its 16-byte chunks in 128-byte swizzle order.  Per pair of
// columns (2e, 2e+1): one byte permute and one LOP3 place the two unsigned
// nibbles (code + 8) in the mantissas of bf16 128.0, one bf16x2 fma subtracts
// 136 (the codes, exactly), one bf16x2 multiply applies the scale s2 = (s, s)
// (the fp16 scale rounded to bf16): two roundings to bf16, relative error at
// most 2^-8 per weight.
SFFN_DEV uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

SFFN_DEV void dequant_row64(const uint4 &c0, const uint4 &c1, uint32_t s2, unsigned char *dst_row, int key) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t v = w[c] ^ 0x88888888u;  // code + 8 per nibble; column k in bits 4k
        const uint32_t lo = v & 0x0F0F0F0Fu, hi = (v >> 4) & 0x0F0F0F0Fu;  // byte e: column 2e / 2e + 1
        uint32_t pk[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t p = (__byte_perm(lo, hi, (uint32_t)(e | ((4 + e) << 8))) & 0x00FF00FFu) | 0x43004300u;
            const uint32_t code = bf16x2_fma(p, 0x3F803F80u, 0xC308C308u);  // p * 1 - 136
            pk[e] = bf16x2_fma(code, s2, 0x80008000u);                     // code * s + (-0)
        }
        *reinterpret_cast<uint4 *>(dst_row + ((c ^ key) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
}

template <int EPI, bool QB>
__global__ void __launch_bounds__(kGemmThreads + (QB ? kDequantThreads : 0), 1)
    k_gemm(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b0,
           const __grid_constant__ CUtensorMap map_b1, const GemmArgs a) {
    extern __shared__ unsigned char gsm_raw[];
    unsigned char *gsm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(gsm + GSTAGES * G_STAGE_BYTES);
    uint64_t *empty = full + GSTAGES;
    uint64_t *tfull = empty + GSTAGES;    // [2] accumulator ready
    uint64_t *tempty = tfull + 2;         // [2] accumulator drained
    uint64_t *mdone = tempty + 2;         // all MMAs of this CTA complete
    uint64_t *bready = mdone + 1;         // [GSTAGES] int4: the stage's weight tile is written
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bready + GSTAGES);
    __shared__ volatile int s_abort;
    __shared__ int s_consumed;            // k-blocks consumed by the MMA warp (for draining)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < GSTAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(mdone, 1);
        if (QB)
            for (int s = 0; s < GSTAGES; ++s) mbar_init(&bready[s], kDequantThreads / 32);
        s_abort = 0;
        s_consumed = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&map_a);
        if (!QB) {
            tc::prefetch_tensormap(&map_b0);
            if (EPI == EPI_SWIGLU) tc::prefetch_tensormap(&map_b1);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    griddep_wait();  // Ysel / H / sel come from the previous kernels
    int nsel = *a.n_sel;
    if (nsel < 0 || nsel > a.L) {
        if (tid == 0 && blockIdx.x == 0) record_error(a.err, SFFN_ERR_DEVICE);
        nsel = nsel < 0 ? 0 : a.L;
    }
    const int m_tiles = (nsel + GBM - 1) / GBM;
    const int n_tiles = (a.n_out + a.tile_n - 1) / a.tile_n;
    const int num_tiles = m_tiles * n_tiles;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int it = 0;
            for (int t = blockIdx.x; t < num_tiles && !s_abort; t += gridDim.x) {
                int mt, nt;
                tile_coords(t, m_tiles, n_tiles, a.group_m, mt, nt);
                for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
                    const int s = it % GSTAGES, r = it / GSTAGES;
                    if (!mbar_wait(&empty[s], (uint32_t)((r & 1) ^ 1))) {
                        s_abort = 1;
                        record_error(a.err, SFFN_ERR_TIMEOUT);
                        break;
                    }
                    unsigned char *st = gsm + s * G_STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], QB ? G_A_BYTES : G_STAGE_BYTES);
                    const uint64_t pol = tc::l2_evict_last_policy();
                    tc::tma_load_2d(st, &map_a, kb * GBK, mt * GBM, &full[s], pol);
                    if (QB) {
                        // the weight tile is written by the dequantising warps
                    } else if (EPI == EPI_SWIGLU) {
                        tc::tma_load_2d(st + G_A_BYTES, &map_b0, kb * GBK, nt * 128, &full[s], pol);
                        tc::tma_load_2d(st + G_A_BYTES + G_B_BYTES / 2, &map_b1, kb * GBK, nt * 128, &full[s], pol);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tc::tma_load_2d(st + G_A_BYTES + q * (G_B_BYTES / 4), &map_b0, nt * GMMA_N + q * 64,
                                            kb * GBK, &full[s], pol);
                    }
                }
            }
            if (s_abort) {
                // let this CTA's copies in flight land before the CTA can exit
                __threadfence_block();
                const int done = s_consumed;
                for (int j = done; j < it; ++j) mbar_wait(&full[j % GSTAGES], (uint32_t)((j / GSTAGES) & 1));
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_f32(GBM, GMMA_N, EPI == EPI_DOWN);
            int it = 0, tcount = 0;
            for (int t = blockIdx.x; t < num_tiles && !s_abort; t += gridDim.x, ++tcount) {
                const int b = tcount & 1, rr = tcount >> 1;
                if (!mbar_wait(&tempty[b], (uint32_t)((rr & 1) ^ 1))) {
                    s_abort = 1;
                    record_error(a.err, SFFN_ERR_TIMEOUT);
                    break;
                }
                tc::fence_after_sync();
                const uint32_t dtm = tmem + (uint32_t)(b * GMMA_N);
                for (int kb = 0; kb < a.kblocks; ++kb, ++it) {
                    const int s = it % GSTAGES, r = it / GSTAGES;
                    if (!mbar_wait(&full[s], (uint32_t)(r & 1)) || (QB && !mbar_wait(&bready[s], (uint32_t)(r & 1)))) {
                        s_abort = 1;
                        record_error(a.err, SFFN_ERR_TIMEOUT);
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a_addr = smem_u32(gsm + s * G_STAGE_BYTES);
                    const uint32_t b_addr = a_addr + G_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < GBK / 16; ++kk) {
                        const uint64_t ad = tc::smem_desc_sw128(a_addr + kk * 32, 16, 1024);
                        const uint64_t bd = EPI == EPI_SWIGLU ? tc::smem_desc_sw128(b_addr + kk * 32, 16, 1024)
                                                              : tc::smem_desc_sw128(b_addr + kk * 2048, G_B_BYTES / 4, 1024);
                        tc::mma_bf16(dtm, ad, bd, idesc, (kb | kk) != 0);
                    }
                    tc::mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
                    s_consumed = it + 1;
                }
                if (s_abort) break;
                tc::mma_commit(&tfull[b]);
            }
            // every MMA of this CTA has completed before teardown
            tc::mma_commit(mdone);
            mbar_wait(mdone, 0);
        }
    } else if (QB && warp >= 6) {
        // ---------------- int4 weights: dequantise each stage's weight tile ----------------
        const int u = tid - kGemmThreads;  // this thread's 64-code run of the tile
        const int key = u & 7;             // 128-byte swizzle: chunk c lands at c ^ (row & 7)
        // unit u of item (tile t, k-block kb): source codes, scale and tile row
        auto src_of = [&](int t, int kb, const uint8_t *&cp, const __half *&sp, int &off) -> bool {
            int mt, nt;
            tile_coords(t, m_tiles, n_tiles, a.group_m, mt, nt);
            (void)mt;
            if (EPI == EPI_SWIGLU) {
                const int half = u >> 7, i = u & 127, n = nt * 128 + i;
                cp = (half ? a.qw1 : a.qw0) + (size_t)n * (a.qd / 2) + kb * 32;
                sp = (half ? a.qs1 : a.qs0) + (size_t)n * (a.qd / 64) + kb;
                off = half * (G_B_BYTES / 2) + i * 128;
                return true;
            } else {
                const int q = u >> 6, k = u & 63, row = kb * GBK + k, col = nt * GMMA_N + q * 64;
                off = q * (G_B_BYTES / 4) + k * 128;
                if (col >= a.n_out) return false;  // beyond d_model: zeros
                cp = a.qw0 + (size_t)row * (a.qd / 2) + col / 2;
                sp = a.qs0 + (size_t)row * (a.qd / 64) + col / 64;
                return true;
            }
        };
        struct Run {
            uint4 c0, c1;
            uint32_t s2;  // the group scale as a bf16 pair
            bool ok;
        };
        auto fetch = [&](int t, int kb) {
            Run rn{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), 0u, false};
            const uint8_t *cp;
            const __half *sp;
            int off;
            if (t < num_tiles && src_of(t, kb, cp, sp, off)) {
                rn.c0 = ldg_stream(cp);
                rn.c1 = ldg_stream(cp + 16);
                const uint32_t sb = f32_to_bf16_bits(__half2float(__ldg(sp)));
                rn.s2 = sb | (sb << 16);
                rn.ok = true;
            }
            return rn;
        };
        auto advance = [&](int &t, int &kb) {
            if (++kb == a.kblocks) {
                kb = 0;
                t += gridDim.x;
            }
        };
        // kLook items ahead: the code loads of item it + kLook are issued when item
        // it has been written (registers, rotated by a fully unrolled inner loop)
        constexpr int kLook = 6;
        Run q[kLook];
        int t = blockIdx.x, kb = 0, tf = blockIdx.x, kbf = 0;
#pragma unroll
        for (int i = 0; i < kLook; ++i) {
            q[i] = fetch(tf, kbf);
            advance(tf, kbf);
        }
        bool run = true;
        for (int it0 = 0; run; it0 += kLook) {
#pragma unroll
            for (int i = 0; i < kLook; ++i) {
                if (!run) break;
                if (t >= num_tiles || s_abort) {
                    run = false;
                    break;
                }
                const int it = it0 + i, s = it % GSTAGES, r = it / GSTAGES;
                const bool ok = mbar_wait(&empty[s], (uint32_t)((r & 1) ^ 1));
                if (!__all_sync(0xffffffffu, ok && !s_abort)) {
                    if (lane == 0 && !ok) {
                        s_abort = 1;
                        record_error(a.err, SFFN_ERR_TIMEOUT);
                    }
                    run = false;
                    break;
                }
                const uint8_t *cp;
                const __half *sp;
                int off;
                src_of(t, kb, cp, sp, off);
                unsigned char *dst = gsm + s * G_STAGE_BYTES + G_A_BYTES + off;
                if (q[i].ok) {
                    dequant_row64(q[i].c0, q[i].c1, q[i].s2, dst, key);
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(dst + 16 * c) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();  // the tile is read by the tensor cores (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(&bready[s]);
                q[i] = fetch(tf, kbf);
                advance(tf, kbf);
                advance(t, kb);
            }
        }
    } else {
        // ---------------- epilogue: warps 2..5, TMEM lane quadrant warp % 4 ----------------
        const int q = warp & 3;
        int tcount = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tcount) {
            int mt, nt;
            tile_coords(t, m_tiles, n_tiles, a.group_m, mt, nt);
            const int b = tcount & 1, rr = tcount >> 1;
            const bool ok = mbar_wait(&tfull[b], (uint32_t)(rr & 1));
            if (!__all_sync(0xffffffffu, ok && !s_abort)) {
                if (lane == 0 && !ok) {
                    s_abort = 1;
                    record_error(a.err, SFFN_ERR_TIMEOUT);
                }
                break;
            }
            tc::fence_after_sync();
            const int row = mt * GBM + q * 32 + lane;
            const bool valid = row < nsel;
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * GMMA_N);
            if (EPI == EPI_SWIGLU) {
                uint16_t *hrow = a.out + (size_t)row * a.n_out + (size_t)nt * 128;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], u[32];
                    tc::tmem_ld32(tbase + c * 32, g);
                    tc::tmem_ld32(tbase + 128 + c * 32, u);
                    tc::tmem_wait_ld();
                    if (valid && nt * 128 + c * 32 < a.n_out) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                            const float h0 = act_fn(SFFN_ACT_SILU, g0) * __uint_as_float(u[2 * i]);
                            const float h1 = act_fn(SFFN_ACT_SILU, g1) * __uint_as_float(u[2 * i + 1]);
                            pk[i] = (uint32_t)f32_to_bf16_bits(h0) | ((uint32_t)f32_to_bf16_bits(h1) << 16);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(hrow + c * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
            } else {
                int tok = 0;
                bool ok_row = valid;
                if (valid) {
                    tok = a.sel_idx[row];
                    if (tok < 0 || tok >= a.L) {
                        record_error(a.err, SFFN_ERR_DEVICE);
                        ok_row = false;
                    }
                }
                const uint16_t *yrow = a.ysel + (size_t)row * a.n_out + (size_t)nt * GMMA_N;
                uint16_t *orow = a.out + (size_t)tok * a.n_out + (size_t)nt * GMMA_N;
#pragma unroll 1
                for (int c = 0; c < GMMA_N / 32; ++c) {
                    uint32_t z[32];
                    tc::tmem_ld32(tbase + c * 32, z);
                    tc::tmem_wait_ld();
                    if (ok_row && nt * GMMA_N + c * 32 < a.n_out) {
                        const uint4 *ys = reinterpret_cast<const uint4 *>(yrow + c * 32);
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const uint4 yv = ys[v];
                            const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
                            uint32_t o[4];
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                const float lo = bf16lo(yw[w]) + __uint_as_float(z[8 * v + 2 * w]);
                                const float hi = bf16hi(yw[w]) + __uint_as_float(z[8 * v + 2 * w + 1]);
                                o[w] = (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
                            }
                            dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }
    griddep_launch_dependents();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled get_encode() {
    static PFN_encodeTiled fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled>(p);
    }
    return fn;
}

// 2-D bf16 row-major tensor [rows, cols] with 128-byte swizzled boxes
// {box_cols (<= 64), box_rows}; out-of-range elements read as zero.
static bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                     uint32_t box_rows) {
    PFN_encodeTiled enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

PrefillPlan make_prefill_plan(int L, int d, int F) {
    PrefillPlan p = {};
    p.L = L;
    p.d = d;
    p.F = F;
    size_t o = 0;
    p.off_err = o; o = align_up(o + kControlBytes);  // the control block
    p.off_ysel = o; o = align_up(o + sizeof(uint16_t) * (size_t)L * d);
    p.off_h = o; o = align_up(o + sizeof(uint16_t) * (size_t)L * F);
    p.total = o;
    return p;
}

sffn_status run_prefill(const void *x, const void *y_attn, int L, const sffn_ffn_weights *w, const int32_t *sel_idx,
                        const int32_t *n_sel, void *out, void *ws, const PrefillPlan &p, cudaStream_t s) {
    char *wsb = static_cast<char *>(ws);
    int32_t *err = reinterpret_cast<int32_t *>(wsb + p.off_err);
    uint16_t *ysel = reinterpret_cast<uint16_t *>(wsb + p.off_ysel);
    uint16_t *h = reinterpret_cast<uint16_t *>(wsb + p.off_h);
    const int d = p.d, F = p.F;
    const int sms = device_sm_count();

    const bool q = w->wdtype == SFFN_INT4_G64;
    CUtensorMap m_ysel, m_wg, m_wu, m_h, m_wd;
    if (!make_map(&m_ysel, ysel, (uint64_t)L, (uint64_t)d, GBK, GBM) ||
        !make_map(&m_h, h, (uint64_t)L, (uint64_t)F, GBK, GBM))
        return SFFN_ERR_UNSUPPORTED;
    if (q) {  // the weight tiles are dequantised in the kernel: no weight maps
        m_wg = m_wu = m_ysel;
        m_wd = m_h;
    } else if (!make_map(&m_wg, w->w_gate, (uint64_t)F, (uint64_t)d, GBK, 128) ||
               !make_map(&m_wu, w->w_up, (uint64_t)F, (uint64_t)d, GBK, 128) ||
               !make_map(&m_wd, w->w_downT, (uint64_t)F, (uint64_t)d, 64, GBK)) {
        return SFFN_ERR_UNSUPPORTED;
    }

    long long items = 2LL * L;
    int grid = (int)((items + kResWarps - 1) / kResWarps);
    if (grid > 8 * sms) grid = 8 * sms;
    cudaError_t e = launch_k(k_residual_gather, dim3(grid), dim3(32 * kResWarps), 0, s,
                             static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(y_attn), L, d, sel_idx,
                             n_sel, static_cast<uint16_t *>(out), ysel, err);
    if (e != cudaSuccess) return SFFN_ERR_CUDA;

    GemmArgs g1 = {};
    g1.n_sel = n_sel;
    g1.out = h;
    g1.L = L;
    g1.n_out = F;
    g1.tile_n = 128;
    g1.kblocks = (d + GBK - 1) / GBK;
    g1.group_m = 16;
    g1.err = err;
    g1.qw0 = static_cast<const uint8_t *>(w->w_gate);
    g1.qw1 = static_cast<const uint8_t *>(w->w_up);
    g1.qs0 = static_cast<const __half *>(w->s_gate);
    g1.qs1 = static_cast<const __half *>(w->s_up);
    g1.qd = d;
    if (q) {
        e = set_max_smem((const void *)k_gemm<EPI_SWIGLU, true>, (int)kGemmSmem);
        if (e == cudaSuccess)
            e = launch_k(k_gemm<EPI_SWIGLU, true>, dim3(sms), dim3(kGemmThreads + kDequantThreads), kGemmSmem, s,
                         m_ysel, m_wg, m_wu, g1);
    } else {
        e = set_max_smem((const void *)k_gemm<EPI_SWIGLU, false>, (int)kGemmSmem);
        if (e == cudaSuccess)
            e = launch_k(k_gemm<EPI_SWIGLU, false>, dim3(sms), dim3(kGemmThreads), kGemmSmem, s, m_ysel, m_wg, m_wu,
                         g1);
    }
    if (e != cudaSuccess) return SFFN_ERR_CUDA;

    GemmArgs g2 = {};
    g2.n_sel = n_sel;
    g2.sel_idx = sel_idx;
    g2.ysel = ysel;
    g2.out = static_cast<uint16_t *>(out);
    g2.L = L;
    g2.n_out = d;
    g2.tile_n = GMMA_N;
    g2.kblocks = (F + GBK - 1) / GBK;
    g2.group_m = 8;
    g2.err = err;
    g2.qw0 = static_cast<const uint8_t *>(w->w_downT);
    g2.qs0 = static_cast<const __half *>(w->s_downT);
    g2.qd = d;
    if (q) {
        e = set_max_smem((const void *)k_gemm<EPI_DOWN, true>, (int)kGemmSmem);
        if (e == cudaSuccess)
            e = launch_k(k_gemm<EPI_DOWN, true>, dim3(sms), dim3(kGemmThreads + kDequantThreads), kGemmSmem, s, m_h,
                         m_wd, m_wd, g2);
    } else {
        e = set_max_smem((const void *)k_gemm<EPI_DOWN, false>, (int)kGemmSmem);
        if (e == cudaSuccess)
            e = launch_k(k_gemm<EPI_DOWN, false>, dim3(sms), dim3(kGemmThreads), kGemmSmem, s, m_h, m_wd, m_wd, g2);
    }
    return e == cudaSuccess ? SFFN_OK : SFFN_ERR_CUDA;
}

}  // namespace sffn
