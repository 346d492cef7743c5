// predict.cu -- decode with a low-rank gate predictor (sm_103a).
//
// denseflux ("skipping most of a dense FFN", sec. 4.3, cheap predictors):
// exact gating reads all of W_gate, a third of the layer, and a predictor may
// skip most of that read; the best untrained predictor there is low-rank.  Read
// as: offline factors W_gate ~= A B (A [F, r], B [r, d], fp32, e.g. a rank-r
// truncated SVD), per token p = A (B x) + b_gate, candidates p_j >= -alpha
// (alpha = +inf: every neuron, the exact decode), the exact gate g_j only on the
// candidates, and the exact rule (active iff act(g_j) != 0) on them; a neuron
// that is not a candidate is skipped even when it would have been active.
//
//   k_lr_project  y = B x (fp32): one CTA per factor row, 16-byte loads, four
//                 in flight per thread, block reduction
//   k_lr_ffn      one CTA per gate chunk of R neurons: the chunk's rows of A
//                 are one contiguous block, streamed into shared memory by
//                 bulk copies (two pieces in flight, issued before the kernel
//                 waits for y, since A is an input); p_j = A_j . y + b_j per
//                 row (one warp per row), the candidates in ascending order;
//                 g_j = W_gate[j] . x + b_j on the candidates only and then
//                 u_j = W_up[j] . x on the active ones (one warp per two rows,
//                 both rows' 16-byte units in flight); the chunk's ascending
//                 list; and its partial output sum_j a_j u_j W_downT[j, :]
//                 (each thread owns fixed columns, four rows' loads in flight)
// then the decode's fixed-order reduction of the chunk partials, which also
// writes the token's list.  Bytes per token: 4 r (F + d) for the factors, the
// candidates' gate rows, and the active rows of W_up and W_downT.
#include <cmath>

#include "common.cuh"
#include "decode_finish.cuh"
#include "internal.h"
#include "wformat.cuh"

namespace sffn {

namespace {

constexpr int kLrThreads = 256;
constexpr int kLrMaxChunk = 256;  // R of the decode plan never exceeds this
constexpr int kLrPieceBytes = 48 * 1024;  // A's rows per bulk copy (at least one row)

// Four consecutive x elements (x in the weights' activation dtype) as fp32.
template <class W>
SFFN_DEV float4 load_x4(const void *x, int i4) {
    if constexpr (sizeof(typename W::X) == 4) {
        return __ldg(reinterpret_cast<const float4 *>(x) + i4);
    } else {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(x) + i4);
        return make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
    }
}

template <class W>
__global__ void __launch_bounds__(kLrThreads) k_lr_project(const float *fb, int d, const void *x, float *y) {
    __shared__ float red[kLrThreads / 32];
    griddep_wait();
    griddep_launch_dependents();
    const int k = blockIdx.x, n4 = d / 4;
    const float4 *row = reinterpret_cast<const float4 *>(fb + (size_t)k * d);
    constexpr int U = 4;
    float acc = 0.f;
    for (int i0 = threadIdx.x; i0 < n4; i0 += U * kLrThreads) {
        float4 bv[U], xv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * kLrThreads;
            bv[u] = i < n4 ? __ldg(row + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            xv[u] = i < n4 ? load_x4<W>(x, i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            acc = fmaf(bv[u].x, xv[u].x, acc);
            acc = fmaf(bv[u].y, xv[u].y, acc);
            acc = fmaf(bv[u].z, xv[u].z, acc);
            acc = fmaf(bv[u].w, xv[u].w, acc);
        }
    }
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < kLrThreads / 32; ++w) s += red[w];
        y[k] = s;
    }
}

// Dot products of x (fp32, shared memory) with rows ja and jb (jb < 0: none)
// of a stored [*, units] matrix, by one warp: both rows' units are loaded
// before any is used (16 per lane per row in flight).
template <class W>
SFFN_DEV void warp_dot2(const void *m, int units, const float *xs, int ja, int jb, float &sa, float &sb) {
    constexpr int U = 16;
    const int lane = threadIdx.x & 31;
    const uint4 *ra = reinterpret_cast<const uint4 *>(static_cast<const char *>(m) + (size_t)ja * units * 16);
    const uint4 *rb = reinterpret_cast<const uint4 *>(static_cast<const char *>(m) + (size_t)(jb < 0 ? ja : jb) * units * 16);
    float s0 = 0.f, s1 = 0.f;
    for (int u0 = 0; u0 < units; u0 += 32 * U) {
        uint4 va[U], vb[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + 32 * i + lane;
            va[i] = u < units ? ldg_stream(ra + u) : make_uint4(0, 0, 0, 0);
            vb[i] = (u < units && jb >= 0) ? ldg_stream(rb + u) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int u = u0 + 32 * i + lane;
            if (u < units) {
                float fa[W::E], fb[W::E];
                W::unpack(va[i], fa);
                W::unpack(vb[i], fb);
                const float *xp = xs + (size_t)u * W::E;
#pragma unroll
                for (int e = 0; e < W::E; ++e) {
                    s0 = fmaf(fa[e], xp[e], s0);
                    s1 = fmaf(fb[e], xp[e], s1);
                }
            }
        }
    }
    sa = warp_sum(s0);
    sb = warp_sum(s1);
}

struct LrArgs {
    const void *wg, *wu, *wdT;  // W_gate, W_up, W_downT [F, d]
    int32_t *err;       // the workspace's error word (a bulk copy that never lands)
    const float *bias;  // [F] or null
    const void *x;      // [d]
    const float *fa;    // A [F, r]
    const float *y;     // [r] = B x
    int d, F, R, r, act;
    int all;            // alpha = +inf: every neuron is a candidate (A and y unused)
    int piece_rows;     // > 0: rows of A per bulk-copy piece; 0: per-warp loads (rank % 4 != 0)
    float alpha;
    int *cnt, *lidx;    // [C], [C, R]: the chunk's active neurons, ascending
    float *part;        // [C, d]: the chunk's partial output
    unsigned *gbar;     // non-null: every chunk's CTA is resident; finish the call here
    void *out;
    int out_f32;
    int32_t *active_idx, *n_active;
};

constexpr int kLrMaxUnits = 4;  // 16-byte units of a W_downT row per thread (d_model <= 4096)

template <class W>
__global__ void __launch_bounds__(kLrThreads) k_lr_ffn(LrArgs a) {
    // dynamic: [2] mbarriers (128 bytes), xs [d] fp32, ys [r] fp32, then two
    // pieces of A of piece_rows * r floats each
    extern __shared__ __align__(128) unsigned char lsm_raw[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(lsm_raw);
    float *xs = reinterpret_cast<float *>(lsm_raw + 128), *ys = xs + a.d;
    float *abuf = ys + ((a.r + 3) & ~3);
    __shared__ int clist[kLrMaxChunk];
    __shared__ float gact[kLrMaxChunk];
    __shared__ uint8_t cflag[kLrMaxChunk];
    __shared__ int alist[kLrMaxChunk];
    __shared__ float hval[kLrMaxChunk];
    __shared__ int s_n, s_na;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = kLrThreads / 32;
    const int j0 = blockIdx.x * a.R, nrows = min(a.R, a.F - j0);
    const unsigned lt = (1u << lane) - 1u;
    const int pr = a.piece_rows;
    const bool bulk = !a.all && pr > 0;
    const int npieces = bulk ? (nrows + pr - 1) / pr : 0;
    const uint32_t row_bytes = (uint32_t)a.r * 4u;
    auto issue = [&](int k) {  // piece k of the chunk's rows of A into buffer k & 1
        const int r0 = k * pr, nr = min(pr, nrows - r0);
        mbar_arrive_expect_tx(&bar[k & 1], (uint32_t)nr * row_bytes);
        bulk_load(abuf + (size_t)(k & 1) * pr * a.r, a.fa + (size_t)(j0 + r0) * a.r, (uint32_t)nr * row_bytes,
                  &bar[k & 1], l2_evict_first_policy());
    };
    if (bulk && tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_fence_init();
        // A is an input of the call: stream it before waiting for y
        for (int k = 0; k < min(2, npieces); ++k) issue(k);
    }
    // x may be the previous call's output: with the projection kernel in front
    // (which waited for that call) it can be read now; otherwise only after the wait
    if (!a.all) stage_x<W>(xs, a.x, 1, 1, a.d);
    griddep_wait();
    griddep_launch_dependents();
    if (a.all) stage_x<W>(xs, a.x, 1, 1, a.d);
    const unsigned bar_base = a.gbar ? *reinterpret_cast<volatile unsigned *>(a.gbar + 1) : 0u;

    // ---- predicted pre-activations and candidates
    if (a.all) {
        for (int i = tid; i < nrows; i += kLrThreads) cflag[i] = 1;
    } else {
        for (int k = tid; k < a.r; k += kLrThreads) ys[k] = a.y[k];
        __syncthreads();
        auto decide = [&](int i, float dot) {
            const float pj = dot + (a.bias ? a.bias[j0 + i] : 0.f);
            cflag[i] = pj >= -a.alpha ? 1 : 0;
        };
        if (bulk) {
            bool ok = true;
            for (int k = 0; k < npieces; ++k) {
                ok = ok && mbar_wait(&bar[k & 1], (uint32_t)(k >> 1) & 1u);
                if (ok) {
                    const float *ab = abuf + (size_t)(k & 1) * pr * a.r;
                    const int r0 = k * pr, nr = min(pr, nrows - r0);
                    for (int i = warp; i < nr; i += nwarps) {
                        const float *arow = ab + (size_t)i * a.r;
                        float sdot = 0.f;
                        for (int q = lane; q < a.r; q += 32) sdot = fmaf(arow[q], ys[q], sdot);
                        sdot = warp_sum(sdot);
                        if (lane == 0) decide(r0 + i, sdot);
                    }
                }
                __syncthreads();  // buffer k & 1 is free again
                if (tid == 0 && ok && k + 2 < npieces) {
                    fence_proxy_async_smem();
                    issue(k + 2);
                }
            }
            if (!ok) {
                // a copy that never landed: report it, let the copies in flight
                // finish (bounded), and leave this chunk without candidates
                if (tid == 0) {
                    record_error(a.err, SFFN_ERR_TIMEOUT);
                    for (int k = 0; k < npieces; ++k) mbar_wait(&bar[k & 1], (uint32_t)(k >> 1) & 1u);
                }
                for (int i = tid; i < nrows; i += kLrThreads) cflag[i] = 0;
            }
        } else {
            for (int i = warp; i < nrows; i += nwarps) {
                const float *arow = a.fa + (size_t)(j0 + i) * a.r;
                float sdot = 0.f;
                for (int k0 = 0; k0 < a.r; k0 += 128) {
                    float av[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int k = k0 + 32 * q + lane;
                        av[q] = k < a.r ? __ldg(arow + k) : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int k = k0 + 32 * q + lane;
                        if (k < a.r) sdot = fmaf(av[q], ys[k], sdot);
                    }
                }
                sdot = warp_sum(sdot);
                if (lane == 0) decide(i, sdot);
            }
        }
    }
    __syncthreads();
    if (warp == 0) {  // candidates, ascending
        int n = 0;
        for (int b0 = 0; b0 < nrows; b0 += 32) {
            const int i = b0 + lane;
            const bool f = i < nrows && cflag[i];
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            if (f) clist[n + __popc(bal & lt)] = j0 + i;
            n += __popc(bal);
        }
        if (lane == 0) s_n = n;
    }
    __syncthreads();
    const int ncand = s_n;

    // ---- the exact gate on the candidates only
    const int units = a.d / W::E;  // 16-byte units per stored row
    for (int q = 2 * warp; q < ncand; q += 2 * nwarps) {
        float ga, gb;
        const int jb = q + 1 < ncand ? clist[q + 1] : -1;
        warp_dot2<W>(a.wg, units, xs, clist[q], jb, ga, gb);
        if (lane == 0) {
            gact[q] = act_fn(a.act, ga + (a.bias ? a.bias[clist[q]] : 0.f));
            if (jb >= 0) gact[q + 1] = act_fn(a.act, gb + (a.bias ? a.bias[jb] : 0.f));
        }
    }
    __syncthreads();
    if (warp == 0) {  // the chunk's active neurons, ascending
        int n = 0;
        for (int b0 = 0; b0 < ncand; b0 += 32) {
            const int q = b0 + lane;
            const float av = q < ncand ? gact[q] : 0.f;
            const bool on = q < ncand && av != 0.f;
            const unsigned bal = __ballot_sync(0xffffffffu, on);
            if (on) {
                const int m = n + __popc(bal & lt);
                alist[m] = clist[q];
                hval[m] = av;
                a.lidx[(size_t)blockIdx.x * a.R + m] = clist[q];
            }
            n += __popc(bal);
        }
        if (lane == 0) {
            s_na = n;
            a.cnt[blockIdx.x] = n;
        }
    }
    __syncthreads();
    const int nact = s_na;

    // ---- up rows of the active neurons: h_j = a_j * u_j
    for (int q = 2 * warp; q < nact; q += 2 * nwarps) {
        float ua, ub;
        const int jb = q + 1 < nact ? alist[q + 1] : -1;
        warp_dot2<W>(a.wu, units, xs, alist[q], jb, ua, ub);
        if (lane == 0) {
            hval[q] *= ua;
            if (jb >= 0) hval[q + 1] *= ub;
        }
    }
    __syncthreads();

    // ---- the chunk's partial output: sum over its active j of h_j W_downT[j, :]
    float acc[kLrMaxUnits][W::E];
#pragma unroll
    for (int k = 0; k < kLrMaxUnits; ++k)
#pragma unroll
        for (int e = 0; e < W::E; ++e) acc[k][e] = 0.f;
    constexpr int RB = 4;  // rows in flight
    for (int q0 = 0; q0 < nact; q0 += RB) {
        uint4 v[RB][kLrMaxUnits];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const uint4 *row = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.wdT) +
                                                               (size_t)(q0 + r < nact ? alist[q0 + r] : 0) * units * 16);
#pragma unroll
            for (int k = 0; k < kLrMaxUnits; ++k) {
                const int u = tid + k * kLrThreads;
                v[r][k] = (q0 + r < nact && u < units) ? ldg_stream(row + u) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const float h = q0 + r < nact ? hval[q0 + r] : 0.f;
#pragma unroll
            for (int k = 0; k < kLrMaxUnits; ++k) {
                float f[W::E];
                W::unpack(v[r][k], f);
#pragma unroll
                for (int e = 0; e < W::E; ++e) acc[k][e] = fmaf(h, f[e], acc[k][e]);
            }
        }
    }
    float *dst = a.part + (size_t)blockIdx.x * a.d;
#pragma unroll
    for (int k = 0; k < kLrMaxUnits; ++k) {
        const int u = tid + k * kLrThreads;
        if (u < units) {
            float4 *d4 = reinterpret_cast<float4 *>(dst + (size_t)u * W::E);
#pragma unroll
            for (int e = 0; e < W::E; e += 4) d4[e / 4] = make_float4(acc[k][e], acc[k][e + 1], acc[k][e + 2], acc[k][e + 3]);
        }
    }
    if (a.gbar) {
        // the grid barrier, the fixed-order sum of the chunks' partials and the
        // token's list (decode_finish.cuh), as the gate kernel ends an exact call
        FinishArgs fa = {};
        fa.gbar = a.gbar;
        fa.part = a.part;
        fa.nb = 1;
        fa.d = a.d;
        fa.F = a.F;
        fa.C = gridDim.x;
        fa.R = a.R;
        fa.cnt = a.cnt;
        fa.lidx = a.lidx;
        fa.out = a.out;
        fa.out_f32 = a.out_f32;
        fa.active_idx = a.active_idx;
        fa.n_active = a.n_active;
        fa.err = a.err;
        finish_call(fa, bar_base, false);
    }
}

template <class W>
cudaError_t predicted_t(const DecodeCall &c, const DecodePlan &p, const float *fa, const float *fb, int rank,
                        float alpha, cudaStream_t s) {
    char *ws = static_cast<char *>(c.ws);
    float *y = reinterpret_cast<float *>(ws + p.off_score);  // [rank] (rank <= F)
    const bool all = std::isinf(alpha);
    cudaError_t e = cudaSuccess;
    if (!all) e = launch_k(k_lr_project<W>, dim3(rank), dim3(kLrThreads), 0, s, fb, p.d, c.x, y);
    if (e != cudaSuccess) return e;
    LrArgs la = {};
    la.wg = c.w->w_gate;
    la.wu = c.w->w_up;
    la.wdT = c.w->w_downT;
    la.err = reinterpret_cast<int32_t *>(ws + p.off_err);
    la.bias = c.w->b_gate;
    la.x = c.x;
    la.fa = fa;
    la.y = y;
    la.d = p.d;
    la.F = p.F;
    la.R = p.R;
    la.r = all ? 0 : rank;
    la.act = c.w->act;
    la.all = all ? 1 : 0;
    la.alpha = all ? 0.f : alpha;
    la.cnt = reinterpret_cast<int *>(ws + p.off_cnt);
    la.lidx = reinterpret_cast<int *>(ws + p.off_lidx);
    la.part = reinterpret_cast<float *>(ws + p.off_part);
    // every chunk's CTA resident: the kernel finishes the call itself
    if (p.C <= device_sm_count()) {
        la.gbar = reinterpret_cast<unsigned *>(ws + p.off_err + kCtlBar);
        la.out = c.out;
        la.out_f32 = c.w->wdtype == SFFN_F32;
        la.active_idx = c.active_idx;
        la.n_active = c.n_active;
    }
    // A's rows stream in bulk pieces when every row starts on a 16-byte boundary
    const bool bulk = !all && rank % 4 == 0 && (reinterpret_cast<uintptr_t>(fa) & 15u) == 0;
    la.piece_rows = 0;
    if (bulk) {
        int pr = kLrPieceBytes / (4 * rank);
        la.piece_rows = pr < 1 ? 1 : (pr > p.R ? p.R : pr);
    }
    const size_t smem = 128 + sizeof(float) * ((size_t)p.d + (size_t)((la.r + 3) & ~3)) +
                        (bulk ? 2 * sizeof(float) * (size_t)la.piece_rows * rank : 0);
    e = set_max_smem((const void *)k_lr_ffn<W>, (int)smem);
    if (e == cudaSuccess) e = launch_k(k_lr_ffn<W>, dim3(p.C), dim3(kLrThreads), smem, s, la);
    return e;
}

}  // namespace

sffn_status run_decode_predicted(const DecodeCall &c, const DecodePlan &p, const float *factor_a,
                                 const float *factor_b, int rank, float alpha, cudaStream_t s) {
    if (p.R > kLrMaxChunk || p.d / 4 > kLrMaxUnits * kLrThreads) return SFFN_ERR_SHAPE;
    cudaError_t e;
    switch (c.w->wdtype) {
    case SFFN_F32: e = predicted_t<WF32>(c, p, factor_a, factor_b, rank, alpha, s); break;
    case SFFN_BF16: e = predicted_t<WBF16>(c, p, factor_a, factor_b, rank, alpha, s); break;
    default: return SFFN_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return SFFN_ERR_CUDA;
    if (p.C <= device_sm_count()) return SFFN_OK;  // k_lr_ffn finished the call
    return run_reduce_chunks(c, p, s);
}

}  // namespace sffn
