// wformat.cuh -- stored weight formats of the decode kernels and the staging
// of the activations in shared memory (sm_103a).
#pragma once
#include <type_traits>

#include "common.cuh"

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
    static constexpr bool Q = false;  // no group scales
    static SFFN_DEV float scale_at(const unsigned char *, uint32_t) { return 1.f; }
    static SFFN_DEV void dequant(const uint4 &v, float, float *f) { unpack(v, f); }
    // x elements matching weight unit u (x stored in its own dtype, 16-byte units)
    static SFFN_DEV void load_xu(const uint4 *xrow, uint32_t u, float *f) { unpack(xrow[u], f); }
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
    static constexpr bool Q = false;
    static SFFN_DEV float scale_at(const unsigned char *, uint32_t) { return 1.f; }
    static SFFN_DEV void dequant(const uint4 &v, float, float *f) { unpack(v, f); }
    static SFFN_DEV void load_xu(const uint4 *xrow, uint32_t u, float *f) { unpack(xrow[u], f); }
};

// Symmetric int4 with one fp16 scale per 64 consecutive elements of a stored
// row: a 16-byte unit holds 32 two's-complement codes (low nibble = even
// column) and lies in group u / 2.  code * scale is exact in fp32, and so is its
// product with a bf16 activation (at most 23 significant bits).
struct WINT4 {
    using X = __nv_bfloat16;
    static constexpr int E = 32;
    static constexpr bool Q = true;
    static SFFN_DEV float scale_at(const unsigned char *srow, uint32_t u) {
        return __half2float(*reinterpret_cast<const __half *>(srow + (u >> 1) * 2));
    }
    // nibble n (two's complement) -> n ^ 8 is the code + 8 as an unsigned value;
    // OR-ing it into the mantissa of 2^23 gives 2^23 + code + 8 exactly
    static SFFN_DEV void codes(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x ^ 0x88888888u, v.y ^ 0x88888888u, v.z ^ 0x88888888u, v.w ^ 0x88888888u};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int k = 0; k < 8; ++k)
                f[8 * q + k] = __uint_as_float(0x4B000000u | ((w[q] >> (4 * k)) & 0xFu)) - 8388616.0f;
    }
    static SFFN_DEV void dequant(const uint4 &v, float s, float *f) {
        codes(v, f);
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] *= s;
    }
    static SFFN_DEV void load_xu(const uint4 *xrow, uint32_t u, float *f) {
#pragma unroll
        for (int q = 0; q < 4; ++q) WBF16::unpack(xrow[4 * u + q], f + 8 * q);
    }
};

// Eight consecutive columns (col0 a multiple of 8) of a stored row, loaded
// raw: fp32 two 16-byte units, bf16 one, int4 one 32-bit word of 8 codes.
struct Row8 {
    uint4 v0, v1;
};

template <class W>
SFFN_DEV Row8 load_row8(const void *row, int col0) {
    const char *p = static_cast<const char *>(row);
    Row8 r{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if constexpr (W::E == 4) {
        r.v0 = ldg_stream(p + (size_t)col0 * 4);
        r.v1 = ldg_stream(p + (size_t)col0 * 4 + 16);
    } else if constexpr (W::E == 8) {
        r.v0 = ldg_stream(p + (size_t)col0 * 2);
    } else {
        r.v0.x = ldg_stream_u32(p + (size_t)col0 / 2);
    }
    return r;
}

// The row's group scale at col0 (int4: fp16 scales [d/64] per stored row), else 1.
template <class W>
SFFN_DEV float row_scale8(const void *scales, size_t row, int d, int col0) {
    if constexpr (W::Q) {
        const __half *sr = static_cast<const __half *>(scales) + row * (size_t)(d / 64);
        return __half2float(sr[col0 / 64]);
    } else {
        return 1.f;
    }
}

// The eight columns as fp32 (int4: code * scale, exact).
template <class W>
SFFN_DEV void unpack_row8(const Row8 &r, float s, float *f) {
    if constexpr (W::E == 4) {
        W::unpack(r.v0, f);
        W::unpack(r.v1, f + 4);
    } else if constexpr (W::E == 8) {
        W::unpack(r.v0, f);
    } else {
        const uint32_t w = r.v0.x ^ 0x88888888u;
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = (__uint_as_float(0x4B000000u | ((w >> (4 * k)) & 0xFu)) - 8388616.0f) * s;
    }
}

// The format of the activations that go with weights W (fp32 with fp32
// weights, else bf16).
template <class W>
using XFormat = typename std::conditional<sizeof(typename W::X) == 4, WF32, WBF16>::type;

// Copy the activations x [nb, d] into shared memory in their own dtype
// [NBpad, d] (rows >= nb zero), 128-bit units, four loads in flight per thread.
template <class W>
SFFN_DEV void stage_x_raw(void *xs, const void *x, int nb, int NBpad, int d) {
    constexpr int XE = 16 / (int)sizeof(typename W::X);
    const int per_row = d / XE;
    const int total = NBpad * per_row;
    uint4 *dst = static_cast<uint4 *>(xs);
    for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int u = base + k * blockDim.x;
            v[k] = (u < total && u / per_row < nb) ? ldg_v4(static_cast<const char *>(x) + (size_t)u * 16)
                                                   : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int u = base + k * blockDim.x;
            if (u < total) dst[u] = v[k];
        }
    }
}

// Stage the activations x [nb, d] into shared memory as fp32 [NBpad, d]
// (rows >= nb zero).  128-bit loads, four in flight per thread, so staging
// costs one memory round trip instead of one per element.
template <class W>
SFFN_DEV void stage_x(float *xs, const void *x, int nb, int NBpad, int d) {
    constexpr int XE = 16 / (int)sizeof(typename W::X);  // elements per 16-byte unit of x
    const int per_row = d / XE;
    const int total = NBpad * per_row;
    for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int u = base + k * blockDim.x;
            v[k] = (u < total && u / per_row < nb) ? ldg_v4(static_cast<const char *>(x) + (size_t)u * 16)
                                                   : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int u = base + k * blockDim.x;
            if (u < total) {
                float f[XE];
                XFormat<W>::unpack(v[k], f);
                float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)u * XE);
#pragma unroll
                for (int q = 0; q < XE / 4; ++q) dst[q] = make_float4(f[4 * q], f[4 * q + 1], f[4 * q + 2], f[4 * q + 3]);
            }
        }
    }
}

}  // namespace sffn
