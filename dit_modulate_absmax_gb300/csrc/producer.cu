// producer.cu -- the two-pass NVFP4 activation producer for sm_103a.
//
// Pass 1 ("NVFP4 Modulation Producer Fusion", Dataflow, prototype step 1;
// "NVFP4 Streaming Design", Numerical Constraint items 1-2): re-derive the
// bf16 producer values y (AdaLN modulation, or BF16 SwiGLU for the FC2 input),
// reduce one exact global max |y| and turn it into the FP32 tensor scale.
//
// Pass 2 (prototype step 2; Numerical Constraint items 3-4): re-derive the same
// y, compute one E4M3 block scale per 16 values and the E2M1 codes, and write
// packed QDATA plus the scales directly in the GEMM's 128x4-atom scale layout.
//
// Both passes walk the activation in tiles of 128 rows x 256 columns.  Each
// thread owns one 16-value block (32 bytes) of a row, so half a warp covers a
// 512-byte row segment and every load is coalesced; the block maximum, the
// E4M3 scale and the reciprocal of the block's scale product are computed
// once per block, with no cross-lane traffic.  A pass-2 tile produces exactly
// four scale atoms (2 KB, contiguous in the scale layout), which are assembled
// in shared memory and written with 16-byte stores.  Pass 2 walks the tiles in
// the reverse of pass 1's order so that its first tiles are the ones pass 1
// read last, which are still resident in L2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "launch.h"
#include "ptx.cuh"

namespace h3fp4 {

// Device error bits of the producer kernels (read and cleared with the GEMM's by read_device_error).
__device__ uint32_t g_producer_error;
namespace {

// kSiluLut: uint16[65536], the correctly rounded bf16 silu of every bf16
// pattern (generated at build time); used where the FP32 evaluation below is
// too close to a bf16 rounding boundary, and for g < -16, |g| < 2^-100 and
// NaN (silu_needs_table).
#include "silu_lut.inc"

constexpr int kTileRows = 128;
constexpr int kTileCols = 256;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = 16;                          // values per thread and row = one scale block
constexpr int kRowsPerStep = 2 * kWarps;            // two rows per warp (one per half-warp)
constexpr int kSteps = kTileRows / kRowsPerStep;    // 8
constexpr int kUnroll = 2;                          // rows in flight per thread

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u)
{
    __nv_bfloat162 r;
    memcpy(&r, &u, 4);
    return r;
}

__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v)
{
    uint32_t r;
    memcpy(&r, &v, 4);
    return r;
}

// Correctly rounded bf16x2 multiply and add (no contraction into an FMA).
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) { return as_u32(__hmul2_rn(as_bf2(a), as_bf2(b))); }
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) { return as_u32(__hadd2_rn(as_bf2(a), as_bf2(b))); }

__device__ __forceinline__ uint4 ld16(const uint16_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Segment of row r and its row range [begin, end): s is the number of
// interior boundaries off[1..nseg-1] at or below r (offsets are
// non-decreasing), begin the largest of off[0..nseg-1] at or below r, end the
// smallest of off[1..nseg] above r.  Fully unrolled with constant indices so
// that the table stays in kernel-parameter space.
__device__ __forceinline__ int segment_of(const SegTable &t, int64_t r, int64_t &begin, int64_t &end)
{
    int s = 0;
    begin = 0;
    end = INT64_MAX;
#pragma unroll
    for (int i = 1; i <= H3FP4_MAX_SEGMENTS; ++i) {
        const int64_t v = t.off[i];
        const bool valid = i <= t.nseg;
        const bool interior = i < t.nseg;
        s += (interior && r >= v) ? 1 : 0;
        begin = (interior && r >= v && v > begin) ? v : begin;
        end = (valid && v > r && v < end) ? v : end;
    }
    return s;
}

// Exact value of an E4M3 code with the sign bit clear (bias 7, 3 mantissa bits).
__device__ __forceinline__ float e4m3_value(uint32_t c)
{
    // E4M3 -> f16 -> f32 with the hardware conversions: every E4M3 value
    // (subnormals down to 2^-9 included) is exact in f16 and in f32.
    float v;
    asm("{\n\t.reg .b16 c2;\n\t.reg .b32 h2;\n\t.reg .b16 lo, hi;\n\t"
        "cvt.u16.u32 c2, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 h2, c2;\n\t"
        "mov.b32 {lo, hi}, h2;\n\t"
        "cvt.f32.f16 %0, lo;\n\t}"
        : "=f"(v)
        : "r"(c & 0xFFu));
    return v;
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Correctly rounded bf16 silu(g) = g / (1 + e^-g) for the two bf16 halves of
// a word, in FP32 with packed two-lane arithmetic: s = g * rcp(1 + 2^(g *
// -log2 e)).
//  - g >= -16: the rounded exponent argument costs at most 0.7 * 23.1 *
//    2^-23 < 2^-19 relative while e^-g is not negligible (|argument| <= 23.1
//    for g in [-16, 16]; beyond, e^-g shrinks faster than the argument grows),
//    the hardware exp2 and reciprocal approximations about 2^-22 each, the add
//    and multiply 2^-24 each: |s - silu(g)| < 2^-18.5 |s| in all (for large g
//    the exponent underflows to 0 and s = g exactly).  In ulps of s that is
//    below 2^5.5, so RN_bf16(s) is the correctly rounded silu unless s lies
//    within 128 ulps of a bf16 rounding midpoint (the low 16 bits of s within
//    0x7F80 .. 0x807F); those values go to the table.
//  - g < -16, |g| < 2^-100 (where s can leave the normal range) and NaN: the
//    build-time table of correctly rounded values decides.
// Returns both FP32-path results; bit 0 / bit 1 of `bad` flags the low / high
// half for the table.
__device__ __forceinline__ bool silu_needs_table(float g, float s)
{
    return (((__float_as_uint(s) - 0x7F80u) & 0xFFFFu) < 0x100u) || !(g >= -16.0f) || !(fabsf(g) >= 0x1p-100f);
}

__device__ __forceinline__ uint32_t silu2_fast(uint32_t gw, uint32_t &bad)
{
    const float2 g = make_float2(__uint_as_float(gw << 16), __uint_as_float(gw & 0xFFFF0000u));
    const float2 a = __fmul2_rn(g, make_float2(-0x1.715476p+0f, -0x1.715476p+0f));
    const float2 d = __fadd2_rn(make_float2(ex2_approx(a.x), ex2_approx(a.y)), make_float2(1.0f, 1.0f));
    const float2 sv = __fmul2_rn(g, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
    bad = (silu_needs_table(g.x, sv.x) ? 1u : 0u) | (silu_needs_table(g.y, sv.y) ? 2u : 0u);
    return as_u32(__floats2bfloat162_rn(sv.x, sv.y));
}

// ---------------------------------------------------------------------------
// Sources of the producer values y, 8 consecutive bf16 per lane and row.
// ---------------------------------------------------------------------------
struct Vec16 {
    uint4 lo, hi;
};

__device__ __forceinline__ Vec16 ld32(const uint16_t *p)
{
    return Vec16{ld16(p), ld16(p + 8)};
}

__device__ __forceinline__ void words(const Vec16 &v, uint32_t (&w)[8])
{
    w[0] = v.lo.x; w[1] = v.lo.y; w[2] = v.lo.z; w[3] = v.lo.w;
    w[4] = v.hi.x; w[5] = v.hi.y; w[6] = v.hi.z; w[7] = v.hi.w;
}

struct ModulateSrc {
    static constexpr bool kModulated = true;
    static constexpr int kPass1Unroll = 4;   // rows in flight per thread in pass 1
    const uint16_t *x;
    int64_t ldx;
    const uint16_t *shift;
    const uint16_t *scale;
    int64_t ld_mod;
    SegTable seg;

    using Raw = Vec16;

    // The CTA's copy of the modulation parameters for the current tile's 256
    // columns: s1 = RN_bf16(scale + 1) and shift of every segment that the
    // tile's rows touch, as [segment][column half of a 16-column block][block]
    // (4 words each), and the segment of each of the tile's rows.  (Each
    // thread keeping its 16 parameter words and its segment's row range in
    // registers instead cost ~60 instructions per 16-value block of the pack
    // under the 64-register budget of 4 CTAs per SM.)
    struct Smem {
        uint4 s1[H3FP4_MAX_SEGMENTS][2][kTileCols / kBlock];
        uint4 sh[H3FP4_MAX_SEGMENTS][2][kTileCols / kBlock];
        int32_t row_seg[kTileRows];
    };

    // Every thread of the CTA calls this for a tile whose first row row0 < m
    // and first column c0; it begins and ends with a barrier.
    __device__ __forceinline__ void stage(Smem &sm, int64_t row0, int64_t m, int c0) const
    {
        __syncthreads();   // the previous tile's readers are done with sm
        if (threadIdx.x < kTileRows) {
            // rows past m are never modulated; they take row m-1's segment
            const int64_t r = min(row0 + static_cast<int64_t>(threadIdx.x), m - 1);
            int64_t b, e;
            sm.row_seg[threadIdx.x] = segment_of(seg, r, b, e);
        }
        __syncthreads();
        const int first = sm.row_seg[0], count = sm.row_seg[kTileRows - 1] - first + 1;   // monotone in r
        for (int i = threadIdx.x; i < 64 * count; i += kThreads) {
            const int sg = first + (i >> 6), k = i & 63, chunk = k & 31;   // columns c0 + 8 chunk .. + 7
            if (k < 32) {
                uint4 v = ld16(scale + sg * ld_mod + c0 + 8 * chunk);
                const uint32_t one2 = 0x3F803F80u;   // bf16 1.0 in both halves
                v = make_uint4(bf2_add(v.x, one2), bf2_add(v.y, one2), bf2_add(v.z, one2), bf2_add(v.w, one2));
                sm.s1[sg][chunk & 1][chunk >> 1] = v;
            } else {
                sm.sh[sg][chunk & 1][chunk >> 1] = ld16(shift + sg * ld_mod + c0 + 8 * chunk);
            }
        }
        __syncthreads();
    }
    __device__ __forceinline__ Raw load(int64_t r, int col) const { return ld32(x + r * ldx + col); }

    // y = RN_bf16(RN_bf16(x * RN_bf16(scale + 1)) + shift) for the tile's row rr
    // (segment from the table) and 16-column block blk.
    __device__ __forceinline__ void apply(const Smem &sm, int rr, int blk, const Raw &raw, uint32_t (&y)[8]) const
    {
        const int sg = sm.row_seg[rr];
        const uint4 a0 = sm.s1[sg][0][blk], a1 = sm.s1[sg][1][blk];
        const uint4 b0 = sm.sh[sg][0][blk], b1 = sm.sh[sg][1][blk];
        const uint32_t s1[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t sh[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        uint32_t xw[8];
        words(raw, xw);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            y[i] = bf2_add(bf2_mul(xw[i], s1[i]), sh[i]);
    }
    __device__ __forceinline__ void keep(int64_t, int, const uint32_t (&)[8]) const {}
};

struct SwigluSrc {
    static constexpr bool kModulated = false;
    static constexpr int kPass1Unroll = 1;
    const uint16_t *g;
    int64_t ldg;
    const uint16_t *u;
    int64_t ldu;
    uint16_t *h;  // optional output of pass 1 (leading dimension ldh)
    int64_t ldh;

    struct Raw {
        Vec16 g, u;
    };
    struct Smem {};

    __device__ __forceinline__ void stage(Smem &, int64_t, int64_t, int) const {}
    __device__ __forceinline__ Raw load(int64_t r, int col) const
    {
        return Raw{ld32(g + r * ldg + col), ld32(u + r * ldu + col)};
    }

    // h = RN_bf16(silu_bf16(gate) * up).
    __device__ __forceinline__ void apply(const Smem &, int, int, const Raw &raw, uint32_t (&y)[8]) const
    {
        uint32_t gw[8], uw[8], sv[8];
        words(raw.g, gw);
        words(raw.u, uw);
        uint32_t unsure = 0;  // bit 2i / 2i+1: value needs the table
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t bad;
            sv[i] = silu2_fast(gw[i], bad);
            unsure |= bad << (2 * i);
        }
        while (unsure) {  // rare: each flagged value is looked up once
            const int e = __ffs(unsure) - 1;
            unsure &= unsure - 1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (e == 2 * i)
                    sv[i] = (sv[i] & 0xFFFF0000u) | kSiluLut[gw[i] & 0xFFFFu];
                if (e == 2 * i + 1)
                    sv[i] = (sv[i] & 0x0000FFFFu) | (static_cast<uint32_t>(kSiluLut[gw[i] >> 16]) << 16);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
            y[i] = bf2_mul(sv[i], uw[i]);
    }
    __device__ __forceinline__ void keep(int64_t r, int col, const uint32_t (&y)[8]) const
    {
        if (h) {
            uint4 *dst = reinterpret_cast<uint4 *>(h + r * ldh + col);
            dst[0] = make_uint4(y[0], y[1], y[2], y[3]);
            dst[1] = make_uint4(y[4], y[5], y[6], y[7]);
        }
    }
};

struct PlainSrc {  // already-materialised bf16 values (SwiGLU pass 2 with a workspace)
    static constexpr bool kModulated = false;
    static constexpr int kPass1Unroll = kUnroll;
    const uint16_t *h;
    int64_t ldh;

    using Raw = Vec16;
    struct Smem {};
    __device__ __forceinline__ void stage(Smem &, int64_t, int64_t, int) const {}
    __device__ __forceinline__ Raw load(int64_t r, int col) const { return ld32(h + r * ldh + col); }
    __device__ __forceinline__ void apply(const Smem &, int, int, const Raw &raw, uint32_t (&y)[8]) const
    {
        words(raw, y);
    }
    __device__ __forceinline__ void keep(int64_t, int, const uint32_t (&)[8]) const {}
};

// Resident CTAs per SM that a kernel reading values from Src is compiled for
// (the register budget), and rows in flight per thread in pass 1: more warps
// and more loads in flight hide more memory latency, until spills cost more
// than that gains.  Measured at 37,810 x 7,168 (L2 flushed; the modulation
// parameters staged in shared memory): modulation pass 1 at 4 CTAs per SM
// 0.100 ms with 4 rows in flight, 0.102 with 2, 0.110 at 5 CTAs with 2;
// modulation pass 2 (2 rows in flight) 0.131 ms at 5 CTAs per SM, 0.137 at
// 4, 0.143 at 3 with 4 rows; the SwiGLU and plain single-launch producers
// 3 -> 4 -> 5 per SM 0.806 -> 0.770 -> 0.747 ms and 0.251 -> 0.237 -> 0.232 ms
// (the SwiGLU producer at 4 and 6 per SM 0.734 and 0.752 ms against 0.722 at
// 5; with 1 row in flight in pass 1, whose two inputs fill the registers
// that a second row would need, 0.714 ms).
template <class Src>
constexpr int min_blocks()
{
    return Src::kModulated ? 4 : 5;
}
constexpr int kPackMinBlocks = 5;   // pass 2 alone (pack_kernel), every source

template <class Src>
constexpr int pass1_unroll()
{
    return Src::kPass1Unroll;
}

// Row tile and column tile of tile t (column tiles fastest).  A 32-bit
// division whenever t fits in 32 bits (every realistic shape); the 64-bit
// division it replaces cost several percent of the pack pass's instructions.
__device__ __forceinline__ void tile_rc(int64_t t, int col_tiles, int64_t &row_tile, int &col_tile)
{
    if (t <= 0xFFFFFFFFll) {
        const uint32_t u = static_cast<uint32_t>(t), c = static_cast<uint32_t>(col_tiles);
        const uint32_t q = u / c;
        row_tile = q;
        col_tile = static_cast<int>(u - q * c);
    } else {
        row_tile = t / col_tiles;
        col_tile = static_cast<int>(t - row_tile * col_tiles);
    }
}

// Bit pattern of max |y| over 16 bf16 values (two per word), with native
// bf16x2 max on the absolute values; a NaN anywhere gives a NaN pattern
// (above 0x7F80), which wins every later unsigned comparison.
__device__ __forceinline__ uint32_t absmax16(const uint32_t (&y)[8])
{
    // max.xorsign.abs: the magnitude of the result is max(|a|, |b|) (its sign
    // is the xor of the inputs' signs, masked off at the end); .NaN makes a
    // NaN input give a NaN.
    uint32_t v = y[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        asm("max.NaN.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(v) : "r"(y[i]));
    v &= 0x7FFF7FFFu;
    return max(v & 0xFFFFu, v >> 16);   // both non-negative patterns: integer order = value order, NaN above all
}

// ---------------------------------------------------------------------------
// Pass 1: global absmax and tensor scale.  Persistent grid; each CTA folds its
// maximum into scratch[0] with one atomicMax, and the last CTA to finish
// (counted in scratch[1]) converts the maximum into the tensor scale.
// ---------------------------------------------------------------------------
// Pass 1 over the tiles blockIdx.x, blockIdx.x + gridDim.x, ...: this thread's
// maximum |y| bit pattern (the values are also kept by Src, e.g. h).
template <class Src>
__device__ __forceinline__ uint32_t absmax_tiles(const Src &src, int64_t m, int col_tiles, int64_t n_tiles,
                                                typename Src::Smem &ssm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 15, half = lane >> 4;
    uint32_t vmax = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {   // the same count in every thread of the CTA
        int64_t row_tile;
        int col_tile;
        tile_rc(t, col_tiles, row_tile, col_tile);
        const int64_t row0 = row_tile * kTileRows;
        const int col = col_tile * kTileCols + sub * kBlock;
        src.stage(ssm, row0, m, col_tile * kTileCols);   // every tile here has rows below m
        constexpr int kU = pass1_unroll<Src>();
#pragma unroll 1
        for (int i0 = 0; i0 < kSteps; i0 += kU) {
            typename Src::Raw raw[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t r = row0 + kRowsPerStep * (i0 + u) + 2 * warp + half;
                if (r < m)
                    raw[u] = src.load(r, col);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int64_t r = row0 + kRowsPerStep * (i0 + u) + 2 * warp + half;
                if (r < m) {
                    uint32_t y[8];
                    src.apply(ssm, kRowsPerStep * (i0 + u) + 2 * warp + half, sub, raw[u], y);
                    src.keep(r, col, y);
                    vmax = max(vmax, absmax16(y));
                }
            }
        }
    }
    return vmax;
}

// The CTA's maximum of the threads' values (valid in thread 0).
__device__ __forceinline__ uint32_t cta_max(uint32_t vmax)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    vmax = __reduce_max_sync(0xFFFFFFFFu, vmax);
    __shared__ uint32_t wmax[kWarps];
    if (lane == 0)
        wmax[warp] = vmax;
    __syncthreads();
    uint32_t mx = 0;
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            mx = max(mx, wmax[w]);
    }
    return mx;
}

// ts = RN_f32(amax / (6 * 448)); a NaN maximum (pattern above 0x7F80) stays NaN.
__device__ __forceinline__ float tensor_scale_of(uint32_t amax_bits)
{
    return __fdiv_rn(__uint_as_float(amax_bits << 16), 2688.0f);
}

template <class Src>
__global__ void __launch_bounds__(kThreads, min_blocks<Src>()) absmax_kernel(Src src, int64_t m, int col_tiles, int64_t n_tiles,
                                                          uint32_t *scratch, float *ts_out)
{
    __shared__ typename Src::Smem ssm;
    const uint32_t mx = cta_max(absmax_tiles(src, m, col_tiles, n_tiles, ssm));
    if (threadIdx.x == 0) {
        atomicMax(&scratch[0], mx);
        __threadfence();
        const uint32_t done = atomicAdd(&scratch[1], 1u);
        if (done == gridDim.x - 1) {
            __threadfence();
            *ts_out = tensor_scale_of(atomicOr(&scratch[0], 0u));
        }
    }
}

// Correctly rounded quotient a / b from the correctly rounded reciprocal
// rb = RN(1/b), with no division: q = RN(a rb) is within about one ulp of
// a/b, the residual q b - a is then exactly representable and one fused
// multiply-add computes it, and RN(q - (q b - a) rb) is RN(a / b) (the
// residual correction of Markstein's division, IBM J. Res. Dev. 34(1), 1990).
// Checked exhaustively on the host for every bf16 significand of a, every
// f32 significand of b and quotients in [2^-5, 2^5) (9.7e9 cases, both signs,
// IEEE single arithmetic): no difference from the IEEE quotient.  Power-of-two
// scaling carries that to every exponent at which the residual keeps its
// bits: a in the bf16 range and b in [2^-100, 2^100] for the quotients that
// matter here (>= 2^-11); smaller quotients still come out within a few ulps,
// which is all their E4M3 or E2M1 code depends on.  The residual is formed as
// q b - a (not a - q b) so that a = -0 gives q = -0 and the result stays -0.
__device__ __forceinline__ float div_rn_by_rcp(float a, float b, float rb)
{
    const float q = __fmul_rn(a, rb);
    return __fmaf_rn(-__fmaf_rn(q, b, -a), rb, q);
}

__device__ __forceinline__ float2 div2_rn_by_rcp(float2 a, float2 b, float2 rb)
{
    const float2 q = __fmul2_rn(a, rb);
    const float2 e = __ffma2_rn(q, b, make_float2(-a.x, -a.y));
    return __ffma2_rn(make_float2(-e.x, -e.y), rb, q);
}

// Block scale bs = E4M3_RNE_sat(RN_f32(bamax / den)).  With den in
// [2^-88, 2^100] (`den_fma`, a property of the tensor scale alone) the quotient
// comes from rden = RN(1/den) by the residual correction; block maxima below
// 2^-100 then give quotients below 2^-12, whose code is 0 however they round.
// Other dens (tensors whose absolute maximum is below ~2^-80 or above ~2^108,
// zero, or not finite) take the IEEE division.  A block maximum is NaN when
// the block holds a NaN (absmax16), and then so is the tensor scale.
__device__ __forceinline__ uint32_t block_scale(uint32_t bmax_bits, float den, float rden, bool den_fma)
{
    const float b = __uint_as_float(bmax_bits << 16);
    if (den_fma)
        return cvt_e4m3(div_rn_by_rcp(b, den, rden));
    if (bmax_bits == 0)
        return 0u;  // an all-zero block gets scale 0
    const float q = __fdiv_rn(b, den);
    return q != q ? 0x7Fu : cvt_e4m3(q);   // a NaN quotient (NaN or infinite ts) is the E4M3 NaN code
}

// E2M1 codes of a 16-value block with the block's FP32 scale product sc;
// byte i holds element 2i in its low nibble.  A zero or NaN scale product
// (sc is never negative) gives zeros with y's signs.
//
// The code of y is E2M1_RNE_sat(RN_f32(y / sc)).  For sc in [2^-100, 2^100]
// the quotients come from r = RN(1/sc) (one correctly rounded reciprocal per
// block) by the residual correction above, two values at a time with packed
// two-lane multiplies and fused multiply-adds, and are converted four pairs
// per instruction group; RN_f32(y / sc) is then exact, so no value needs a
// second look.  Blocks whose sc lies outside that range (tensors with extreme
// scales) divide each value by the IEEE division.  The sign of y (also of
// y = -0) carries through into the code.
__device__ __forceinline__ uint2 encode16(const uint32_t (&y)[8], float sc)
{
    if (!(sc > 0.0f)) {
        uint32_t signs[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i)
            signs[i >> 2] |= (((y[i] >> 12) & 0x8u) | ((y[i] >> 24) & 0x80u)) << (8 * (i & 3));
        return make_uint2(signs[0], signs[1]);
    }
    uint32_t out[2];
    if (sc >= 0x1p-100f && sc <= 0x1p100f) {
        const float r = __frcp_rn(sc);
        const float2 r2 = make_float2(r, r), s2 = make_float2(sc, sc);
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {   // 8 values (4 words) at a time
            float2 q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = y[4 * hlf + i];
                q[i] = div2_rn_by_rcp(make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)), s2, r2);
            }
            out[hlf] = cvt_e2m1x8(q[0], q[1], q[2], q[3]);
        }
    } else {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
            uint32_t lo = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w = y[4 * hlf + i];
                lo |= cvt_e2m1x2(__fdiv_rn(__uint_as_float(w & 0xFFFF0000u), sc), __fdiv_rn(__uint_as_float(w << 16), sc))
                      << (8 * i);
            }
            out[hlf] = lo;
        }
    }
    return make_uint2(out[0], out[1]);
}

// ---------------------------------------------------------------------------
// Pass 2: one CTA per 128 x 256 tile (tiles visited in reverse order).
// ---------------------------------------------------------------------------
// Pass 2 of output tile t (128 rows x 256 columns): QDATA and the tile's four
// scale atoms, assembled in the CTA's 2 KB `sft` and written with 16-byte stores.
template <class Src>
__device__ __forceinline__ void pack_tile(const Src &src, int64_t t, int64_t m, int64_t m_pad, int64_t d,
                                          int col_tiles, float ts, float den, float rden, bool den_fma,
                                          uint8_t *qdata, uint8_t *sf, uint8_t *sft, typename Src::Smem &ssm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane & 15, half = lane >> 4;
    int64_t row_tile;
    int col_tile;
    tile_rc(t, col_tiles, row_tile, col_tile);
    const int64_t row0 = row_tile * kTileRows;
    const int col = col_tile * kTileCols + sub * kBlock;
    const int64_t qld = d / 2;
    if (row0 < m)   // the same in every thread of the CTA
        src.stage(ssm, row0, m, col_tile * kTileCols);

#pragma unroll 1
    for (int i0 = 0; i0 < kSteps; i0 += kUnroll) {
        typename Src::Raw raw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = row0 + kRowsPerStep * (i0 + u) + 2 * warp + half;
            if (r < m)
                raw[u] = src.load(r, col);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int rr = kRowsPerStep * (i0 + u) + 2 * warp + half;
            const int64_t r = row0 + rr;
            uint32_t y[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (r < m)
                src.apply(ssm, rr, sub, raw[u], y);
            // bs = E4M3_RNE_sat(RN_f32(block_amax / RN_f32(6 ts))); an all-zero block gets 0.
            const uint32_t bs = block_scale(absmax16(y), den, rden, den_fma);
            const float sc = __fmul_rn(e4m3_value(bs), ts);
            const uint2 packed = encode16(y, sc);
            if (r < m_pad)
                *reinterpret_cast<uint2 *>(qdata + r * qld + col / 2) = packed;
            sft[(sub >> 2) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (sub & 3)] = static_cast<uint8_t>(bs);
        }
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int64_t atoms_per_row_tile = d / 64;
        uint8_t *dst = sf + (row_tile * atoms_per_row_tile + col_tile * 4) * 512;
        reinterpret_cast<uint4 *>(dst)[threadIdx.x] = reinterpret_cast<const uint4 *>(sft)[threadIdx.x];
    }
}

struct PackConsts {
    float ts, den, rden;
    bool den_fma;
};

__device__ __forceinline__ PackConsts pack_consts(float ts)
{
    PackConsts c;
    c.ts = ts;
    c.den = __fmul_rn(6.0f, ts);
    c.den_fma = c.den >= 0x1p-88f && c.den <= 0x1p100f;
    c.rden = c.den_fma ? __frcp_rn(c.den) : 0.0f;
    return c;
}

// ---------------------------------------------------------------------------
// Pass 2: one CTA per 128 x 256 tile (tiles visited in reverse order).
// ---------------------------------------------------------------------------
template <class Src>
__global__ void __launch_bounds__(kThreads, kPackMinBlocks) pack_kernel(Src src, int64_t m, int64_t m_pad, int64_t d, int col_tiles,
                                                        int64_t n_tiles, const float *ts_ptr, uint8_t *qdata,
                                                        uint8_t *sf)
{
    __shared__ __align__(16) uint8_t sft[4 * 512];
    __shared__ typename Src::Smem ssm;
    const PackConsts c = pack_consts(*ts_ptr);
    pack_tile(src, n_tiles - 1 - blockIdx.x, m, m_pad, d, col_tiles, c.ts, c.den, c.rden, c.den_fma, qdata, sf,
              sft, ssm);
}

// ---------------------------------------------------------------------------
// Both passes in one cooperative launch ("NVFP4 Streaming Design", P2 "next":
// a single-launch cooperative producer, pass 1 and pass 2 around a grid
// barrier with a bounded wait).  Every CTA of the (co-resident) grid reduces
// its pass-1 tiles, adds its maximum to scratch[0] and arrives on scratch[1];
// it then waits until all gridDim.x CTAs have arrived (giving up after 2 s
// with a device error instead of hanging), derives ts from the global maximum
// itself and claims pass-2 tiles from a shared counter in reverse order, so
// that the first tiles packed are the ones pass 1 read last, still in L2, and
// no CTA waits at the end on a fixed share of slow (fallback-heavy) tiles.
// `extra_arrivals` (0 in every product call) raises the barrier's arrival
// target above the grid size and `wait_ns` sets its limit: the
// failure-detection entry point uses them to make the wait give up.
// ---------------------------------------------------------------------------
constexpr uint64_t kGridWaitLimitNs = 2000000000ull;
constexpr uint32_t ERR_GRID_WAIT = 1u << 8;   // the cooperative producer's grid barrier timed out

template <class Src1, class Src2>
__global__ void __launch_bounds__(kThreads, min_blocks<Src1>())
    producer_coop_kernel(Src1 src1, Src2 src2, int64_t m, int64_t m_pad, int64_t d, int col_tiles,
                         int64_t n_tiles1, int64_t n_tiles2, uint32_t *scratch, float *ts_out, uint8_t *qdata,
                         uint8_t *sf, uint32_t extra_arrivals, uint64_t wait_ns)
{
    __shared__ __align__(16) uint8_t sft[4 * 512];
    __shared__ float ts_sh;
    __shared__ int ok_sh;
    __shared__ uint32_t claim_sh[2];
    __shared__ union {   // pass 1's parameter copy, then pass 2's (a barrier lies between)
        typename Src1::Smem p1;
        typename Src2::Smem p2;
    } ssm;
    const uint32_t mx = cta_max(absmax_tiles(src1, m, col_tiles, n_tiles1, ssm.p1));
    if (threadIdx.x == 0) {
        atomicMax(&scratch[0], mx);
        __threadfence();
        atomicAdd(&scratch[1], 1u);
        // grid barrier: every CTA's maximum is in scratch[0] once all have arrived
        bool ok = true;
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            uint32_t arrived;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(arrived) : "l"(scratch + 1) : "memory");
            if (arrived >= gridDim.x + extra_arrivals)
                break;
            if (globaltimer_ns() - t0 > wait_ns) {
                ok = false;
                atomicOr(&g_producer_error, ERR_GRID_WAIT);
                break;
            }
            __nanosleep(256);
        }
        const float ts = tensor_scale_of(atomicOr(&scratch[0], 0u));
        if (ok && blockIdx.x == 0)
            *ts_out = ts;
        ts_sh = ts;
        ok_sh = ok ? 1 : 0;
    }
    __syncthreads();
    if (!ok_sh)
        return;
    // Pass 2 hands tiles out dynamically: past the barrier scratch[1] only
    // grows from gridDim.x, so each atomicAdd on it claims the next tile
    // (claim - gridDim.x, counted from the end).  Thread 0 claims one tile
    // ahead into the other slot of claim_sh while the CTA packs the current one.
    const PackConsts c = pack_consts(ts_sh);
    int slot = 0;
    if (threadIdx.x == 0)
        claim_sh[0] = atomicAdd(&scratch[1], 1u) - gridDim.x;
    __syncthreads();
    while (true) {
        const uint32_t idx = claim_sh[slot];
        if (idx >= n_tiles2)
            break;
        if (threadIdx.x == 0)
            claim_sh[slot ^ 1] = atomicAdd(&scratch[1], 1u) - gridDim.x;
        pack_tile(src2, n_tiles2 - 1 - static_cast<int64_t>(idx), m, m_pad, d, col_tiles, c.ts, c.den, c.rden,
                  c.den_fma, qdata, sf, sft, ssm.p2);
        __syncthreads();   // sft and the claim slot just read are reused by the next tile
        slot ^= 1;
    }
}

// Logical [rows, cols] (leading dimension ld) -> 128x4-atom scale layout.
__global__ void swizzle_kernel(const uint8_t *src, int64_t rows, int64_t cols, int64_t ld, uint8_t *dst,
                               int64_t total)
{
    for (int64_t o = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t atom = o / 512, within = o % 512;
        const int64_t atoms_per_row_tile = cols / 4;
        const int64_t r = (atom / atoms_per_row_tile) * 128 + (within / 16) + ((within % 16) / 4) * 32;
        const int64_t c = (atom % atoms_per_row_tile) * 4 + (within % 4);
        dst[o] = r < rows ? src[r * ld + c] : 0;
    }
}

template <class Src>
cudaError_t run_absmax(const Src &src, int64_t m, int64_t d, float *ts, uint32_t *scratch, cudaStream_t st)
{
    if (m == 0)
        return cudaMemsetAsync(ts, 0, sizeof(float), st);
    cudaError_t e = cudaMemsetAsync(scratch, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess)
        return e;
    const int col_tiles = static_cast<int>(d / kTileCols);
    const int64_t n_tiles = ((m + kTileRows - 1) / kTileRows) * col_tiles;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    const int grid = static_cast<int>(n_tiles < cap ? n_tiles : cap);
    absmax_kernel<Src><<<grid, kThreads, 0, st>>>(src, m, col_tiles, n_tiles, scratch, ts);
    return cudaGetLastError();
}

// Both passes in one cooperative launch: a grid of co-resident CTAs (the
// occupancy-derived count, capped by the tile count) so that the in-kernel
// grid barrier cannot wait on a CTA that is not running.
template <class Src1, class Src2>
cudaError_t run_coop(const Src1 &src1, const Src2 &src2, int64_t m, int64_t m_pad, int64_t d, float *ts,
                     uint32_t *scratch, uint8_t *qdata, uint8_t *sf, cudaStream_t st, uint32_t extra_arrivals = 0,
                     uint64_t wait_ns = kGridWaitLimitNs)
{
    const int col_tiles = static_cast<int>(d / kTileCols);
    const int64_t n_tiles1 = ((m + kTileRows - 1) / kTileRows) * col_tiles;
    const int64_t n_tiles2 = ((m_pad + kTileRows - 1) / kTileRows) * col_tiles;
    if (n_tiles2 == 0)
        return m == 0 ? cudaMemsetAsync(ts, 0, sizeof(float), st) : cudaSuccess;
    cudaError_t e = cudaMemsetAsync(scratch, 0, 2 * sizeof(uint32_t), st);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, producer_coop_kernel<Src1, Src2>, kThreads, 0);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorCooperativeLaunchTooLarge;
    const int64_t resident = static_cast<int64_t>(per_sm) * sm_count();
    const int64_t want = n_tiles2 > n_tiles1 ? n_tiles2 : n_tiles1;
    const unsigned grid = static_cast<unsigned>(want < resident ? want : resident);
    if (n_tiles2 + 2ll * grid >= 0xFFFFFFFFll)   // the 32-bit arrival/claim counter must not wrap
        return cudaErrorInvalidValue;
    void *args[] = {const_cast<Src1 *>(&src1), const_cast<Src2 *>(&src2), &m, &m_pad, &d,
                    const_cast<int *>(&col_tiles), const_cast<int64_t *>(&n_tiles1), const_cast<int64_t *>(&n_tiles2),
                    &scratch, &ts, &qdata, &sf, &extra_arrivals, &wait_ns};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(producer_coop_kernel<Src1, Src2>), dim3(grid),
                                       dim3(kThreads), args, 0, st);
}

template <class Src>
cudaError_t run_pack(const Src &src, int64_t m, int64_t m_pad, int64_t d, const float *ts, uint8_t *qdata,
                     uint8_t *sf, cudaStream_t st)
{
    const int col_tiles = static_cast<int>(d / kTileCols);
    const int64_t row_tiles = (m_pad + kTileRows - 1) / kTileRows;
    const int64_t n_tiles = row_tiles * col_tiles;
    if (n_tiles == 0)
        return cudaSuccess;
    if (n_tiles > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    pack_kernel<Src><<<static_cast<unsigned>(n_tiles), kThreads, 0, st>>>(src, m, m_pad, d, col_tiles, n_tiles, ts,
                                                                           qdata, sf);
    return cudaGetLastError();
}

}  // namespace

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

cudaError_t launch_modulate_absmax(const uint16_t *x, int64_t ldx, int64_t m, int64_t d, const uint16_t *shift,
                                   const uint16_t *scale, int64_t ld_mod, const SegTable &seg, float *ts,
                                   uint32_t *scratch, cudaStream_t st)
{
    ModulateSrc src{x, ldx, shift, scale, ld_mod, seg};
    return run_absmax(src, m, d, ts, scratch, st);
}

cudaError_t launch_modulate_pack(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                 const uint16_t *shift, const uint16_t *scale, int64_t ld_mod, const SegTable &seg,
                                 const float *ts, uint8_t *qdata, uint8_t *sf, cudaStream_t st)
{
    ModulateSrc src{x, ldx, shift, scale, ld_mod, seg};
    return run_pack(src, m, m_pad, d, ts, qdata, sf, st);
}

cudaError_t launch_quantize_pack(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad, int64_t d, float *ts,
                                 uint32_t *scratch, uint8_t *qdata, uint8_t *sf, cudaStream_t st)
{
    PlainSrc src{x, ldx};
    return run_coop(src, src, m, m_pad, d, ts, scratch, qdata, sf, st);
}

cudaError_t launch_quantize_pack_barrier_timeout(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad,
                                                int64_t d, float *ts, uint32_t *scratch, uint8_t *qdata, uint8_t *sf,
                                                uint64_t wait_ns, cudaStream_t st)
{
    PlainSrc src{x, ldx};
    return run_coop(src, src, m, m_pad, d, ts, scratch, qdata, sf, st, 1u, wait_ns);
}

cudaError_t launch_modulate_produce(const uint16_t *x, int64_t ldx, int64_t m, int64_t m_pad, int64_t d,
                                    const uint16_t *shift, const uint16_t *scale, int64_t ld_mod, const SegTable &seg,
                                    float *ts, uint32_t *scratch, uint8_t *qdata, uint8_t *sf, cudaStream_t st)
{
    ModulateSrc src{x, ldx, shift, scale, ld_mod, seg};
    return run_coop(src, src, m, m_pad, d, ts, scratch, qdata, sf, st);
}

cudaError_t read_producer_error(uint32_t *code)
{
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_producer_error, sizeof(v));
    if (e != cudaSuccess)
        return e;
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_producer_error, &zero, sizeof(zero));
    *code = v;
    return e;
}

cudaError_t launch_swiglu_pack(const uint16_t *gate, int64_t ldg, const uint16_t *up, int64_t ldu, int64_t m,
                               int64_t m_pad, int64_t f, float *ts, uint32_t *scratch, uint8_t *qdata, uint8_t *sf,
                               uint16_t *h, cudaStream_t st)
{
    SwigluSrc src{gate, ldg, up, ldu, h, f};
    if (h != nullptr) {   // pass 1 keeps h, pass 2 packs it after the grid barrier
        PlainSrc plain{h, f};
        return run_coop(src, plain, m, m_pad, f, ts, scratch, qdata, sf, st);
    }
    SwigluSrc recompute{gate, ldg, up, ldu, nullptr, f};
    return run_coop(src, recompute, m, m_pad, f, ts, scratch, qdata, sf, st);
}

cudaError_t launch_swizzle_scales(const uint8_t *src, int64_t rows, int64_t cols, int64_t ld, uint8_t *dst,
                                  cudaStream_t st)
{
    const int64_t total = ((rows + 127) / 128) * 128 * cols;
    if (total == 0)
        return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
    swizzle_kernel<<<grid, 256, 0, st>>>(src, rows, cols, ld, dst, total);
    return cudaGetLastError();
}

}  // namespace h3fp4
