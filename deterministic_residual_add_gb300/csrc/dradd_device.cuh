// dradd_device.cuh -- device helpers for the residual-add + RMSNorm kernels:
// bf16 widening and round-to-nearest-even narrowing, the canonical pairwise
// reduction pieces, and thin wrappers over the PTX for mbarriers and bulk
// asynchronous copies (TMA engine).
//
// Every floating-point step uses an explicit round-to-nearest intrinsic
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn) so that no multiply-add is
// ever contracted and each operation is exactly one IEEE fp32 rounding.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#ifndef DRADD_RNE_HW_CVT
#define DRADD_RNE_HW_CVT 1
#endif

namespace dradd {

// ------------------------------------------------------------ bf16 <-> fp32
// A bf16 value is the top half of an fp32 word, so widening is exact.  A
// 32-bit word holds two bf16 values, the lower-addressed element in the low
// half.
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// Round-half-even by integer arithmetic: adding 0x7FFF plus the lowest kept
// bit carries into the kept half exactly when the discarded half is above
// 0x8000, or equal to it with an odd kept half.  NaN keeps its sign and
// becomes the quiet NaN 0x7FC0.
__device__ __forceinline__ uint32_t rne_bits_int(float f)
{
    const uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return ((u >> 16) & 0x8000u) | 0x7FC0u;
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// The hardware conversion: cvt.rn.bf16x2.f32 rounds both operands to
// nearest-even (subnormals kept) and packs them, first operand in the high
// half.  Equal to rne_bits_int on every non-NaN input (checked exhaustively
// by the test suite); NaN becomes a NaN.
__device__ __forceinline__ uint32_t pack_rne_cvt(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t pack_rne_int(float lo, float hi)
{
    return rne_bits_int(lo) | (rne_bits_int(hi) << 16);
}

__device__ __forceinline__ uint32_t pack_rne(float lo, float hi)
{
#if DRADD_RNE_HW_CVT
    return pack_rne_cvt(lo, hi);
#else
    return pack_rne_int(lo, hi);
#endif
}

// ------------------------------------------------------- packed fp32 pairs
// Blackwell issues add, sub, mul and fma on two fp32 values per instruction
// (the .f32x2 forms); each lane is the IEEE operation rounded to nearest
// with subnormals kept, so the results equal the scalar forms' bit for bit
// (the parity tests hold every kernel to the oracle).  Half the
// floating-point instructions of the element-wise steps.  Never feed a
// packed multiply straight into a packed add: the pair can come out fused
// (see fold8_squares).
__device__ __forceinline__ void add2_rn(float a0, float a1, float b0, float b1, float& d0, float& d1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void sub2_rn(float a0, float a1, float b0, float b1, float& d0, float& d1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void mul2_rn(float a0, float a1, float b0, float b1, float& d0, float& d1)
{
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma2_rn(float a0, float a1, float b0, float b1, float c0, float c1, float& d0,
                                        float& d1)
{
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// 8 consecutive bf16 elements = one 16-byte vector.
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8])
{
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x);
    f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z);
    f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8_rne(const float (&f)[8])
{
    uint4 u;
    u.x = pack_rne(f[0], f[1]);
    u.y = pack_rne(f[2], f[3]);
    u.z = pack_rne(f[4], f[5]);
    u.w = pack_rne(f[6], f[7]);
    return u;
}

// acc = fp32(x) + fp32(residual), element by element.
__device__ __forceinline__ void add8(const uint4& xv, const uint4& rv, float (&acc)[8])
{
    float xf[8], rf[8];
    unpack8(xv, xf);
    unpack8(rv, rf);
#pragma unroll
    for (int e = 0; e < 8; e += 2)
        add2_rn(xf[e], xf[e + 1], rf[e], rf[e + 1], acc[e], acc[e + 1]);
}

// The lowest three levels of the pairwise tree: squares of one aligned
// 8-element block, summed as ((s0+s1)+(s2+s3)) + ((s4+s5)+(s6+s7)).
__device__ __forceinline__ float fold8_squares(const float (&a)[8])
{
    // The squares stay scalar: a packed multiply whose only use is a packed
    // add was found fused into one packed fma by the code generator (a
    // different rounding), which the scalar mul.rn never is.  The first
    // level adds are packed: (s0 + s1, s2 + s3) and (s4 + s5, s6 + s7).
    float s[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        s[e] = __fmul_rn(a[e], a[e]);
    float l0, l1, l2, l3;
    add2_rn(s[0], s[2], s[1], s[3], l0, l1);
    add2_rn(s[4], s[6], s[5], s[7], l2, l3);
    return __fadd_rn(__fadd_rn(l0, l1), __fadd_rn(l2, l3));
}

// y = (acc * inv) * w for one block, the two products rounded in that order.
__device__ __forceinline__ void scale8(float (&a)[8], float inv, const uint4& w)
{
    float wf[8];
    unpack8(w, wf);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        mul2_rn(a[e], a[e + 1], inv, inv, a[e], a[e + 1]);
        mul2_rn(a[e], a[e + 1], wf[e], wf[e + 1], a[e], a[e + 1]);
    }
}

// Pairwise fold of K partial sums held by one thread (K a power of two,
// adjacent pairs first).  Used for the top levels of the tree, where the
// K subtrees of a thread are adjacent aligned blocks of T * 8 elements.
template <int K>
__device__ __forceinline__ float fold_k(float (&p)[K])
{
#pragma unroll
    for (int width = 1; width < K; width *= 2) {
#pragma unroll
        for (int j = 0; j < K; j += 2 * width)
            p[j] = __fadd_rn(p[j], p[j + width]);
    }
    return p[0];
}

// One level-by-level butterfly over `width` lanes (a power of two <= 32):
// after the step with offset d every lane holds the sum of its aligned
// 2d-lane group, formed as (lower d-group) + (upper d-group).  fp32
// addition is commutative, so both partners hold the same bits.
__device__ __forceinline__ float butterfly_sum(float v, int width)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        if (d < width)
            v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    }
    return v;
}

// The maximum over `width` lanes (a power of two <= 32; all 32 lanes of
// the warp take part), in every lane.
__device__ __forceinline__ float butterfly_max(float v, int width)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        if (d < width)
            v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    }
    return v;
}

// The maximum over all 32 lanes of a warp (every lane active), in every
// lane, by one redux.sync: NaN is ignored unless every lane holds NaN (as
// fmaxf), or with warp_max_nan a NaN in any lane gives NaN.  The maximum is
// exact, so this equals the butterfly.
__device__ __forceinline__ float warp_max(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float warp_max_nan(float v)
{
    float r;
    asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// The K per-block partial sums of every lane of a full warp, reduced over
// the warp's 32 lanes by recursive halving: at the level with offset d
// (d = 1, 2, ..., K / 2) a lane keeps one half of its current list of
// subtree sums (the upper half if lane bit d is set) and sends the other
// half to lane ^ d, which keeps the opposite half, and adds what it
// receives to what it keeps; past K the single remaining sum goes through
// the ordinary butterfly.  Both partners of a level hold the sums of the
// same subtrees j over their aligned d-lane groups, so each addition is
// (lower group) + (upper group) of the canonical tree, as in
// butterfly_sum, with K / 2 + K / 4 + ... + 1 + (5 - log2 K) shuffles
// instead of 5 K.  Returns the sum over the warp of subtree j_out, where
// j_out is lane bit 0 -> K / 2, bit 1 -> K / 4, ... (the lane's low
// log2 K bits reversed).
template <int K>
__device__ __forceinline__ float warp_halving_sum(float (&p)[K], int lane, int& j_out)
{
    static_assert(K >= 1 && K <= 32 && (K & (K - 1)) == 0, "K: a power of two up to 32");
    int j = 0;
#pragma unroll
    for (int d = 1, c = K; d < K; d <<= 1, c >>= 1) {
        const bool upper = (lane & d) != 0;
        const int h = c >> 1;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float keep = upper ? p[h + i] : p[i];
            const float send = upper ? p[i] : p[h + i];
            p[i] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, d));
        }
        j += upper ? h : 0;
    }
    float v = p[0];
#pragma unroll
    for (int d = K; d < 32; d <<= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    j_out = j;
    return v;
}

// After warp_halving_sum in a one-warp row: the top log2 K levels of the
// tree, across the lanes that hold the K subtree sums.  Subtree j ^ 1 sits
// on lane ^ (K / 2), j ^ 2 on lane ^ (K / 4), ...; every lane ends with the
// row's sum.
template <int K>
__device__ __forceinline__ float fold_lane_subtrees(float v)
{
#pragma unroll
    for (int d = K >> 1; d >= 1; d >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    return v;
}

// The rest of the tree from red[j * W + w] = the sum of subtree j over warp
// w (W = T / 32 warps of a row, published by lanes 0 .. K - 1 after
// warp_halving_sum): over the warps of each subtree, then over the
// subtrees, adjacent pairs first at every level.  Every lane returns the
// row's sum.
template <int K, int W>
__device__ __forceinline__ float cross_warp_sum(const float* red, int lane)
{
    if constexpr (K * W <= 32) {
        // one value per lane: index j * W + w, so offsets below W join
        // warps and offsets W, 2W, ... join adjacent subtrees
        float v = red[lane & (K * W - 1)];
#pragma unroll
        for (int d = 1; d < K * W; d <<= 1)
            v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
        return v;
    } else {
        float q[K];
#pragma unroll
        for (int j = 0; j < K; ++j)
            q[j] = butterfly_sum(red[j * W + (lane & (W - 1))], W);
        return fold_k<K>(q);
    }
}

// max |y| over K blocks of 8 as a tree of max instructions (the maximum is
// exact, so any order gives the same value; the tree keeps the dependent
// chain short).  NAN_PROP: a NaN anywhere gives NaN (max.NaN, so a NaN y in
// a row shows in its amax and the row can take the exact path), else NaN is
// ignored (NaN only if every value is NaN).
template <bool NAN_PROP>
__device__ __forceinline__ float max2(float a, float b)
{
    float d;
    if constexpr (NAN_PROP)
        asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    else
        d = fmaxf(a, b);
    return d;
}

// max(a, b, c) in one three-input instruction, NaN propagating as in max2.
template <bool NAN_PROP>
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    if constexpr (NAN_PROP)
        asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    else
        asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Level by level: each level replaces consecutive triples of the N values
// by their max3 (a last pair by max2, a last single value passes), so N
// values take about N / 2 instructions.
template <int N, bool NAN_PROP>
__device__ __forceinline__ float max_tree(float (&v)[N])
{
    if constexpr (N == 1) {
        return v[0];
    } else {
        constexpr int M = (N + 2) / 3;
        float u[M];
#pragma unroll
        for (int i = 0; i < M; ++i) {
            const int k = 3 * i;
            if (k + 2 < N)
                u[i] = max3<NAN_PROP>(v[k], v[k + 1], v[k + 2]);
            else if (k + 1 < N)
                u[i] = max2<NAN_PROP>(v[k], v[k + 1]);
            else
                u[i] = v[k];
        }
        return max_tree<M, NAN_PROP>(u);
    }
}

template <int K, bool NAN_PROP>
__device__ __forceinline__ float tree_max_abs(const float (&y)[K][8])
{
    float a[K * 8];
#pragma unroll
    for (int j = 0; j < K; ++j) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            a[j * 8 + e] = fabsf(y[j][e]);
    }
    return max_tree<K * 8, NAN_PROP>(a);
}

// y = (acc * inv) * w for one block, with its 8 weights already in fp32
// (w_lo: elements 0-3, w_hi: 4-7).
__device__ __forceinline__ void scale8_f32(float (&a)[8], float inv, const float4& w_lo, const float4& w_hi)
{
    mul2_rn(a[0], a[1], inv, inv, a[0], a[1]);
    mul2_rn(a[2], a[3], inv, inv, a[2], a[3]);
    mul2_rn(a[4], a[5], inv, inv, a[4], a[5]);
    mul2_rn(a[6], a[7], inv, inv, a[6], a[7]);
    mul2_rn(a[0], a[1], w_lo.x, w_lo.y, a[0], a[1]);
    mul2_rn(a[2], a[3], w_lo.z, w_lo.w, a[2], a[3]);
    mul2_rn(a[4], a[5], w_hi.x, w_hi.y, a[4], a[5]);
    mul2_rn(a[6], a[7], w_hi.z, w_hi.w, a[6], a[7]);
}

// butterfly_max with NaN propagation: NaN in any lane gives NaN in all.
__device__ __forceinline__ float butterfly_max_nan(float v, int width)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        if (d < width) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v, d);
            asm("max.NaN.f32 %0, %1, %2;" : "=f"(v) : "f"(v), "f"(o));
        }
    }
    return v;
}

// inv = 1 / sqrt(S / hidden + eps), each operation rounded once.
// inv_hidden is 1 / hidden when hidden is a power of two (else 0): S / hidden
// and S * 2^-k are then the same real number, so rounding the product gives
// the correctly rounded quotient bit for bit.  1 / sqrt(v) is the correctly
// rounded reciprocal of the correctly rounded square root.
__device__ __forceinline__ float inv_rms(float sum_sq, int hidden, float inv_hidden, float eps)
{
    const float mean = inv_hidden != 0.0f ? __fmul_rn(sum_sq, inv_hidden)
                                          : __fdiv_rn(sum_sq, static_cast<float>(hidden));
    const float v = __fadd_rn(mean, eps);
    return __frcp_rn(__fsqrt_rn(v));
}

// q = clamp(rint(RN(y / scale)), -127, 127) with rint ties to even, where
// RN(y / scale) is the correctly rounded fp32 quotient; scale == 0 gives 0.
//
// Fast path, for a normal finite scale (every row with amax >= 127 * 2^-126):
// with c = RN(1 / scale) and z = y * c exactly, the relative error of c is
// at most 2^-24 and |y / scale| <= amax / RN(amax / 127) <= 127 / (1 - 2^-24),
// so |z - y/scale| <= 2^-24 * 127.00001; also |RN(y/scale) - y/scale| <=
// 2^-24 * 127.00001: z and RN(y / scale) are less than 1.6e-5 apart.  When z
// is at least 2^-15 - 2^-25 away from the nearest half-integer, no
// half-integer lies between the two and both round to the same integer,
// rint(z) (see quantize8).  Otherwise (for about 2^-14 of all values, so for
// about one 8-value block in 1,000) the block's quotients are computed
// exactly with a correctly rounded division.
struct QuantScale {
    float scale;
    float recip;  // RN(1 / scale)
    bool fast;
};

__device__ __forceinline__ QuantScale make_quant_scale(float scale)
{
    QuantScale s;
    s.scale = scale;
    s.fast = scale >= 0x1p-126f && scale <= 3.40282347e38f;
    s.recip = s.fast ? __frcp_rn(scale) : 0.0f;
    return s;
}

// The reference path for one element: correctly rounded quotient, then
// rint ties to even (cvt.rni; NaN -> 0, saturating), then the clamp.
__device__ __forceinline__ int32_t quantize_exact(float y, float scale)
{
    if (scale == 0.0f)
        return 0;
    int32_t q = __float2int_rn(__fdiv_rn(y, scale));
    q = q > 127 ? 127 : q;
    q = q < -127 ? -127 : q;
    return q;
}

// Low bytes of four words packed into one word, first in the lowest byte.
__device__ __forceinline__ uint32_t pack4_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    const uint32_t ab = __byte_perm(a, b, 0x0040);
    const uint32_t cd = __byte_perm(c, d, 0x0040);
    return __byte_perm(ab, cd, 0x5410);
}

// Eight int8 codes for eight consecutive y values.  Fast path: with z the
// exact product y * c, m = fma(y, c, 1.5 * 2^23) rounds z (|z| < 2^22) to an
// integer, ties to even, held in m's low mantissa bits: t = m - 1.5 * 2^23
// is rint(z) exactly, and the low byte of m's bit pattern is the low byte of
// that integer (the constant's own low byte is zero), i.e. the int8 code.
// d = fma(y, c, -t) is z - t rounded once (error below 2^-25 near a half),
// and |z - RN(y / scale)| <= 2^-24 * 127.00001 * 2 < 1.6e-5; so when
// |d| <= 0.5 - 2^-15, no half-integer lies between z and RN(y / scale) and
// rint(z) = rint(RN(y / scale)).  |z| <= 127.0001 here, so no clamp is
// needed.  If any of the eight is nearer a half-integer (or the scale is not
// a normal number) the block is redone with quantize_exact.
__device__ __forceinline__ uint2 quantize8(const float (&y)[8], const QuantScale& s)
{
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    uint32_t bits[8];
    bool near_tie = !s.fast;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float m0, m1, nt0, nt1, d0, d1;
        fma2_rn(y[e], y[e + 1], s.recip, s.recip, kRound, kRound, m0, m1);
        sub2_rn(kRound, kRound, m0, m1, nt0, nt1);  // -t, exactly
        fma2_rn(y[e], y[e + 1], s.recip, s.recip, nt0, nt1, d0, d1);
        near_tie |= !(fabsf(d0) <= 0.5f - 0x1p-15f) || !(fabsf(d1) <= 0.5f - 0x1p-15f);
        bits[e] = __float_as_uint(m0);
        bits[e + 1] = __float_as_uint(m1);
    }
    if (near_tie) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            bits[e] = static_cast<uint32_t>(quantize_exact(y[e], s.scale));
    }
    uint2 u;
    u.x = pack4_low_bytes(bits[0], bits[1], bits[2], bits[3]);
    u.y = pack4_low_bytes(bits[4], bits[5], bits[6], bits[7]);
    return u;
}

// Int8 codes by a bracket of the quotient.  With c the hardware reciprocal
// of scale (rcp.approx, documented to be within 1 ulp, so a relative error
// below 2^-22 where scale and 1 / scale are normal), c_lo = RN(c (1 - 2^-21)) and
// c_hi = RN(c (1 + 2^-21)) satisfy, for y >= 0 and a normal quotient,
//   y c_lo <= y/scale (1 + 2^-22)(1 - 2^-21)(1 + 2^-24) < y/scale (1 - 2^-24)
//          <= RN(y / scale) <= y/scale (1 + 2^-24)
//          < y/scale (1 - 2^-22)(1 + 2^-21)(1 - 2^-24) <= y c_hi
// (mirrored for y < 0; a subnormal quotient is below 2^-126 and every
// candidate then rounds to 0).  fma(y, c, 1.5 * 2^23) is 1.5 * 2^23 plus
// the exact product rounded to an integer, ties to even (|y c| < 2^22 here),
// and rounding to an integer is monotone, so when the two ends give the
// same bits, rint(RN(y / scale)) is that integer; |y / scale| <= 127.00001,
// so no clamp is needed.  The low byte of those bits is the int8 code.
// fast: scale normal and below 2^120; rows with a NaN y or another scale
// take quantize_exact.
struct Int8Bracket {
    float scale;
    float c_lo, c_hi;
    bool fast;
};

__device__ __forceinline__ Int8Bracket make_int8_bracket(float scale)
{
    Int8Bracket s;
    s.scale = scale;
    s.fast = scale >= 0x1p-126f && scale < 0x1p120f;
    // a normal scale below 2^120 has a normal reciprocal: the flush-to-zero
    // form of rcp.approx gives the same value without subnormal handling
    float c = 0.0f;
    if (s.fast)
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(c) : "f"(scale));
    s.c_lo = __fmul_rn(c, 1.0f - 0x1p-21f);
    s.c_hi = __fmul_rn(c, 1.0f + 0x1p-21f);
    return s;
}

// Eight codes; `differ` collects the bits in which any pair of ends
// differs (nonzero: redo the block with quantize_exact).
__device__ __forceinline__ uint2 quantize8_bracket(const float (&y)[8], const Int8Bracket& s, uint32_t& differ)
{
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
    uint32_t lo[8], d[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float l0, l1, h0, h1;
        fma2_rn(y[e], y[e + 1], s.c_lo, s.c_lo, kRound, kRound, l0, l1);
        fma2_rn(y[e], y[e + 1], s.c_hi, s.c_hi, kRound, kRound, h0, h1);
        lo[e] = __float_as_uint(l0);
        lo[e + 1] = __float_as_uint(l1);
        d[e / 2] = (lo[e] ^ __float_as_uint(h0)) | (lo[e + 1] ^ __float_as_uint(h1));
    }
    differ |= (d[0] | d[1]) | (d[2] | d[3]);
    uint2 u;
    u.x = pack4_low_bytes(lo[0], lo[1], lo[2], lo[3]);
    u.y = pack4_low_bytes(lo[4], lo[5], lo[6], lo[7]);
    return u;
}

__device__ __forceinline__ uint2 quantize8_exact(const float (&y)[8], float scale)
{
    uint32_t q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        q[e] = static_cast<uint32_t>(quantize_exact(y[e], scale));
    uint2 u;
    u.x = pack4_low_bytes(q[0], q[1], q[2], q[3]);
    u.y = pack4_low_bytes(q[4], q[5], q[6], q[7]);
    return u;
}

// ------------------------------------------------------------ fp8 e4m3 codes
// cvt.rn.satfinite.e4m3x2.f32 rounds two fp32 values to nearest-even e4m3
// (OCP e4m3fn: subnormals kept, magnitudes past 448 saturate to 448, NaN to
// NaN) and packs them, the first operand in the high byte.  Equal to the
// oracle's encoder on every non-NaN fp32 input (checked exhaustively by the
// test suite).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// RN(m / d) for an amax m >= 0 and the divisor d of a quantised format
// (127 for int8, 448 for fp8 e4m3, 6 for fp4 e2m1), by division with one
// correction step (Markstein): q0 = RN(m * c) with c = RN(1 / d); the
// remainder m - q0 * d is exact in one fused multiply-add; q = RN(q0 +
// remainder * c).  Every operation scales exactly with m by powers of two
// while q0 and the remainder stay normal, so checking every significand in
// a few binades proves the identity for all m in [2^-100, 2^128): the test
// suite checks every m in that range against the correctly rounded
// quotient, for each of the three divisors and constants.  Anything else
// (0, subnormal or tiny m, Inf, NaN) takes the IEEE division.
template <int D>
__device__ __forceinline__ float div_const_rn(float m)
{
    static_assert(D == 127 || D == 448 || D == 6, "divisor: 127, 448 or 6");
    constexpr float kInv = D == 127 ? 0x1.020408p-7f : D == 448 ? 0x1.24924ap-9f : 0x1.555556p-3f;  // RN(1 / D)
    constexpr float kD = static_cast<float>(D);
    if (!(m >= 0x1p-100f && m <= 3.40282347e38f))
        return __fdiv_rn(m, kD);
    const float q0 = __fmul_rn(m, kInv);
    const float r = __fmaf_rn(-q0, kD, m);
    return __fmaf_rn(r, kInv, q0);
}

__device__ __forceinline__ float div448_rn(float m)
{
    return div_const_rn<448>(m);
}

// Per-row (or per-group) fp8 / fp4 scale (scale = RN(amax / 448) or
// RN(amax / 6)) and two multipliers that bracket 1 / scale:
// c_lo = RN(c * (1 - 2^-20)) and c_hi = RN(c * (1 + 2^-20)), where c is
// 1 / scale to within a relative 2^-22.  fast: scale is a normal number
// below 2^120 (so 1 / scale is normal too); else quantisation divides.
struct E4m3Scale {
    float scale;
    float c_lo, c_hi;
    bool fast;
};

__device__ __forceinline__ E4m3Scale make_e4m3_scale(float scale)
{
    E4m3Scale s;
    s.scale = scale;
    s.fast = scale >= 0x1p-126f && scale < 0x1p120f;
    // a normal scale below 2^120 has a normal reciprocal: the flush-to-zero
    // form of rcp.approx gives the same value without subnormal handling
    float c = 0.0f;
    if (s.fast)
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(c) : "f"(scale));
    s.c_lo = __fmul_rn(c, 1.0f - 0x1p-20f);
    s.c_hi = __fmul_rn(c, 1.0f + 0x1p-20f);
    return s;
}

// Eight e4m3 codes for eight consecutive y values: e4m3(RN(y / scale)).
// Fast path: c is within a relative 2^-22 of 1 / scale and every rounding
// is relative and at most 2^-24, so for y >= 0 RN(y * c_lo) <=
// y/scale * (1 - 2^-20 + 2^-22 + 3 * 2^-24) < y/scale * (1 - 2^-24) <=
// RN(y / scale), and likewise RN(y / scale) <= RN(y * c_hi) (mirrored for
// y < 0; values too small for a relative bound are below half the smallest
// e4m3 step and give code 0 at both ends).  Rounding to e4m3 is monotone, so when
// both ends give the same code, RN(y / scale) gives it too.  A block where
// any pair of ends differs (a quotient within about 2^-20 of an e4m3
// rounding boundary), or a scale that is not a normal number, is redone with
// the correctly rounded division; scale == 0 gives code 0.
__device__ __forceinline__ uint2 quantize8_e4m3(const float (&y)[8], const E4m3Scale& s)
{
    uint32_t lo[4], hi[4];
    bool boundary = !s.fast;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float l0, l1, h0, h1;
        mul2_rn(y[2 * p], y[2 * p + 1], s.c_lo, s.c_lo, l0, l1);
        mul2_rn(y[2 * p], y[2 * p + 1], s.c_hi, s.c_hi, h0, h1);
        lo[p] = e4m3x2(l0, l1);
        hi[p] = e4m3x2(h0, h1);
        boundary |= lo[p] != hi[p];
    }
    if (boundary) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            lo[p] = s.scale == 0.0f
                        ? 0u
                        : e4m3x2(__fdiv_rn(y[2 * p], s.scale), __fdiv_rn(y[2 * p + 1], s.scale));
        }
    }
    uint2 u;
    u.x = lo[0] | (lo[1] << 16);
    u.y = lo[2] | (lo[3] << 16);
    return u;
}

// ------------------------------------------------------------ fp4 e2m1 codes
// cvt.rn.satfinite.e2m1x2.f32 rounds two fp32 values to nearest-even e2m1
// (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; past 6 saturates) and packs them
// into one byte, the first operand in the high nibble.  Equal to the
// oracle's encoder on every non-NaN fp32 input (checked exhaustively by the
// test suite).
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint16_t d;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u16.u8 %0, t;\n\t}"
        : "=h"(d)
        : "f"(hi), "f"(lo));
    return d;
}

// Eight e2m1 codes (four bytes, even elements in the low nibbles) for eight
// consecutive y values: e2m1(RN(y / scale)), by the same bracket as
// quantize8_e4m3 (rounding to e2m1 is monotone too); `s` is built by
// make_e4m3_scale from scale = RN(amax / 6).
__device__ __forceinline__ uint32_t quantize8_e2m1(const float (&y)[8], const E4m3Scale& s)
{
    uint32_t lo[4], hi[4];
    bool boundary = !s.fast;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float l0, l1, h0, h1;
        mul2_rn(y[2 * p], y[2 * p + 1], s.c_lo, s.c_lo, l0, l1);
        mul2_rn(y[2 * p], y[2 * p + 1], s.c_hi, s.c_hi, h0, h1);
        lo[p] = e2m1x2(l0, l1);
        hi[p] = e2m1x2(h0, h1);
        boundary |= lo[p] != hi[p];
    }
    if (boundary) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            lo[p] = s.scale == 0.0f
                        ? 0u
                        : e2m1x2(__fdiv_rn(y[2 * p], s.scale), __fdiv_rn(y[2 * p + 1], s.scale));
        }
    }
    return lo[0] | (lo[1] << 8) | (lo[2] << 16) | (lo[3] << 24);
}

// ------------------------------------------------------ mbarrier and bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Makes the initialised barriers visible to the asynchronous proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses before later
// asynchronous-proxy (bulk copy) accesses to shared memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity to complete, giving up
// after `limit_ns` nanoseconds or 2^26 polls, whichever comes first.
// Returns false on giving up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < (1u << 26); ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> this CTA's shared memory, completing `bytes`
// transaction bytes on `bar`.  Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src_gmem,
                                              uint32_t bytes, uint64_t* bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// An L2 prefetch of `bytes` bytes at `src` (16-byte aligned, a multiple of
// 16 bytes).  A hint only: it brings lines into L2 and moves nothing to the
// SM, so a load issued later still reads what the memory holds then.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------- thread-block clusters
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x()
{
    uint32_t r;
    asm("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives, then waits for all the
// others; shared-memory writes before it are visible to the whole cluster
// after it (release / acquire at cluster scope).  Callers keep the number
// of calls equal on every CTA of a cluster.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// A float in the shared memory of CTA `rank` of this cluster, at the address
// `local` has in this CTA's shared memory.
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// ---------------------------------------------- programmatic dependent launch
// Blocks until every grid this one depends on in the stream has completed
// and its memory is visible; a no-op when the grid was launched without
// programmatic stream serialization.  Called before any global access.
__device__ __forceinline__ void wait_prior_grids()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next grid in the stream be scheduled now; its CTAs then start as
// SMs free up and block in wait_prior_grids() until this grid is done.
__device__ __forceinline__ void allow_next_grid()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ global access
// Streaming (read-once / write-once) 16-byte accesses.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint2* p, const uint2& v) { __stcs(p, v); }

}  // namespace dradd
